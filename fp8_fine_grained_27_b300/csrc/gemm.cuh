// gemm.cuh -- block-scaled E4M3 GEMM with FP32 promotion every 128 K, on the
// sm_103a fifth-generation tensor cores (V3 report §6: FP8 Fprop/Dgrad/Wgrad
// GEMMs, BF16 or FP32 outputs; §6.2: partial sums promoted to FP32 after
// every 128 FP8 products).
//
// The pages' design promotes on Hopper CUDA cores because the Hopper FP8
// tensor-core accumulator is short.  Here the promotion is re-shaped for
// tcgen05: each 128-wide K chunk is one chain of four M128 x BN x K32 MMAs
// into a fresh FP32 partial in tensor memory (TMEM); promotion warps read the
// partial with tcgen05.ld and fold it into FP32 register accumulators,
//     acc[m][n] = fmaf(sa[kb][m] * sb(n, kb), P_kb[m][n], acc[m][n]),
// while the MMA warp already fills the other TMEM buffer with chunk kb+1.
//
// CTA layout (persistent, one CTA per SM), for an output tile 128 x BN:
//   warp 0      TMA producer: A and B K-chunks (128 bytes of K per row, the
//               128-byte swizzle) into a STAGES-deep shared-memory ring.
//   warps 1, 3  MMA issuers (one thread each): warp 1 issues the even K
//               chunks, warp 3 the odd ones.  Issuing a tcgen05.mma costs the
//               issuing thread about as long as a 128 x 128 x 32 MMA takes to
//               execute, so two issuers keep the tensor pipe fed; each one
//               commits its own chunks.  Warp 1 also owns the TMEM allocation.
//   warp 2      idle.  Warpgroup 0 gives registers away (setmaxnreg 40).
//   warps 4..   promotion + epilogue, NWG warpgroups (setmaxnreg raised).
//               Warp w reads TMEM lanes 32*(w%4) .. +31 (its 32 tile rows);
//               warpgroup g owns columns [g*CPW, (g+1)*CPW) of the tile.
//   BN = 256: 2 promotion warpgroups x 128 columns, 2 TMEM partials
//             (four 32-column TMEM loads per chunk, software-pipelined);
//   BN = 192: 3 promotion warpgroups x 64 columns, 2 TMEM partials;
//   BN = 128: 2 promotion warpgroups x 64 columns, 4 TMEM partials.
//   With block scales and 64 columns per thread both 32-column loads of a
//   chunk are issued before a single wait.  Per-row scales (BMODE 1) read the
//   partial in the 16x256b shape at every width (see the promotion below);
//   the library picks 256 for block scales and 192 for per-row scales.
//
// Synchronisation (all mbarriers, all waits bounded):
//   full[s]   TMA bytes of stage s landed          (producer -> MMA)
//   empty[s]  MMAs reading stage s are complete    (tcgen05.commit -> producer)
//   tfull[b]  partial in TMEM buffer b is complete (tcgen05.commit -> promotion)
//   tempty[b] promotion has read buffer b          (one arrival per promotion warp -> MMA)
//   sbfull/sbempty  B row scales of a chunk (row-scale mode only), freed by
//             the promotion when it has folded the chunk
//
// The last round of tiles (FP32 output).  When the tiles do not fill the
// last round of the persistent grid (Wgrad: 608 tiles of 128 x 192 on 148
// CTAs is four rounds and 16 tiles), the tiles from the second-to-last round on are
// shared out by K chunks instead: CTA b takes the b-th of G equal runs of
// their chunks, in tile order, so every CTA does the same number of chunks.
// A tile then falls to at most two CTAs (every run is longer than a tile).
// Its first K chunks go to the CTA that holds the tile's end of the run
// order (CTA b+1, which meets the tile first), and that CTA stores its FP32
// accumulators in C and raises a flag; CTA b, which meets the tile at the
// end of its run, waits for the flag, takes those accumulators as its
// starting values and promotes the remaining chunks.  Every output element
// is promoted chunk by chunk in K order from zero, exactly as in a whole
// tile, so the result is bit-identical.  The flag holds a per-launch value,
// in a ring of flag slots that concurrent launches do not share.
//
// SwiGLU variant (V3 report §2: SwiGLU experts; §6.1: the down projection
// takes the 1x128-quantised SwiGLU output): B holds the gate rows [0, N) and
// the up rows [N, 2N) of the up projection.  A 128 x 256 MMA tile loads gate
// block j and up block j (two 128-row TMA boxes) and yields the 128 channels
// 128j .. 128j+127: each promotion thread owns the gate and the up columns
// of the same 64 channels, forms h = silu(g) * u from its FP32 accumulators,
// the two warpgroups exchange their row amax, and the epilogue writes the
// E4M3 codes and 1x128 scales of h instead of C.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace gemm {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int kFirstPromoWarp = 4;
// Raster: group_m M tiles sweep N together, so that the tiles in flight share
// their A panels, which stay in L2 for the whole sweep while each B panel is
// read once per group.  The host picks 32 when the group's A panels
// (32 x 128 rows x K bytes) fit in 32 MB, else 16: at K = 7168 that halves
// the B re-reads; at K = 18432 a 32-tile group no longer stays in L2.
constexpr int kGroupMSmall = 16, kGroupMLarge = 32;
__host__ __device__ inline int group_m_for(int64_t K)
{
    return (int64_t(kGroupMLarge) * 128 * K <= (int64_t(32) << 20)) ? kGroupMLarge : kGroupMSmall;
}
constexpr int kMaxGroups = 1024; // grouped GEMM: experts per call
constexpr int kMaxSmem = 232448; // dynamic shared memory per CTA on sm_103

template <int BN_, int BMODE_, bool GROUPED_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int CPW = (BN == 256) ? 128 : 64;  // columns per promotion thread
    static constexpr int NWG = BN / CPW;                // promotion warpgroups
    static constexpr int NPW = 4 * NWG;                 // promotion warps
    static constexpr int THREADS = 128 * (1 + NWG);
    static constexpr int NP = CPW / 32;                 // 32-column TMEM loads per chunk
    static constexpr int NTMEM = (BN <= 128) ? 4 : 2;   // TMEM partial buffers
    static constexpr int TMEM_COLS = 512;
    // registers: warpgroup 0 drops to 40; the promotion warpgroups share the
    // rest of the launch's pool (THREADS x launch registers, 168 at 384
    // threads, 128 at 512 threads)
    static constexpr int LAUNCH_REGS = (THREADS == 384) ? 168 : 128;
    static constexpr int PROMO_REGS = ((THREADS * LAUNCH_REGS - 128 * 40) / (128 * NWG)) / 8 * 8;
    static_assert(128 * 40 + 128 * NWG * PROMO_REGS <= THREADS * LAUNCH_REGS, "setmaxnreg split exceeds the pool");
    static_assert(PROMO_REGS <= 256 && PROMO_REGS >= CPW + 64 + 16, "promotion registers");
    static_assert(NTMEM * BN <= TMEM_COLS, "TMEM partials");
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SBROW_BYTES = (BMODE_ == 1) ? BN * 4 : 0;
    static constexpr int SAROW_BYTES = (BMODE_ == 1) ? BM * 4 : 0;  // the chunk's A row scales (Params::sa_smem)
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SBROW_BYTES + SAROW_BYTES;
    static constexpr int EPI_BYTES = NPW * 2048;
    static constexpr int TABLE_BYTES = GROUPED_ ? (kMaxGroups + 1) * 4 : 0;
    static constexpr int XCH_BYTES = 2048;  // SwiGLU row-amax exchange, two tiles deep
    static constexpr int FIXED = EPI_BYTES + XCH_BYTES + TABLE_BYTES + 512 + 1024;  // + barriers, + alignment slack
    // Even, so that every use of a stage falls to the same MMA issuer (chunks
    // c and c + STAGES have the same parity): each issuer then waits the
    // phases of its stages in order and can never mistake a stage's previous
    // completed phase for the one it needs.
    static constexpr int FIT = (kMaxSmem - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = (FIT < 6 ? FIT : 6) / 2 * 2;
    static_assert(STAGES >= 4 && STAGES % 2 == 0, "pipeline depth");
    // Row-scale slots.  A ring twice as deep (so that the producer, which
    // loads a chunk's scales right after its operands, never waits for the
    // promotion to free one) measured the same.
    static constexpr int SB_STAGES = STAGES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SBROW = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SAROW = OFF_SBROW + SB_STAGES * SBROW_BYTES;
    static constexpr int OFF_EPI = OFF_SAROW + SB_STAGES * SAROW_BYTES;
    static constexpr int OFF_XCH = OFF_EPI + EPI_BYTES;
    static constexpr int OFF_BAR = OFF_XCH + XCH_BYTES;
    static constexpr int NBAR = 2 * STAGES + 2 * SB_STAGES + 2 * NTMEM + 3;  // + SwiGLU exchange, two K-split
    static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
    static constexpr int OFF_TILESTART = (OFF_TMEMSLOT + 4 + 15) / 16 * 16;
    static constexpr int BYTES = OFF_TILESTART + TABLE_BYTES;
    static constexpr int ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
    static_assert(NBAR * 8 + 32 <= 512, "barrier area");
    static_assert(ALLOC <= kMaxSmem, "shared memory per CTA");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

struct Params {
    const float *sa;
    int64_t ldsa;
    const float *sb;     // BMODE 0: sb[nb*ldsb + kb] (per expert: + e*sb_estride)
    int64_t ldsb;
    int64_t sb_estride;
    void *C;             // output; SwiGLU: E4M3 codes of h
    int64_t ldc;
    float *s_out;        // SwiGLU: 1x128 scales of h, [N/128][lds_out]
    int64_t lds_out;
    int M, N, K;         // M = rows of A (M_total when grouped); N = output columns
    int tile_n;          // output columns per tile (BN; SwiGLU: 128)
    int b_rows;          // rows of B per expert (N; SwiGLU: 2N)
    int group_m;         // raster group (dense only; group_m_for(K))
    const int32_t *offs; // grouped: [G+1] row offsets (device)
    int G;
    int sk_first = 0x7FFFFFFF;  // first tile shared out by K chunks (dense FP32 output); none by default
    uint32_t *sk_flags = nullptr;  // flag of the tile split between CTA b and b+1: sk_flags[b]
    uint32_t sk_epoch = 0;         // this launch's flag value (never 0)
    // BMODE 1: the producer copies each chunk's A row scales
    // (sa[kb*ldsa + m0 ..], min(128, M - m0) floats) into the chunk's scale
    // slot beside its B scale row; the host sets it when sa is 16-byte
    // aligned and ldsa and M are multiples of 4, so that the copy is a
    // legal bulk copy
    int sa_smem = 0;
};

// One piece of work of a CTA: tile t, K chunks [kb0, kb1).
enum : int { ITEM_FULL = 0, ITEM_HEAD = 1, ITEM_TAIL = 2 };
struct Item {
    int t, kb0, kb1, mode;
};

// The K-split run of one CTA (in shared memory, written once at its start):
// n_rr whole tiles b, b + G, ... below skf, then the chunks [u0, u1) of tiles
// skf .. total-1, counted from tile skf's first chunk; s0 = the run's first
// tile boundary.  The host keeps (total - skf) x nk below 2^31.
struct SplitRun {
    int n_rr, skf, u0, u1, s0;
};

__device__ __forceinline__ void split_run_init(SplitRun &r, int b, int G, int total, int sk_first, int nk)
{
    const int skf = min(sk_first, total);
    r.skf = skf;
    r.n_rr = skf > b ? (skf - b + G - 1) / G : 0;
    const int64_t U = static_cast<int64_t>(total - skf) * nk;
    const int64_t u0 = U * b / G, u1 = U * (b + 1) / G;
    r.u0 = static_cast<int>(u0);
    r.u1 = static_cast<int>(u1);
    r.s0 = static_cast<int>((u0 + nk - 1) / nk * nk);
}

// Piece j of the work of CTA b of G (the same sequence for its producer, MMA
// and promotion roles); false past the last piece.  Without the K split
// (SPLIT false) the pieces are the whole tiles b, b + G, ... below total.
// The run is read from shared memory for every piece, so that the roles keep
// only j live across their loops.
template <bool SPLIT>
__device__ __forceinline__ bool item_of(int j, int b, int G, int total, int nk, const volatile SplitRun *r, Item &it)
{
    if constexpr (!SPLIT) {
        it = Item{b + j * G, 0, nk, ITEM_FULL};
        return it.t < total;
    } else {
        const int n_rr = r->n_rr;
        if (j < n_rr) {
            it = Item{b + j * G, 0, nk, ITEM_FULL};
            return true;
        }
        const int k = j - n_rr;
        const int u0 = r->u0, u1 = r->u1, s0 = r->s0;
        const int head = u0 < s0 ? 1 : 0;
        const int start = k < head ? u0 : s0 + (k - head) * nk;
        const int end = k < head ? min(u1, s0) : min(u1, start + nk);
        if (start >= u1)
            return false;
        const int rel = start / nk;
        const int lo = rel * nk, hi = lo + nk;
        const int len = end - start;
        it.t = r->skf + rel;
        if (start > lo) {  // the tile's end of the run order: its first len chunks, to hand on
            it.kb0 = 0;
            it.kb1 = len;
            it.mode = ITEM_HEAD;
        } else if (end < hi) {  // the tile's start of the run order: its last len chunks, to finish
            it.kb0 = nk - len;
            it.kb1 = nk;
            it.mode = ITEM_TAIL;
        } else {
            it.kb0 = 0;
            it.kb1 = nk;
            it.mode = ITEM_FULL;
        }
        dbg_ok(!(start > lo && end < hi), DBG_GEMM_SPLIT);
        return true;
    }
}

struct Tile {
    int m0, m_end, n0, brow0;
    const float *sbp;    // block scales of this tile's B (BMODE 0)
    bool valid;
};

template <int BN, bool GROUPED>
__device__ __forceinline__ Tile tile_of(int t, const Params &p, const int *tile_start)
{
    Tile r;
    const int num_n = (p.N + p.tile_n - 1) / p.tile_n;
    if constexpr (!GROUPED) {
        const int num_m = (p.M + BM - 1) / BM;
        const int per_group = p.group_m * num_n;
        const int g = t / per_group;
        const int first_m = g * p.group_m;
        const int gsize = min(num_m - first_m, p.group_m);
        const int local = t - g * per_group;
        const int mt = first_m + local % gsize;
        const int nt = local / gsize;
        r.m0 = mt * BM;
        r.m_end = p.M;
        r.n0 = nt * p.tile_n;
        r.brow0 = r.n0;
        r.sbp = p.sb;
        r.valid = true;
    } else {
        int lo = 0, hi = p.G;  // largest e with tile_start[e] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid;
        }
        const int e = lo;
        const int base = p.offs[e];
        const int m_e = p.offs[e + 1] - base;
        dbg_ok(e >= 0 && e < p.G && base >= 0 && m_e > 0 && base + m_e <= p.M, DBG_GEMM_GROUP);
        const int mtiles = (m_e + BM - 1) / BM;
        const int local = t - tile_start[e];
        const int nt = local / mtiles;
        const int mt = local - nt * mtiles;
        r.m0 = base + mt * BM;
        r.m_end = base + m_e;
        r.n0 = nt * p.tile_n;
        r.brow0 = e * p.b_rows + r.n0;
        r.sbp = p.sb + static_cast<int64_t>(e) * p.sb_estride;
        r.valid = true;
    }
    return r;
}

// Prefix sum of per-expert tile counts, computed by the promotion warps.
// Malformed ranges (negative length or past M) count as empty.
template <int NPW>
__device__ void build_tile_start(const Params &p, int *tile_start, int ptid)
{
    const int num_n = (p.N + p.tile_n - 1) / p.tile_n;
    __shared__ int warp_sums[NPW];
    // each promotion thread owns up to PER consecutive experts
    constexpr int PER = (kMaxGroups + NPW * 32 - 1) / (NPW * 32);
    int cnt[PER];
    int local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = ptid * PER + i;
        int c = 0;
        if (e < p.G) {
            const int a = p.offs[e], b = p.offs[e + 1];
            const int m_e = b - a;
            if (a >= 0 && m_e > 0 && b <= p.M)
                c = ((m_e + BM - 1) / BM) * num_n;
        }
        cnt[i] = c;
        local += c;
    }
    const int lane = ptid & 31, w = ptid >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_sums[w] = incl;
    asm volatile("bar.sync 1, %0;" ::"n"(NPW * 32));
    int before = 0;
    for (int i = 0; i < w; ++i)
        before += warp_sums[i];
    int run = before + incl - local;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = ptid * PER + i;
        if (e < p.G)
            tile_start[e] = run;
        run += cnt[i];
    }
    if (ptid == NPW * 32 - 1)
        tile_start[p.G] = run;
}

// Per-row B scales: acc.{x,y} = fl32(sa * sb.{x,y}) * P.{x,y} + acc.{x,y},
// each product and sum rounded exactly as the scalar mul and fmaf would be,
// two columns per instruction.
__device__ __forceinline__ void fold_rowscale2(float &a0, float &a1, uint64_t sa2, float sb0, float sb1, uint32_t p0,
                                               uint32_t p1)
{
    uint64_t acc, sc2;
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tmul.rn.f32x2 %0, %3, t;\n\t}"
        : "=l"(sc2)
        : "f"(sb0), "f"(sb1), "l"(sa2));
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tfma.rn.f32x2 %0, %3, t, %0;\n\t}"
        : "+l"(acc)
        : "r"(p0), "r"(p1), "l"(sc2));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Wait for the registers of the last tcgen05.ld and tie them to the wait so
// that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31])
                 :
                 : "memory");
}

// As tmem_ld_wait_regs2, for two 16-register loads.
__device__ __forceinline__ void tmem_ld_wait_regs16x2(uint32_t (&r)[16], uint32_t (&q)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]), "+r"(q[4]),
                   "+r"(q[5]), "+r"(q[6]), "+r"(q[7]), "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]),
                   "+r"(q[12]), "+r"(q[13]), "+r"(q[14]), "+r"(q[15])
                 :
                 : "memory");
}

// Wait for both outstanding tcgen05.ld of this warp and tie their registers
// to the wait, so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait_regs2(uint32_t (&r)[32], uint32_t (&q)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(q[0]), "+r"(q[1]), "+r"(q[2]),
                   "+r"(q[3]), "+r"(q[4]), "+r"(q[5]), "+r"(q[6]), "+r"(q[7]), "+r"(q[8]), "+r"(q[9]),
                   "+r"(q[10]), "+r"(q[11]), "+r"(q[12]), "+r"(q[13]), "+r"(q[14]), "+r"(q[15]), "+r"(q[16]),
                   "+r"(q[17]), "+r"(q[18]), "+r"(q[19]), "+r"(q[20]), "+r"(q[21]), "+r"(q[22]), "+r"(q[23]),
                   "+r"(q[24]), "+r"(q[25]), "+r"(q[26]), "+r"(q[27]), "+r"(q[28]), "+r"(q[29]), "+r"(q[30]),
                   "+r"(q[31])
                 :
                 : "memory");
}

template <int BN, int BMODE, bool OUT_F32, bool GROUPED, bool SWIGLU = false>
__global__ void __launch_bounds__(Cfg<BN, BMODE, GROUPED>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSB, const Params p)
{
    using L = Cfg<BN, BMODE, GROUPED>;
    static_assert(!SWIGLU || (BN == 256 && BMODE == 0 && !OUT_F32), "SwiGLU: 128 x 256 tiles, block scales");
    constexpr int STAGES = L::STAGES;
    constexpr int NTMEM = L::NTMEM;
    extern __shared__ uint8_t dyn_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dyn_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t bar_full = sbase + L::OFF_BAR;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    constexpr int SB_STAGES = L::SB_STAGES;
    const uint32_t bar_sbfull = bar_empty + 8 * STAGES;
    const uint32_t bar_sbempty = bar_sbfull + 8 * SB_STAGES;
    const uint32_t bar_tfull = bar_sbempty + 8 * SB_STAGES;
    const uint32_t bar_tempty = bar_tfull + 8 * NTMEM;
    const uint32_t bar_xch = bar_tempty + 8 * NTMEM;
    const uint32_t bar_skhead = bar_xch + 8;  // promotion warps' K-split partial stored
    const uint32_t bar_sktail = bar_xch + 16; // the partial to continue from is in C
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_TMEMSLOT);
    int *tile_start = reinterpret_cast<int *>(smem + L::OFF_TILESTART);
    // raised by the first wait of this CTA that gives up (see mbar_wait)
    __shared__ int s_abort;
    // K-split instances: this CTA's run of pieces
    constexpr bool SPLIT_OK = OUT_F32 && !GROUPED && !SWIGLU;
    __shared__ SplitRun s_run;

    if (threadIdx.x == 0) {
        s_abort = 0;
        if constexpr (SPLIT_OK)
            split_run_init(s_run, blockIdx.x, gridDim.x, ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN), p.sk_first,
                           p.K / BK);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int q = 0; q < SB_STAGES; ++q) {
            mbar_init(bar_sbfull + 8 * q, 1);
            mbar_init(bar_sbempty + 8 * q, L::NPW);
        }
        for (int b = 0; b < NTMEM; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, L::NPW);
        }
        mbar_init(bar_xch, L::NPW * 32);
        mbar_init(bar_skhead, L::NPW);
        mbar_init(bar_sktail, 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (BMODE == 1)
            tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    // the set-up above overlaps the end of the kernel that produced the inputs
    grid_dependency_wait();
    if constexpr (GROUPED) {
        if (warp >= kFirstPromoWarp)
            build_tile_start<L::NPW>(p, tile_start, threadIdx.x - kFirstPromoWarp * 32);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    KernelClock kclock{0, 0};
    if (blockIdx.x == 0 && threadIdx.x == 0)
        kclock = kernel_clock_begin();

    const int num_kb = p.K / BK;
    int total_tiles;
    if constexpr (GROUPED)
        total_tiles = tile_start[p.G];
    else
        total_tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    const volatile SplitRun *run = &s_run;

    if (warp < kFirstPromoWarp) {
        regs_dec<40>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- TMA producer
            uint32_t c = 0;
            uint32_t ab_issued = 0, sb_issued = 0;  // chunks whose operand / scale loads are in flight or landed
            bool ok = true;
            Item it;
            for (int j = 0; ok && item_of<SPLIT_OK>(j, blockIdx.x, gridDim.x, total_tiles, num_kb, run, it); ++j) {
                const Tile tl = tile_of<BN, GROUPED>(it.t, p, tile_start);
                for (int kb = it.kb0; kb < it.kb1; ++kb, ++c) {
                    const int s = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, ERR_TIMEOUT_PRODUCER, &s_abort)) {
                        ok = false;
                        break;
                    }
                    ab_issued = c + 1;
                    mbar_arrive_expect_tx(bar_full + 8 * s, L::A_BYTES + L::B_BYTES);
                    tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmA, kb * BK, tl.m0, bar_full + 8 * s);
                    if constexpr (SWIGLU) {  // gate block, then up block (128-row boxes)
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, kb * BK, tl.brow0, bar_full + 8 * s);
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES + 128 * BK, &tmB, kb * BK, tl.brow0 + p.N,
                                    bar_full + 8 * s);
                    } else {
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, kb * BK, tl.brow0, bar_full + 8 * s);
                    }
                    if constexpr (BMODE == 1) {
                        const int q = c % SB_STAGES;
                        if (!mbar_wait(bar_sbempty + 8 * q, ((c / SB_STAGES) & 1) ^ 1, ERR_TIMEOUT_PRODUCER,
                                       &s_abort)) {
                            ok = false;
                            break;
                        }
                        sb_issued = c + 1;
                        // the A row scales ride on the same barrier (rows past M are not copied)
                        uint32_t sab = p.sa_smem ? static_cast<uint32_t>(min(BM, p.M - tl.m0)) * 4u : 0u;
                        if (sab != 0 &&
                            !dbg_ok(sab % 16 == 0 && tl.m0 + sab / 4 <= p.ldsa && kb < p.K / BK, DBG_GEMM_SCALE_A))
                            sab = 0;
                        mbar_arrive_expect_tx(bar_sbfull + 8 * q, L::SBROW_BYTES + sab);
                        tma_load_2d(sbase + L::OFF_SBROW + q * L::SBROW_BYTES, &tmSB, tl.n0, kb,
                                    bar_sbfull + 8 * q);
                        if (sab != 0)
                            bulk_load(sbase + L::OFF_SAROW + q * L::SAROW_BYTES,
                                      p.sa + static_cast<int64_t>(kb) * p.ldsa + tl.m0, sab, bar_sbfull + 8 * q);
                    }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA exits
                for (uint32_t d = (ab_issued > STAGES ? ab_issued - STAGES : 0); d < ab_issued; ++d)
                    mbar_wait(bar_full + 8 * (d % STAGES), (d / STAGES) & 1, ERR_TIMEOUT_PRODUCER, nullptr, 100000000ull);
                for (uint32_t d = (sb_issued > SB_STAGES ? sb_issued - SB_STAGES : 0); d < sb_issued; ++d)
                    mbar_wait(bar_sbfull + 8 * (d % SB_STAGES), (d / SB_STAGES) & 1, ERR_TIMEOUT_PRODUCER, nullptr,
                              100000000ull);
            }
        } else if ((warp == 1 || warp == 3) && lane == 0) {
            // -------------------------------------------------------- MMA issuers
            const uint32_t mine = (warp == 1) ? 0u : 1u;  // chunk parity this thread issues
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            uint32_t c = 0;
            bool ok = true;
            Item it;
            for (int j = 0; ok && item_of<SPLIT_OK>(j, blockIdx.x, gridDim.x, total_tiles, num_kb, run, it); ++j) {
                for (int kb = it.kb0; kb < it.kb1; ++kb, ++c) {
                    if ((c & 1u) != mine)
                        continue;
                    const int s = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    const int b = c % NTMEM;
                    const uint32_t tph = (c / NTMEM) & 1;
                    // The operands are normally in place long before the partial
                    // buffer is free: wait for them first, so that the MMAs go out
                    // as soon as the promotion releases the buffer (the loop's
                    // critical path).  Same-box A/B, FFN GEMM at equal clock:
                    // 2786-2847 -> 3089-3138 TFLOP/s-at-2032-MHz.
                    if (!mbar_wait(bar_full + 8 * s, ph, ERR_TIMEOUT_MMA, &s_abort) ||
                        !mbar_wait(bar_tempty + 8 * b, tph ^ 1, ERR_TIMEOUT_MMA, &s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sdesc_k128_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = sdesc_k128_sw128(sbase + L::OFF_B + s * L::B_BYTES);
                    const uint32_t d_tmem = tmem_base + b * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)  // +32 bytes of K = +2 in the address field
                        mma_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                    mma_commit(bar_tfull + 8 * b);
                }
            }
            if (!ok) {
                // wait for this thread's last committed chain before TMEM is released
                uint32_t d = c;
                while (d > 0 && ((d - 1) & 1u) != mine)
                    --d;
                if (d > 0) {
                    --d;
                    mbar_wait(bar_tfull + 8 * (d % NTMEM), (d / NTMEM) & 1, ERR_TIMEOUT_MMA, nullptr, 100000000ull);
                }
            }
        }
    } else {
        regs_inc<L::PROMO_REGS>();
        // ------------------------------------------------------------ promotion + epilogue
        constexpr int CPW = L::CPW;
        constexpr int NP = L::NP;
        const int pw = warp - kFirstPromoWarp;
        const int quarter = warp & 3;
        const int grp = pw >> 2;
        const int row = quarter * 32 + lane;
        const int col0 = grp * CPW;
        const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t *epi = smem + L::OFF_EPI + pw * 2048;
        const float *sbrow_smem = reinterpret_cast<const float *>(smem + L::OFF_SBROW);

        uint32_t c = 0;
        uint32_t tcount = 0;  // tiles finished (SwiGLU exchange phase)
        (void)tcount;
        bool ok = true;

        // K split: a TAIL piece waits for the flag of CTA b+1's partial (one
        // thread waits, the others wait on it); a HEAD piece, once its partial
        // is in C, publishes it to CTA b-1 when every promotion warp's stores
        // are visible at GPU scope.
        auto split_tail_wait = [&]() -> bool {
            bool got = true;
            if (threadIdx.x == kFirstPromoWarp * 32) {
                got = flag_wait(p.sk_flags + blockIdx.x, p.sk_epoch, ERR_TIMEOUT_SPLIT, &s_abort);
                if (got)
                    mbar_arrive(bar_sktail);
            }
            got = mbar_wait(bar_sktail, 0, ERR_TIMEOUT_SPLIT, &s_abort);
            return __all_sync(0xFFFFFFFFu, got);
        };
        auto split_head_publish = [&]() {
            __threadfence();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_skhead);
            if (threadIdx.x == kFirstPromoWarp * 32) {
                if (mbar_wait(bar_skhead, 0, ERR_TIMEOUT_SPLIT, &s_abort) && dbg_ok(blockIdx.x >= 1, DBG_GEMM_SPLIT))
                    flag_release(p.sk_flags + blockIdx.x - 1, p.sk_epoch);
            }
        };
        (void)split_tail_wait;
        (void)split_head_publish;

        // ---------------------------------- per-row scales (every tile width)
        // The partial is read from TMEM in the 16x256b shape, pieces of 16
        // registers: a thread holds rows quarter*32 + 8i + lane/4 (i = 0..3)
        // and the column pairs col0 + 8k + 2(lane%4) (k < CPW/8) of its
        // warpgroup's CPW columns, acc[AR*i + 2k + e].  At CPW = 128 it then
        // needs 32 of the chunk's B scales instead of 128.  With one row and 128 columns per
        // thread every lane read all 128 as 16-byte shared-memory broadcasts,
        // about five wavefronts each, and those loads kept the shared-memory
        // data pipe 59% busy (ncu, Wgrad GEMM) beside the MMAs' operand reads.
        // Wgrad GEMM 0.404 -> 0.379 ms, bit-identical.  (Pieces of 32
        // registers spilled and ran slower.)  The buffer is freed after the
        // last fold: freeing it after the last loads but before the last folds
        // let the next chunk's MMAs corrupt this chunk's values (in about one
        // launch in 20 of the Wgrad workload, found by repeating it and
        // comparing outputs bit for bit; never after the last fold).
        constexpr bool RS16 = (BMODE == 1);
        constexpr int KP = L::CPW / 8;   // column pairs per row of a thread
        constexpr int AR = 2 * KP;       // accumulators per row of a thread
        constexpr int NQ = L::CPW / 32;  // 32-column quarters of a warpgroup's columns
        auto item_rs16 = [&](const Tile &tl, const Item &it) -> bool {
            const int t4 = lane >> 2, p2 = (lane & 3) * 2;
            const int rbase = tl.m0 + quarter * 32 + t4;  // rows rbase + 8i
            float acc[4 * AR];
#pragma unroll
            for (int j = 0; j < 4 * AR; ++j)
                acc[j] = 0.0f;
            if constexpr (SPLIT_OK) {
                if (it.mode == ITEM_TAIL) {
                    if (!split_tail_wait())
                        return false;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = rbase + 8 * i;
                        if (m >= tl.m_end)
                            continue;
                        const float *crow = reinterpret_cast<const float *>(p.C) + static_cast<int64_t>(m) * p.ldc;
#pragma unroll
                        for (int k = 0; k < KP; ++k) {
                            const int n = tl.n0 + col0 + 8 * k + p2;
                            if (n < p.N && dbg_ok(m < p.M && n + 2 <= p.N && p.N <= p.ldc, DBG_GEMM_SPLIT)) {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(crow + n));
                                acc[AR * i + 2 * k] = v.x;
                                acc[AR * i + 2 * k + 1] = v.y;
                            }
                        }
                    }
                }
            }
            auto ld_sa4 = [&](int kb, float (&v)[4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = min(rbase + 8 * i, p.M - 1);
                    v[i] = (kb < it.kb1 && dbg_ok(m >= 0 && m < p.ldsa, DBG_GEMM_SCALE_A))
                               ? __ldg(p.sa + static_cast<int64_t>(kb) * p.ldsa + m)
                               : 0.0f;
                }
            };
            // acc(i, k) += fl32(sa_i * sb_k) * P(i, k), two columns per instruction,
            // each rounded as the scalar mul and fmaf would be; piece (h, q):
            // rows 16h + 8ri + lane/4, column pairs k = 4q + j (j = 0..3)
            auto fold4 = [&](int h, int q, const uint32_t(&r)[16], const float2(&sbp)[4], const uint64_t(&sa2)[4]) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint64_t sb2;
                    asm("mov.b64 %0, {%1, %2};" : "=l"(sb2) : "f"(sbp[jj].x), "f"(sbp[jj].y));
#pragma unroll
                    for (int ri = 0; ri < 2; ++ri) {
                        const int i = 2 * h + ri, k = 4 * q + jj;
                        uint64_t sc2, a2, p2v;
                        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(sc2) : "l"(sa2[i]), "l"(sb2));
                        asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "f"(acc[AR * i + 2 * k]), "f"(acc[AR * i + 2 * k + 1]));
                        asm("mov.b64 %0, {%1, %2};" : "=l"(p2v) : "r"(r[4 * jj + 2 * ri]), "r"(r[4 * jj + 2 * ri + 1]));
                        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a2) : "l"(sc2), "l"(p2v));
                        asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[AR * i + 2 * k]), "=f"(acc[AR * i + 2 * k + 1]) : "l"(a2));
                    }
                }
            };
            const float *sarow_smem = reinterpret_cast<const float *>(smem + L::OFF_SAROW) + quarter * 32 + t4;
            for (int kb = it.kb0; kb < it.kb1; ++kb) {
                // the row scales come with the chunk's scale slot (a bulk copy
                // by the producer, issued chunks ahead) or, where that copy is
                // not allowed, straight from global memory; the global loads
                // stood on the loop's critical path (knocked out in a probe
                // copy, the Wgrad GEMM ran 12% faster)
                float sa[4];
                if (!p.sa_smem)
                    ld_sa4(kb, sa);
                const int b = c % NTMEM;
                const uint32_t tph = (c / NTMEM) & 1;
                const int s = c % SB_STAGES;
                bool got = mbar_wait(bar_tfull + 8 * b, tph, ERR_TIMEOUT_CONSUMER, &s_abort);
                got = got && mbar_wait(bar_sbfull + 8 * s, (c / SB_STAGES) & 1, ERR_TIMEOUT_CONSUMER, &s_abort);
                if (!__all_sync(0xFFFFFFFFu, got))
                    return false;
                if (p.sa_smem) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        sa[i] = sarow_smem[s * BM + 8 * i];
                }
                tc_fence_after();
                if (!dbg_ok(b * BN + col0 + L::CPW <= L::TMEM_COLS, DBG_GEMM_TMEM))
                    return false;
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * BN + col0;
                const float *sbr = sbrow_smem + s * BN + col0 + p2;
                uint64_t sa2[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm("mov.b64 %0, {%1, %1};" : "=l"(sa2[i]) : "f"(sa[i]));
                uint32_t ra[16], rb[16];
                tmem_ld16x4(tb, ra);                 // rows +0, +8;   columns 0..31
                tmem_ld16x4(tb + (16u << 16), rb);   // rows +16, +24; columns 0..31
                tmem_ld_wait_regs16x2(ra, rb);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    float2 sbp[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        sbp[jj] = *reinterpret_cast<const float2 *>(sbr + 32 * q + 8 * jj);
                    fold4(0, q, ra, sbp, sa2);
                    if (q < NQ - 1)
                        tmem_ld16x4(tb + 32 * (q + 1), ra);
                    fold4(1, q, rb, sbp, sa2);
                    if (q < NQ - 1) {
                        tmem_ld16x4(tb + (16u << 16) + 32 * (q + 1), rb);
                        tmem_ld_wait_regs16x2(ra, rb);
                    }
                }
                // freed after the last fold (see the race noted above)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_tempty + 8 * b);
                    mbar_arrive(bar_sbempty + 8 * s);
                }
                ++c;
            }
            // epilogue: two columns per store, straight from the registers
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = rbase + 8 * i;
                if (m >= tl.m_end)
                    continue;
#pragma unroll
                for (int k = 0; k < KP; ++k) {
                    const int n = tl.n0 + col0 + 8 * k + p2;
                    if (n < p.N && dbg_ok(m < p.M && n + 2 <= p.N && p.N <= p.ldc, DBG_GEMM_STORE)) {
                        const int64_t off = static_cast<int64_t>(m) * p.ldc + n;
                        if constexpr (OUT_F32)
                            *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.C) + off) =
                                make_float2(acc[AR * i + 2 * k], acc[AR * i + 2 * k + 1]);
                        else
                            *reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(p.C) + off) =
                                pack_bf16x2(acc[AR * i + 2 * k], acc[AR * i + 2 * k + 1]);
                    }
                }
            }
            if constexpr (SPLIT_OK) {
                if (it.mode == ITEM_HEAD)
                    split_head_publish();
            }
            return true;
        };
        (void)item_rs16;

        Item it;
        for (int j = 0; ok && item_of<SPLIT_OK>(j, blockIdx.x, gridDim.x, total_tiles, num_kb, run, it); ++j) {
            const Tile tl = tile_of<BN, GROUPED>(it.t, p, tile_start);
            if constexpr (RS16) {
                if (!item_rs16(tl, it))
                    ok = false;
                continue;
            }
            const int m_row = min(tl.m0 + row, p.M - 1);
            const float *sa_ptr = p.sa + m_row;
            // CPW columns starting at a multiple of CPW never straddle a
            // 128-column scale block
            int nb = (tl.n0 + col0) / 128;
            nb = min(nb, (p.N - 1) / 128);
            if constexpr (SWIGLU)
                nb = tl.n0 / 128;  // gate block; the up block is N/128 rows further
            const float *sb_ptr = tl.sbp + static_cast<int64_t>(nb) * p.ldsb;
            const float *sbu_ptr = sb_ptr + static_cast<int64_t>(p.N / 128) * p.ldsb;

            float acc[CPW];
#pragma unroll
            for (int j = 0; j < CPW; ++j)
                acc[j] = 0.0f;
            if constexpr (SPLIT_OK) {
                if (it.mode == ITEM_TAIL) {
                    // continue from the accumulators CTA b+1 stored for this
                    // tile's first chunks
                    if (!split_tail_wait()) {
                        ok = false;
                        break;
                    }
                    const int m = tl.m0 + row;
                    if (m < tl.m_end) {
                        const float *crow = reinterpret_cast<const float *>(p.C) + static_cast<int64_t>(m) * p.ldc;
#pragma unroll
                        for (int j = 0; j < CPW; j += 4) {
                            const int n = tl.n0 + col0 + j;
                            if (n < p.N && dbg_ok(m < p.M && n + 4 <= p.N && p.N <= p.ldc, DBG_GEMM_SPLIT)) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(crow + n));
                                acc[j] = v.x;
                                acc[j + 1] = v.y;
                                acc[j + 2] = v.z;
                                acc[j + 3] = v.w;
                            }
                        }
                    }
                }
            }

            // One K chunk: wait for its partial, read it from TMEM, release the
            // buffer, fold it into acc with the chunk's scales.
            auto promote = [&](float sa_v, float sb_v, float sbu_v) -> bool {
                const int b = c % NTMEM;
                const uint32_t tph = (c / NTMEM) & 1;
                const int s = c % STAGES;
                // every lane waits, then the warp reconverges before the
                // .sync.aligned TMEM loads
                bool got = mbar_wait(bar_tfull + 8 * b, tph, ERR_TIMEOUT_CONSUMER, &s_abort);
                if constexpr (BMODE == 1)
                    got = got && mbar_wait(bar_sbfull + 8 * (c % SB_STAGES), (c / SB_STAGES) & 1, ERR_TIMEOUT_CONSUMER,
                                           &s_abort);
                if (!__all_sync(0xFFFFFFFFu, got))
                    return false;
                tc_fence_after();
                // TMEM column of 32-column piece pc of this thread's columns
                auto pcol = [&](int pc) -> uint32_t {
                    if constexpr (SWIGLU)
                        return static_cast<uint32_t>(pc < 2 ? grp * 64 + pc * 32 : 128 + grp * 64 + (pc - 2) * 32);
                    else
                        return static_cast<uint32_t>(col0 + pc * 32);
                };
                const uint32_t tbase = tmem_base + t_lane + b * BN;
                if (!dbg_ok(b * BN + pcol(NP - 1) + 32 <= L::TMEM_COLS, DBG_GEMM_TMEM))
                    return false;
                const float sc = sa_v * sb_v;
                const float scu = SWIGLU ? sa_v * sbu_v : sc;  // up-block scale (SwiGLU)
                (void)scu;
                const float *sbr = sbrow_smem + (c % SB_STAGES) * BN + col0;
                (void)sbr;

                auto fold = [&](int pc, const uint32_t(&cur)[32]) {
                    if constexpr (BMODE == 0) {
                        // fmaf(sc, P, acc) two columns per instruction (each lane rounds
                        // exactly as the scalar fmaf)
                        const float scp = (SWIGLU && pc >= 2) ? scu : sc;
                        uint64_t sc2;
                        asm("mov.b64 %0, {%1, %1};" : "=l"(sc2) : "f"(scp));
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            uint64_t a2, p2;
                            asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "f"(acc[pc * 32 + j]), "f"(acc[pc * 32 + j + 1]));
                            asm("mov.b64 %0, {%1, %2};" : "=l"(p2) : "r"(cur[j]), "r"(cur[j + 1]));
                            asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a2) : "l"(sc2), "l"(p2));
                            asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[pc * 32 + j]), "=f"(acc[pc * 32 + j + 1]) : "l"(a2));
                        }
                    } else {
                        uint64_t sa2;
                        asm("mov.b64 %0, {%1, %1};" : "=l"(sa2) : "f"(sa_v));
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const float4 sb4 = *reinterpret_cast<const float4 *>(sbr + pc * 32 + j);
                            fold_rowscale2(acc[pc * 32 + j + 0], acc[pc * 32 + j + 1], sa2, sb4.x, sb4.y, cur[j + 0],
                                           cur[j + 1]);
                            fold_rowscale2(acc[pc * 32 + j + 2], acc[pc * 32 + j + 3], sa2, sb4.z, sb4.w, cur[j + 2],
                                           cur[j + 3]);
                        }
                    }
                };
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar_tempty + 8 * b);
                };

                uint32_t ra[32], rb[32];
                if constexpr (NP == 2) {
                    // both loads in flight, one wait, release, then fold
                    tmem_ld32(tbase + pcol(0), ra);
                    tmem_ld32(tbase + pcol(1), rb);
                    tmem_ld_wait_regs2(ra, rb);
                    release();
                    fold(0, ra);
                    fold(1, rb);
                } else {
                    // (per-row scales take the 16x256b path above)
                    // four loads, each overlapped with the fold of the previous one
                    tmem_ld32(tbase + pcol(0), ra);
                    tmem_ld_wait_regs(ra);
#pragma unroll
                    for (int pc = 0; pc < NP; ++pc) {
                        uint32_t(&cur)[32] = (pc & 1) ? rb : ra;
                        uint32_t(&nxt)[32] = (pc & 1) ? ra : rb;
                        if (pc + 1 < NP)
                            tmem_ld32(tbase + pcol(pc + 1), nxt);
                        fold(pc, cur);
                        if (pc + 1 < NP) {
                            tmem_ld_wait_regs(nxt);
                            if (pc + 2 == NP)
                                release();  // the last piece is in registers
                        }
                    }
                }
                if constexpr (BMODE == 1) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar_sbempty + 8 * (c % SB_STAGES));
                }
                ++c;
                return true;
            };

            // Scales are loaded two chunks ahead into two fixed registers per
            // operand (the chunk loop is unrolled by two), so each load has a
            // whole chunk pair to land and no register copy waits on it.
            const int kend = it.kb1;
            auto ld_sa = [&](int kb) {
                return (kb < kend && dbg_ok(m_row >= 0 && m_row < p.M && m_row < p.ldsa, DBG_GEMM_SCALE_A))
                           ? __ldg(sa_ptr + static_cast<int64_t>(kb) * p.ldsa)
                           : 0.0f;
            };
            // block row nb of B's scales (per expert when grouped): rows of B / 128, rounded up
            const int sb_rows = (p.b_rows + 127) / 128;
            auto ld_sb = [&](int kb) {
                return (BMODE == 0 && kb < kend && dbg_ok(nb >= 0 && nb < sb_rows && kb < p.ldsb, DBG_GEMM_SCALE_B))
                           ? __ldg(sb_ptr + kb)
                           : 0.0f;
            };
            auto ld_sbu = [&](int kb) {
                return (SWIGLU && kb < kend && dbg_ok(nb + p.N / 128 < sb_rows, DBG_GEMM_SCALE_B))
                           ? __ldg(sbu_ptr + kb)
                           : 0.0f;
            };
            int kb = it.kb0;
            float sa0 = ld_sa(kb), sb0 = ld_sb(kb), sa1 = ld_sa(kb + 1), sb1 = ld_sb(kb + 1);
            float su0 = ld_sbu(kb), su1 = ld_sbu(kb + 1);
            for (; kb + 1 < kend; kb += 2) {
                if (!promote(sa0, sb0, su0)) {
                    ok = false;
                    break;
                }
                sa0 = ld_sa(kb + 2);
                sb0 = ld_sb(kb + 2);
                su0 = ld_sbu(kb + 2);
                if (!promote(sa1, sb1, su1)) {
                    ok = false;
                    break;
                }
                sa1 = ld_sa(kb + 3);
                sb1 = ld_sb(kb + 3);
                su1 = ld_sbu(kb + 3);
            }
            if (ok && kb < kend && !promote(sa0, sb0, su0))
                ok = false;
            if (!ok)
                break;

            if constexpr (SWIGLU) {
                // ------------------------------------------------ SwiGLU + 1x128 quantisation
                // h = silu(g) * u for this thread's 64 channels (acc[0..63] gate,
                // acc[64..127] up), in FP32 with an IEEE divide
                float am = 0.0f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float g = acc[i];
                    const float h = __fdiv_rn(g, 1.0f + expf(-g)) * acc[64 + i];
                    acc[i] = h;
                    am = fmaxf(am, fabsf(h));
                }
                // the row's other 64 channels belong to the other warpgroup
                float *xch = reinterpret_cast<float *>(smem + L::OFF_XCH) + (tcount & 1) * 256;
                xch[grp * 128 + row] = am;
                mbar_arrive(bar_xch);
                const bool got = mbar_wait(bar_xch, tcount & 1, ERR_TIMEOUT_CONSUMER, &s_abort);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    ok = false;
                    break;
                }
                am = fmaxf(am, xch[(grp ^ 1) * 128 + row]);
                const float scale = am == 0.0f ? 1.0f : __fdiv_rn(am, 448.0f);
                // codes E4M3(h / scale), staged 32 rows x 64 bytes per warp
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t w[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float *h = &acc[j * 16 + q4 * 4];
                        w[q4] = e4m3x2(__fdiv_rn(h[0], scale), __fdiv_rn(h[1], scale)) |
                                (e4m3x2(__fdiv_rn(h[2], scale), __fdiv_rn(h[3], scale)) << 16);
                    }
                    if (dbg_ok(lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16) + 16 <= 2048, DBG_GEMM_EPI_SMEM))
                        *reinterpret_cast<uint4 *>(epi + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                }
                __syncwarp();
                const int grow0 = tl.m0 + quarter * 32;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int idx = lane + 32 * i;
                    const int r = idx >> 2, j = idx & 3;
                    const uint4 v = *reinterpret_cast<const uint4 *>(epi + r * 64 + ((j ^ ((r >> 1) & 3)) * 16));
                    const int m = grow0 + r;
                    if (m < tl.m_end && dbg_ok(m < p.M && tl.n0 + grp * 64 + j * 16 + 16 <= p.N && p.N <= p.ldc,
                                               DBG_GEMM_SWIGLU_STORE))
                        *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.C) + static_cast<int64_t>(m) * p.ldc +
                                                   tl.n0 + grp * 64 + j * 16) = v;
                }
                __syncwarp();
                if (grp == 0 && tl.m0 + row < tl.m_end &&
                    dbg_ok(tl.n0 / 128 < p.N / 128 && tl.m0 + row < p.lds_out, DBG_GEMM_SWIGLU_STORE))
                    p.s_out[static_cast<int64_t>(tl.n0 / 128) * p.lds_out + tl.m0 + row] = scale;
                ++tcount;
            } else {
                // ---------------------------------------------------------- epilogue
                // Each round stages 32 rows x 64 bytes through this warp's 2 KB
                // buffer (16-byte chunks XOR-swizzled by row pair, so that the
                // row-wise writes and the row-contiguous read-back are both free
                // of bank conflicts), then stores with row/column masks.
                const int grow0 = tl.m0 + quarter * 32;
                constexpr int COLS_PER_ROUND = OUT_F32 ? 16 : 32;
                constexpr int ELEMS_PER_CHUNK = OUT_F32 ? 4 : 8;
#pragma unroll
                for (int g = 0; g < CPW / COLS_PER_ROUND; ++g) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float *a = &acc[g * COLS_PER_ROUND + j * ELEMS_PER_CHUNK];
                        uint4 v;
                        if constexpr (OUT_F32) {
                            v = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                           __float_as_uint(a[3]));
                        } else {
                            v = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                                           pack_bf16x2(a[6], a[7]));
                        }
                        if (dbg_ok(lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16) + 16 <= 2048, DBG_GEMM_EPI_SMEM))
                            *reinterpret_cast<uint4 *>(epi + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) = v;
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int idx = lane + 32 * i;
                        const int r = idx >> 2, j = idx & 3;
                        const uint4 v = *reinterpret_cast<const uint4 *>(epi + r * 64 + ((j ^ ((r >> 1) & 3)) * 16));
                        const int m = grow0 + r;
                        const int n = tl.n0 + col0 + g * COLS_PER_ROUND + j * ELEMS_PER_CHUNK;
                        if (m < tl.m_end && n < p.N &&
                            dbg_ok(m < p.M && n + ELEMS_PER_CHUNK <= p.N && p.N <= p.ldc, DBG_GEMM_STORE)) {
                            const int64_t off = static_cast<int64_t>(m) * p.ldc + n;
                            if constexpr (OUT_F32)
                                *reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.C) + off) = v;
                            else
                                *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.C) + off) = v;
                        }
                    }
                    __syncwarp();
                }
                if constexpr (SPLIT_OK) {
                    if (it.mode == ITEM_HEAD)  // the partial is in C
                        split_head_publish();
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        kernel_clock_end(kclock);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace fp8bs
