// mx.cuh -- the power-of-two (UE8M0) scale variant of the block-scaled GEMM
// on the tensor cores' own block scaling: tcgen05.mma kind::mxf8f6f4
// .block_scale applies one UE8M0 scale per row of A and per column of B to
// every 32-wide K block inside the MMA and accumulates the whole K in FP32 in
// tensor memory, so there is no promotion pass at all.  (The pages' method
// scales by amax/448 in FP32, which the hardware cannot apply; this variant
// rounds the scales up to powers of two -- the quantisers' _ue8m0 entry
// points -- and changes the numerics accordingly.)
//
// Scale factors live in TMEM.  For a 128-row operand the scale of row r sits
// in lane r % 32 (the same in each of the four 32-lane quarters), column
// r / 32, and byte j of that 32-bit word serves K block j of a 128-wide K
// group (the instruction descriptor's scale-factor id picks the byte); a
// 256-row B uses eight columns the same way.  The 1x128 / 128x128 tiles give
// one scale per row per 128 K, so all four bytes of a word are equal.
//
// CTA (persistent, one per SM), tile 128 x BN, 512 threads:
//   warp 0       TMA producer (A, B stages as in gemm.cuh)
//   warp 1       MMA issuer: four MMAs per 128-K chunk, one commit per chunk
//                (frees the stage and its scale slot), one per tile (the
//                accumulator is complete)
//   warps 4..7   scale writers: per chunk, the UE8M0 bytes of the chunk's
//                A rows and B columns into the stage's TMEM scale slot
//   warps 8..15  epilogue, two warpgroups of BN/2 columns each: an
//                accumulator to BF16 / FP32 in global memory
// TMEM: NACC accumulators of BN columns, then the scale slots (4 columns for
// A + 8 for B per stage).  BN = 192 fits two accumulators, so a tile's
// epilogue overlaps the next tile's MMAs; BN = 256 fits one.  All waits are
// bounded.
#pragma once
#include <cstdint>

#include "gemm.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace mx {

constexpr int BM = 128, BK = 128;
constexpr int THREADS = 512;
constexpr int A_BYTES = BM * BK;
constexpr int EPI_WARPS = 8;
constexpr int EPI_BYTES = EPI_WARPS * 2048;
constexpr int SF_COLS = 12;  // per stage: 4 for A, 8 for B

template <int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int NACC = (BN <= 192) ? 2 : 1;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SF_COL0 = NACC * BN;
    static constexpr int FIT = (gemm::kMaxSmem - EPI_BYTES - 2048) / (A_BYTES + B_BYTES);
    static constexpr int STAGES = FIT < 6 ? FIT : 6;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NBAR = 3 * STAGES + 2 * NACC;  // full, empty, sffull; tfull, tempty
    static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_TMEMSLOT + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(BN % 32 == 0 && BN <= 256, "tile width");
    static_assert(SF_COL0 + STAGES * SF_COLS <= 512, "TMEM columns");
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(ALLOC <= gemm::kMaxSmem, "shared memory");
};

struct Params {
    const float *sa;  // [K/128][ldsa], powers of two
    int64_t ldsa;
    const float *sb;  // [ceil(N/128)][ldsb], powers of two
    int64_t ldsb;
    void *C;
    int64_t ldc;
    int M, N, K;
    int group_m;  // raster group (M tiles sweeping N together)
};

// UE8M0 byte of a power-of-two FP32 scale (its exponent field; 2^-127 is the
// subnormal 0x00400000, field 0), repeated in all four bytes
__device__ __forceinline__ uint32_t ue8m0_word(float s) { return (__float_as_uint(s) >> 23) * 0x01010101u; }

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Instruction descriptor for kind::mxf8f6f4 with UE8M0 scales: B scale id
// (bits 4-5), A and B E4M3 (7-9, 10-12 = 0), K-major (15, 16 = 0), N >> 3
// (17-22), scale format UE8M0 (23), M >> 4 (24-28), A scale id (29-30).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, int sf_id)
{
    return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}

struct Tile {
    int m0, n0;
};

template <int BN>
__device__ __forceinline__ Tile tile_of(int t, const Params &p)
{
    const int num_n = (p.N + BN - 1) / BN;
    const int num_m = (p.M + BM - 1) / BM;
    const int per_group = p.group_m * num_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(num_m - first_m, p.group_m);
    const int local = t - g * per_group;
    Tile r;
    r.m0 = (first_m + local % gsize) * BM;
    r.n0 = (local / gsize) * BN;
    return r;
}

template <int BN, bool OUT_F32>
__global__ void __launch_bounds__(THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p)
{
    using L = Cfg<BN>;
    constexpr int STAGES = L::STAGES, NACC = L::NACC, B_BYTES = L::B_BYTES, SF_COL0 = L::SF_COL0;
    constexpr int OFF_A = L::OFF_A, OFF_B = L::OFF_B, OFF_EPI = L::OFF_EPI, OFF_BAR = L::OFF_BAR;
    extern __shared__ uint8_t dyn_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dyn_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar_full = sbase + OFF_BAR;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_sffull = bar_empty + 8 * STAGES;
    const uint32_t bar_tfull = bar_sffull + 8 * STAGES;
    const uint32_t bar_tempty = bar_tfull + 8 * NACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_TMEMSLOT);
    // raised by the first wait of this CTA that gives up (see mbar_wait)
    __shared__ int s_abort;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sffull + 8 * s, 128);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, EPI_WARPS * 32);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    // the set-up above overlaps the end of the kernel that produced the inputs
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    KernelClock kclock{0, 0};
    if (blockIdx.x == 0 && threadIdx.x == 0)
        kclock = kernel_clock_begin();
    const int num_kb = p.K / BK;
    const int total_tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------------- TMA producer
            uint32_t c = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const Tile tl = tile_of<BN>(t, p);
                for (int kb = 0; kb < num_kb; ++kb, ++c) {
                    const int s = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, ERR_TIMEOUT_PRODUCER, &s_abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_full + 8 * s, A_BYTES + B_BYTES);
                    tma_load_2d(sbase + OFF_A + s * A_BYTES, &tmA, kb * BK, tl.m0, bar_full + 8 * s);
                    tma_load_2d(sbase + OFF_B + s * B_BYTES, &tmB, kb * BK, tl.n0, bar_full + 8 * s);
                }
            }
            if (!ok) {  // let copies already issued land before the CTA exits
                for (uint32_t d = (c > STAGES ? c - STAGES : 0); d < c; ++d)
                    mbar_wait(bar_full + 8 * (d % STAGES), (d / STAGES) & 1, ERR_TIMEOUT_PRODUCER, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------------- MMA issuer
            uint32_t c = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++tcount) {
                // accumulator b must have been drained by the epilogue of the tile NACC before
                const int b = tcount % NACC;
                if (!mbar_wait(bar_tempty + 8 * b, ((tcount / NACC) & 1) ^ 1, ERR_TIMEOUT_MMA, &s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kb = 0; kb < num_kb; ++kb, ++c) {
                    const int s = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    if (!mbar_wait(bar_full + 8 * s, ph, ERR_TIMEOUT_MMA, &s_abort) ||
                        !mbar_wait(bar_sffull + 8 * s, ph, ERR_TIMEOUT_MMA, &s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sdesc_k128_sw128(sbase + OFF_A + s * A_BYTES);
                    const uint64_t bdesc = sdesc_k128_sw128(sbase + OFF_B + s * B_BYTES);
                    const uint32_t sfa = tmem_base + SF_COL0 + s * SF_COLS;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_mx(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mx(BM, BN, k), sfa, sfa + 4,
                               (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                    if (kb == num_kb - 1)
                        mma_commit(bar_tfull + 8 * b);
                }
            }
            if (!ok && c > 0)  // the last committed chain completes before TMEM is freed
                mbar_wait(bar_empty + 8 * ((c - 1) % STAGES), ((c - 1) / STAGES) & 1, ERR_TIMEOUT_MMA, nullptr,
                          100000000ull);
        }
    } else if (warp >= 4 && warp < 8) {
        // -------------------------------------------------------------- scale writers
        const int q = warp & 3;
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        uint32_t c = 0;
        bool ok = true;
        // At the start of each tile the scale writers prefetch the next
        // tile's scale rows into L2 (and the first tile's at kernel start):
        // each chunk's scales are one dependent global load ahead of the
        // MMAs, and a cold load from HBM made the writers gate the MMAs.
        const int ptid = (warp - 4) * 32 + lane;  // 0..127
        auto prefetch_scales = [&](int t) {
            if (t >= total_tiles)
                return;
            const Tile tn = tile_of<BN>(t, p);
            for (int i = ptid; i < num_kb * 4; i += 128) {
                const int kb = i >> 2;
                const int r = min(tn.m0 + (i & 3) * 32, p.M - 1);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.sa + static_cast<int64_t>(kb) * p.ldsa + r));
            }
            const int nb0 = tn.n0 / 128, nb_last = min((tn.n0 + BN - 1) / 128, (p.N - 1) / 128);
            for (int i = ptid; i < (nb_last - nb0 + 1) * ((num_kb + 31) / 32); i += 128) {
                const int per = (num_kb + 31) / 32;
                const int nb = nb0 + i / per, kb = (i % per) * 32;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.sb + static_cast<int64_t>(nb) * p.ldsb + kb));
            }
        };
        prefetch_scales(blockIdx.x);
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            prefetch_scales(t + gridDim.x);
            const Tile tl = tile_of<BN>(t, p);
            int rows[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                rows[j] = min(tl.m0 + lane + 32 * j, p.M - 1);
            // B column group g (32 columns) lies in one 128-wide scale block
            int nbg[BN / 32];
#pragma unroll
            for (int g = 0; g < BN / 32; ++g)
                nbg[g] = min((tl.n0 + 32 * g) / 128, (p.N - 1) / 128);
            for (int kb = 0; kb < num_kb; ++kb, ++c) {
                const int s = c % STAGES;
                const uint32_t ph = (c / STAGES) & 1;
                const float *sak = p.sa + static_cast<int64_t>(kb) * p.ldsa;
                const uint32_t a0 = ue8m0_word(__ldg(sak + rows[0])), a1 = ue8m0_word(__ldg(sak + rows[1]));
                const uint32_t a2 = ue8m0_word(__ldg(sak + rows[2])), a3 = ue8m0_word(__ldg(sak + rows[3]));
                uint32_t bw[8];
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    bw[g] = (g < BN / 32) ? ue8m0_word(__ldg(p.sb + static_cast<int64_t>(nbg[g < BN / 32 ? g : 0]) * p.ldsb + kb))
                                          : 0x7F7F7F7Fu;
                // the slot is free once the MMAs that read it (chunk c - STAGES) completed
                const bool got = mbar_wait(bar_empty + 8 * s, ph ^ 1, ERR_TIMEOUT_CONSUMER, &s_abort);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t slot = tmem_base + lanes + SF_COL0 + s * SF_COLS;
                tmem_st4(slot, a0, a1, a2, a3);
                tmem_st4(slot + 4, bw[0], bw[1], bw[2], bw[3]);
                tmem_st4(slot + 8, bw[4], bw[5], bw[6], bw[7]);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar_sffull + 8 * s);
            }
        }
    } else if (warp >= 8) {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int half = (warp - 8) >> 2;  // columns [half * BN/2, (half + 1) * BN/2)
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        uint8_t *epi = smem + OFF_EPI + (warp - 8) * 2048;
        uint32_t tcount = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++tcount) {
            const Tile tl = tile_of<BN>(t, p);
            const int b = tcount % NACC;
            const bool got = mbar_wait(bar_tfull + 8 * b, (tcount / NACC) & 1, ERR_TIMEOUT_CONSUMER, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, got))
                break;
            tc_fence_after();
            const int grow0 = tl.m0 + q * 32;
            constexpr int PIECES = BN / 64;  // 32-column pieces of this warp's half
            // one round: 32 rows x 64 bytes staged through the warp's 2 KB
            // (16-byte chunks XOR-swizzled by row pair: conflict-free both
            // ways), then 16-byte stores with row / column masks
            auto stage = [&](const uint32_t *w) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (dbg_ok(lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16) + 16 <= 2048, DBG_MX_EPI_SMEM))
                        *reinterpret_cast<uint4 *>(epi + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) =
                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            };
            auto flush = [&](int n0) {
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int idx = lane + 32 * i;
                    const int rr = idx >> 2, j = idx & 3;
                    const uint4 v = *reinterpret_cast<const uint4 *>(epi + rr * 64 + ((j ^ ((rr >> 1) & 3)) * 16));
                    const int m = grow0 + rr;
                    const int n = n0 + j * (OUT_F32 ? 4 : 8);
                    if (m < p.M && n < p.N && dbg_ok(n + (OUT_F32 ? 4 : 8) <= p.N && p.N <= p.ldc, DBG_MX_STORE)) {
                        const int64_t off = static_cast<int64_t>(m) * p.ldc + n;
                        if constexpr (OUT_F32)
                            *reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.C) + off) = v;
                        else
                            *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.C) + off) = v;
                    }
                }
                __syncwarp();
            };
            if constexpr (!OUT_F32) {
                // Read the whole share as packed BF16 (16 registers a piece;
                // the first piece goes straight to the staging buffer), free
                // the accumulator, then store: the next tile's MMAs run while
                // the stores drain.
                uint32_t packed[PIECES * 16];
#pragma unroll
                for (int pi = 0; pi < PIECES; ++pi) {
                    uint32_t r[32];
                    tmem_ld32(tmem_base + lanes + b * BN + (half * PIECES + pi) * 32, r);
                    gemm::tmem_ld_wait_regs(r);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[pi * 16 + i] = gemm::pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    if (pi == 0)
                        stage(&packed[0]);
                }
                tc_fence_before();
                mbar_arrive(bar_tempty + 8 * b);
                flush(tl.n0 + half * PIECES * 32);
#pragma unroll
                for (int pi = 1; pi < PIECES; ++pi) {
                    stage(&packed[pi * 16]);
                    flush(tl.n0 + (half * PIECES + pi) * 32);
                }
            } else {
                // FP32: a piece at a time (the share does not fit in registers)
#pragma unroll 1
                for (int pi = 0; pi < PIECES; ++pi) {
                    const int pc = half * PIECES + pi;
                    uint32_t r[32];
                    tmem_ld32(tmem_base + lanes + b * BN + pc * 32, r);
                    gemm::tmem_ld_wait_regs(r);
                    if (pi == PIECES - 1) {  // this group's share of the accumulator has been read
                        tc_fence_before();
                        mbar_arrive(bar_tempty + 8 * b);
                    }
                    stage(&r[0]);
                    flush(tl.n0 + pc * 32);
                    stage(&r[16]);
                    flush(tl.n0 + pc * 32 + 16);
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
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace mx
}  // namespace fp8bs
