// quant.cuh -- BF16 -> E4M3 tile quantisers (V3 report §6.1: 1x128 tiles
// for activations, 128x128 blocks for weights, scales computed online).
//
// Every kernel reads BF16 with 16-byte loads, takes the tile amax with the
// BF16 magnitude maximum (exact for finite inputs), forms the scale
// amax / 448 with an IEEE single-precision divide (1.0 for an all-zero tile)
// and each code as E4M3_RNE_sat(x / scale), with the codes identical to those
// of the IEEE single-precision quotient (see Markstein2 below).  The
// power-of-two variant rounds the scale up to 2^e and scales exactly.
// All grids are persistent: a CTA walks tiles with a stride of gridDim.x.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace quant {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Magnitude maximum of two BF16 pairs, lane-wise: the magnitude of each lane
// of the result is max(|a|, |b|) (its sign bit is meaningless, clear it with
// 0x7FFF7FFF before use).  One instruction per pair, exact for every finite
// input including subnormals.
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// magnitude maximum of the 8 BF16 values of a 16-byte group, as a pair (signs unspecified)
__device__ __forceinline__ uint32_t amax8(const uint4 &v)
{
    return absmax2(absmax2(v.x, v.y), absmax2(v.z, v.w));
}

__device__ __forceinline__ float pair_max_to_f32(uint32_t m2)
{
    m2 &= 0x7FFF7FFFu;
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    return __uint_as_float(m << 16);
}

__device__ __forceinline__ float tile_scale(float amax)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Power-of-two (UE8M0) scale 2^e of a tile: e is the smallest integer with
// amax <= 448 * 2^e = 1.75 * 2^(8+e).  With amax = 1.m * 2^E that is E - 8,
// or E - 7 when 1.m > 1.75; kept >= -127 (UE8M0's range); 0 for amax 0.
__device__ __forceinline__ float pow2_scale(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    const uint32_t b = __float_as_uint(amax);
    int E;
    uint32_t m;
    if (b >> 23) {
        E = static_cast<int>(b >> 23) - 127;
        m = b & 0x7FFFFFu;
    } else {  // subnormal: normalise
        const int p = 31 - __clz(b);
        E = p - 149;
        m = (b << (23 - p)) & 0x7FFFFFu;
    }
    const int e = max(E - 8 + (m > 0x600000u ? 1 : 0), -127);
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// 2^-e of a power-of-two scale 2^e (e in [-127, 127))
__device__ __forceinline__ float pow2_inverse(float s)
{
    const uint32_t f = __float_as_uint(s) >> 23;
    return f ? __uint_as_float((254u - f) << 23) : __uint_as_float(0x7F000000u);
}

// codes of BF16 pair word w scaled by a power of two (exact products)
__device__ __forceinline__ uint32_t codes_pow2(uint32_t w, float inv)
{
    return e4m3x2(bf16lo(w) * inv, bf16hi(w) * inv);
}

// x / s for the two values of a BF16 pair, by Markstein's division
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s)
// taken once per tile, q0 = RN(x r), the remainder t = q0 s - x (one fused
// multiply-add) and q = RN(q0 - t r) -- four floating-point operations per
// value pair, issued two values at a time (f32x2), instead of a full IEEE
// divide.  q can differ from the IEEE quotient in its last bit (near
// underflow), but its E4M3 code never does: fp8bs_selftest_division encodes
// both for every BF16 amax and every BF16 x with |x| <= amax (about 2^31
// pairs) and finds no difference.  (RN(x r) alone is not enough: its codes
// differ for about 3e4 of those pairs.)  The remainder is taken as q0 s - x,
// the negative of Markstein's x - q0 s, and subtracted: the same exact value
// and the same rounding for every nonzero x, and for x = +-0 the quotient
// keeps x's sign (x - q0 s would be +0 for both zeros and lose it), so the
// codes carry every input's sign with no further step.  The low and high
// value may have different scales (two columns of the transposed
// quantiser).  Scales below 2^-100 (reciprocal near overflow) take the IEEE
// divide instead.
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ bool markstein_ok(float s) { return s >= 0x1p-100f; }

struct Markstein2 {
    uint64_t r2, nr2, s2;  // RN(1/s), -RN(1/s), s for the low and high value
    __device__ __forceinline__ Markstein2(float s_lo, float s_hi)
    {
        const float r_lo = __frcp_rn(s_lo), r_hi = __frcp_rn(s_hi);
        r2 = pack2(r_lo, r_hi);
        nr2 = pack2(-r_lo, -r_hi);
        s2 = pack2(s_lo, s_hi);
    }
    // with the reciprocals RN(1/s) already formed
    __device__ __forceinline__ Markstein2(float s_lo, float s_hi, float r_lo, float r_hi)
    {
        r2 = pack2(r_lo, r_hi);
        nr2 = pack2(-r_lo, -r_hi);
        s2 = pack2(s_lo, s_hi);
    }
    // quotients of the two values of BF16 pair word w (low half first)
    __device__ __forceinline__ void quot(uint32_t w, float &q_lo, float &q_hi) const
    {
        const uint64_t x2 = pack2(bf16lo(w), bf16hi(w));
        const uint64_t m1 = 0xBF800000BF800000ull;  // (-1, -1)
        uint64_t nx2, q0, t, q;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(nx2) : "l"(x2), "l"(m1));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(r2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(q0), "l"(s2), "l"(nx2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(t), "l"(nr2), "l"(q0));
        unpack2(q, q_lo, q_hi);
    }
    // E4M3 codes of the pair, low value in the low byte (signs of zeros kept)
    __device__ __forceinline__ uint32_t codes(uint32_t w) const
    {
        float lo, hi;
        quot(w, lo, hi);
        return e4m3x2(lo, hi);
    }
};

// codes of BF16 pair word w by the IEEE divide (scales below 2^-100)
__device__ __forceinline__ uint32_t codes_ieee(uint32_t w, float s_lo, float s_hi)
{
    return e4m3x2(__fdiv_rn(bf16lo(w), s_lo), __fdiv_rn(bf16hi(w), s_hi));
}

// four codes (bytes 0 .. 3) from two 16-bit code pairs
__device__ __forceinline__ uint32_t join4(uint32_t c0, uint32_t c1) { return __byte_perm(c0, c1, 0x5410); }

__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Tiles of 128 rows x 128 contiguous columns (one K chunk).  Four lanes share
// a row (8 rows per warp instruction, so the per-row amax, scale and
// reciprocal cost a quarter of what 16 lanes per row would); lane j of a
// row owns the 16-byte column groups j, j+4, j+8, j+12, so each load
// instruction reads 64 contiguous bytes per row and each code store writes
// one full 32-byte sector per row.  A thread holds two rows (64 apart):
// eight 16-byte loads in flight.
//   kBlock = false: one scale per row per chunk (1x128 tiles), reduced over
//                   the row's 4 lanes; s[kb*lds + m].
//   kBlock = true : one scale per 128x128 block, reduced over the CTA;
//                   s[mb*lds + kb].
// row_map (1x128 only, may be null): output row m reads input row
// row_map[m] (a gather, e.g. tokens into expert order); a mapped row outside
// [0, src_rows) reads as zeros.
// Tile order: kb fastest, so neighbouring CTAs read neighbouring columns.
// ---------------------------------------------------------------------------
struct RowsArgs {
    const uint16_t *x;
    int64_t M, K, ldx;
    uint8_t *q;
    int64_t ldq;
    float *s;
    int64_t lds;
    const int32_t *row_map;  // 1x128 only, may be null (see above)
    int64_t src_rows;
};

__host__ __device__ inline int64_t rows_tiles(const RowsArgs &a) { return ((a.M + 127) / 128) * (a.K / 128); }

// one 128 x 128 tile (index `tile`, kb fastest) of the quantisation above
template <bool kBlock, bool kPow2>
__device__ __forceinline__ void rows_tile(const RowsArgs &a, int64_t tile, uint32_t *red)
{
    const uint16_t *__restrict__ x = a.x;
    const int64_t M = a.M, K = a.K, ldx = a.ldx, ldq = a.ldq, lds = a.lds;
    uint8_t *__restrict__ q = a.q;
    float *__restrict__ s = a.s;
    const int32_t *__restrict__ row_map = a.row_map;
    const int64_t src_rows = a.src_rows;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int j = lane & 3;                       // column-group phase within the row
    const int rw = (tid >> 5) * 8 + (lane >> 2);  // 0..63
    const int64_t nkb = K / 128;
    {
        const int64_t kb = tile % nkb;
        const int64_t m0 = (tile / nkb) * 128;
        uint4 v[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t m = m0 + rw + 64 * rr;
            int64_t src = m;
            bool ok = m < M;
            if (!kBlock && row_map != nullptr && ok) {
                src = row_map[m];
                ok = src >= 0 && src < src_rows;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[rr][i] = (ok && dbg_ok(src >= 0 && src < (row_map ? src_rows : M) &&
                                             kb * 128 + (j + 4 * i) * 8 + 8 <= K && K <= ldx,
                                         DBG_QROWS_LOAD))
                               ? ldg_stream(x + src * ldx + kb * 128 + (j + 4 * i) * 8)
                               : make_uint4(0, 0, 0, 0);
        }
        uint32_t am[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
            am[rr] = absmax2(absmax2(amax8(v[rr][0]), amax8(v[rr][1])), absmax2(amax8(v[rr][2]), amax8(v[rr][3])));
        float sc[2];
        if constexpr (!kBlock) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                uint32_t a = am[rr];
                a = absmax2(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
                a = absmax2(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
                sc[rr] = kPow2 ? pow2_scale(pair_max_to_f32(a)) : tile_scale(pair_max_to_f32(a));
            }
        } else {
            uint32_t a = absmax2(am[0], am[1]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                a = absmax2(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            if (lane == 0)
                red[tid >> 5] = a;
            __syncthreads();
            uint32_t b = red[0];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w)
                b = absmax2(b, red[w]);
            sc[0] = sc[1] = kPow2 ? pow2_scale(pair_max_to_f32(b)) : tile_scale(pair_max_to_f32(b));
            __syncthreads();  // red[] is rewritten by the next tile
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t m = m0 + rw + 64 * rr;
            if (m < M) {
                uint2 c[4];
                if constexpr (kPow2) {
                    const float inv = pow2_inverse(sc[rr]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 &x = v[rr][i];
                        c[i].x = __byte_perm(codes_pow2(x.x, inv), codes_pow2(x.y, inv), 0x5410);
                        c[i].y = __byte_perm(codes_pow2(x.z, inv), codes_pow2(x.w, inv), 0x5410);
                    }
                } else if (markstein_ok(sc[rr])) {
                    const Markstein2 d(sc[rr], sc[rr]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 &x = v[rr][i];
                        c[i].x = join4(d.codes(x.x), d.codes(x.y));
                        c[i].y = join4(d.codes(x.z), d.codes(x.w));
                    }
                } else {
                    const float sv = sc[rr];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 &x = v[rr][i];
                        c[i].x = join4(codes_ieee(x.x, sv, sv), codes_ieee(x.y, sv, sv));
                        c[i].y = join4(codes_ieee(x.z, sv, sv), codes_ieee(x.w, sv, sv));
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (dbg_ok(kb * 128 + (j + 4 * i) * 8 + 8 <= K && K <= ldq, DBG_QROWS_STORE))
                        *reinterpret_cast<uint2 *>(q + m * ldq + kb * 128 + (j + 4 * i) * 8) = c[i];
                if (!kBlock && j == 0 && dbg_ok(kb < nkb && m < lds, DBG_QROWS_SCALE))
                    s[kb * lds + m] = sc[rr];
            }
        }
        if (kBlock && tid == 0 && dbg_ok(m0 < M && kb < nkb && kb < lds, DBG_QROWS_SCALE))
            s[(m0 / 128) * lds + kb] = sc[0];
    }
}

template <bool kBlock, bool kPow2 = false>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const RowsArgs a)
{
    __shared__ uint32_t red[kThreads / 32];
    grid_launch_dependents();  // a GEMM launched next may set up meanwhile
    const int64_t ntiles = rows_tiles(a);
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
        rows_tile<kBlock, kPow2>(a, tile, red);
}

// An activation (1x128 tiles) and a weight (128x128 blocks) in one launch:
// the tiles of both form one persistent work list, so two small tensors
// keep the whole GPU busy together instead of one after the other.
template <bool kPow2>
__global__ void __launch_bounds__(kThreads) quant_pair_kernel(const RowsArgs act, const RowsArgs wt)
{
    __shared__ uint32_t red[kThreads / 32];
    grid_launch_dependents();  // a GEMM launched next may set up meanwhile
    const int64_t ta = rows_tiles(act), tw = rows_tiles(wt);
    for (int64_t tile = blockIdx.x; tile < ta + tw; tile += gridDim.x) {
        if (tile < ta)
            rows_tile<false, kPow2>(act, tile, red);
        else
            rows_tile<true, kPow2>(wt, tile - ta, red);
    }
}

// ---------------------------------------------------------------------------
// Tiles whose codes come out transposed.  A CTA takes 128 rows x 128
// contiguous columns of x [R][ldx]: one TMA copy brings the tile into shared
// memory, and the next tile's copy is issued as soon as every thread holds
// this one in registers (after the tile's first CTA barrier), so it lands
// while this tile is quantised and stored.  Loading the next tile into
// registers instead needed 80 registers and so one CTA per SM fewer, which
// cost as much as the overlap gained; the copy needs no registers (Wgrad X
// operand 76.1-77.6 -> 67.6 us, dY 26.7-28.5 -> 24.6-25.0 us, same bits).
// A thread holds two 4-row x 8-column pieces (rows 4g .. 4g+3 for g = its
// row group and g + 16), read from the tile with 16-byte shared loads (each
// warp instruction reads two full 256-byte rows).  Its codes are transposed
// in registers (byte permutes: one
// 32-bit word = 4 consecutive rows of one column) and stored as words into a
// [128 columns][32 words] shared tile whose word index is XOR-swizzled with
// twice the column's 8-group, so that every store and every 16-byte read is
// free of bank conflicts; the tile then leaves as 128-byte row segments of
// qt [C][ldqt] (qt[c*ldqt + r] is the code of x[r][c]).
//   kBlock = false: one scale per column per 128 rows (the 1x128 tiles of a
//                   weight-gradient operand, which run along tokens);
//                   s[rb*lds + c].
//   kBlock = true : one scale per 128x128 block (weights), also written
//                   transposed: s[rb*lds + cb] (may be null) and
//                   st[cb*ldst + rb]; q [R][ldq] receives the untransposed
//                   codes too unless null.
// Rows past R (kBlock, R % 16 == 0) and 8-column groups past C arrive as
// zeros (the copy's fill) and are never written.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t out[4])
{
    // a_i holds row i, byte j = column j; out[j] holds column j, byte i = row i
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a2, a3, 0x5140);
    const uint32_t t2 = __byte_perm(a0, a1, 0x7362), t3 = __byte_perm(a2, a3, 0x7362);
    out[0] = __byte_perm(t0, t1, 0x5410);
    out[1] = __byte_perm(t0, t1, 0x7632);
    out[2] = __byte_perm(t2, t3, 0x5410);
    out[3] = __byte_perm(t2, t3, 0x7632);
}

// Dynamic shared memory of quant_t_kernel: the 128 x 128 BF16 input tile
// (loaded by TMA), plus slack for its 128-byte alignment.
constexpr int kQtTileBytes = 128 * 128 * 2;
constexpr int kQtDynSmem = kQtTileBytes + 128;

template <bool kBlock>
__global__ void __launch_bounds__(kThreads, 4) quant_t_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const uint16_t *__restrict__ x, int64_t R, int64_t C,
                                                           int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                           uint8_t *__restrict__ qt, int64_t ldqt,
                                                           float *__restrict__ s, int64_t lds,
                                                           float *__restrict__ st, int64_t ldst)
{
    __shared__ __align__(16) uint32_t qs[128 * 32];
    __shared__ __align__(16) uint4 red[kThreads / 32][16];
    // 1x128 mode: the tile's 128 column scales and their reciprocals, formed once
    // per tile by warp 0 (every warp needs the same 128)
    __shared__ __align__(16) float col_s[128], col_r[128];
    __shared__ __align__(8) uint64_t tbar;
    __shared__ int t_abort;
    extern __shared__ __align__(128) uint8_t qt_dyn[];
    grid_launch_dependents();  // a GEMM launched next may set up meanwhile
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cg = lane & 15;                   // 8-column group of the tile
    const int g0 = warp * 2 + (lane >> 4);      // 4-row group (and g0 + 16)
    const int64_t nrb = (R + 127) / 128, ncb = (C + 127) / 128;
    const int64_t ntiles = nrb * ncb;
    (void)x;
    (void)ldx;

    // the input tile: TMA fills it (zeros past R and C) one tile ahead
    const uint32_t xt = (smem_addr(qt_dyn) + 127u) & ~127u;
    const uint8_t *xtp = qt_dyn + (xt - smem_addr(qt_dyn));
    const uint32_t bar = smem_addr(&tbar);
    if (tid == 0) {
        t_abort = 0;
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int64_t t) {
        mbar_arrive_expect_tx(bar, kQtTileBytes);
        tma_load_2d(xt, &tmX, static_cast<int32_t>((t % ncb) * 128), static_cast<int32_t>((t / ncb) * 128), bar);
    };
    if (tid == 0 && blockIdx.x < ntiles)
        issue(blockIdx.x);
    uint32_t ph = 0;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t cb = tile % ncb, rb = tile / ncb;
        const int64_t r0 = rb * 128, c0 = cb * 128;
        const bool colok = c0 + cg * 8 < C;
        // bounded; after a give-up every later wait returns at once and the
        // tiles come out as zeros (the error word says so)
        const bool landed = mbar_wait(bar, ph, ERR_TIMEOUT_CONSUMER, &t_abort);
        ph ^= 1;
        uint4 v[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = (g0 + 16 * u) * 4 + i;
                v[u][i] = landed ? *reinterpret_cast<const uint4 *>(xtp + row * 256 + cg * 16) : make_uint4(0, 0, 0, 0);
            }
        // the next tile is loaded once every thread holds this one (after the
        // tile's first CTA barrier below)
        auto issue_next = [&]() {
            if (tid == 0 && tile + gridDim.x < ntiles && t_abort == 0) {
                fence_proxy_async_smem();
                issue(tile + gridDim.x);
            }
        };

        // magnitude maximum of each column pair over this thread's 8 rows
        uint4 m4 = v[0][0];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = (u == 0 ? 1 : 0); i < 4; ++i) {
                m4.x = absmax2(m4.x, v[u][i].x);
                m4.y = absmax2(m4.y, v[u][i].y);
                m4.z = absmax2(m4.z, v[u][i].z);
                m4.w = absmax2(m4.w, v[u][i].w);
            }
        float sc[8], rc[8];
        if constexpr (!kBlock) {
            m4.x = absmax2(m4.x, __shfl_xor_sync(0xFFFFFFFFu, m4.x, 16));
            m4.y = absmax2(m4.y, __shfl_xor_sync(0xFFFFFFFFu, m4.y, 16));
            m4.z = absmax2(m4.z, __shfl_xor_sync(0xFFFFFFFFu, m4.z, 16));
            m4.w = absmax2(m4.w, __shfl_xor_sync(0xFFFFFFFFu, m4.w, 16));
            if (lane < 16)
                red[warp][cg] = m4;
            __syncthreads();
            issue_next();
            if (warp == 0) {
                // lane l: columns 4l .. 4l+3 (two BF16 pair words of group l/2)
                const int gq = lane >> 1, hw = lane & 1;
                const uint4 r0 = red[0][gq];
                uint32_t ma = hw ? r0.z : r0.x, mb = hw ? r0.w : r0.y;
#pragma unroll
                for (int w = 1; w < kThreads / 32; ++w) {
                    const uint4 o = red[w][gq];
                    ma = absmax2(ma, hw ? o.z : o.x);
                    mb = absmax2(mb, hw ? o.w : o.y);
                }
                ma &= 0x7FFF7FFFu;
                mb &= 0x7FFF7FFFu;
                const float s4[4] = {tile_scale(__uint_as_float((ma & 0xFFFFu) << 16)),
                                     tile_scale(__uint_as_float(ma & 0xFFFF0000u)),
                                     tile_scale(__uint_as_float((mb & 0xFFFFu) << 16)),
                                     tile_scale(__uint_as_float(mb & 0xFFFF0000u))};
                *reinterpret_cast<float4 *>(&col_s[4 * lane]) = make_float4(s4[0], s4[1], s4[2], s4[3]);
                *reinterpret_cast<float4 *>(&col_r[4 * lane]) =
                    make_float4(__frcp_rn(s4[0]), __frcp_rn(s4[1]), __frcp_rn(s4[2]), __frcp_rn(s4[3]));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + 4 * lane + j < C && dbg_ok(rb < nrb && c0 + 4 * lane + j < lds, DBG_QT_SCALE))
                        s[rb * lds + c0 + 4 * lane + j] = s4[j];
            }
            __syncthreads();
            const float4 sa4 = *reinterpret_cast<const float4 *>(&col_s[cg * 8]);
            const float4 sb4 = *reinterpret_cast<const float4 *>(&col_s[cg * 8 + 4]);
            const float4 ra4 = *reinterpret_cast<const float4 *>(&col_r[cg * 8]);
            const float4 rb4 = *reinterpret_cast<const float4 *>(&col_r[cg * 8 + 4]);
            sc[0] = sa4.x, sc[1] = sa4.y, sc[2] = sa4.z, sc[3] = sa4.w;
            sc[4] = sb4.x, sc[5] = sb4.y, sc[6] = sb4.z, sc[7] = sb4.w;
            rc[0] = ra4.x, rc[1] = ra4.y, rc[2] = ra4.z, rc[3] = ra4.w;
            rc[4] = rb4.x, rc[5] = rb4.y, rc[6] = rb4.z, rc[7] = rb4.w;
        } else {
            uint32_t a = absmax2(absmax2(m4.x, m4.y), absmax2(m4.z, m4.w));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                a = absmax2(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            if (lane == 0)
                red[warp][0].x = a;
            __syncthreads();
            issue_next();
            uint32_t b = red[0][0].x;
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w)
                b = absmax2(b, red[w][0].x);
            const float sb = tile_scale(pair_max_to_f32(b));
            const float rb_ = __frcp_rn(sb);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                sc[j] = sb, rc[j] = rb_;
            if (tid == 0) {
                if (s && dbg_ok(cb < lds, DBG_QT_SCALE))
                    s[rb * lds + cb] = sb;
                if (dbg_ok(rb < ldst, DBG_QT_SCALE))
                    st[cb * ldst + rb] = sb;
            }
        }

        // codes; straight rows out, transposed words into the shared tile
        uint32_t lo[2][4], hi[2][4];
        float smin = sc[0];
#pragma unroll
        for (int j = 1; j < 8; ++j)
            smin = fminf(smin, sc[j]);
        if (markstein_ok(smin)) {
            const Markstein2 d0(sc[0], sc[1], rc[0], rc[1]), d1(sc[2], sc[3], rc[2], rc[3]),
                d2(sc[4], sc[5], rc[4], rc[5]), d3(sc[6], sc[7], rc[6], rc[7]);
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 &x = v[u][i];
                    lo[u][i] = join4(d0.codes(x.x), d1.codes(x.y));
                    hi[u][i] = join4(d2.codes(x.z), d3.codes(x.w));
                }
        } else {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 &x = v[u][i];
                    lo[u][i] = join4(codes_ieee(x.x, sc[0], sc[1]), codes_ieee(x.y, sc[2], sc[3]));
                    hi[u][i] = join4(codes_ieee(x.z, sc[4], sc[5]), codes_ieee(x.w, sc[6], sc[7]));
                }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int g = g0 + 16 * u;
            if (kBlock && q != nullptr && colok) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t r = r0 + g * 4 + i;
                    if (r < R && dbg_ok(c0 + cg * 8 + 8 <= ldq, DBG_QT_STORE))
                        *reinterpret_cast<uint2 *>(q + r * ldq + c0 + cg * 8) = make_uint2(lo[u][i], hi[u][i]);
                }
            }
            uint32_t cw[8];
            transpose4x4(lo[u][0], lo[u][1], lo[u][2], lo[u][3], cw);
            transpose4x4(hi[u][0], hi[u][1], hi[u][2], hi[u][3], cw + 4);
            const int wsw = g ^ (2 * cg);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                if (dbg_ok(wsw >= 0 && wsw < 32, DBG_QT_SMEM))
                    qs[(cg * 8 + cc) * 32 + wsw] = cw[cc];
        }
        __syncthreads();

        // transposed tile out: 128 columns x 8 chunks of 16 rows
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + kThreads * i;
            const int c = idx >> 3, ch = idx & 7;
            const int f = 2 * (c >> 3);
            const int widx = c * 32 + ((4 * ch) ^ (f & 28));
            uint4 w4 = dbg_ok(widx >= 0 && widx + 4 <= 128 * 32, DBG_QT_SMEM)
                           ? *reinterpret_cast<const uint4 *>(&qs[widx])
                           : make_uint4(0, 0, 0, 0);
            if (f & 2)
                w4 = make_uint4(w4.z, w4.w, w4.x, w4.y);
            if (c0 + c < C && r0 + ch * 16 < R && dbg_ok(r0 + ch * 16 + 16 <= ldqt, DBG_QT_STORE))
                *reinterpret_cast<uint4 *>(qt + (c0 + c) * ldqt + r0 + ch * 16) = w4;
        }
    }
}

// Exhaustive check of the quantisers' division (Markstein2) against the IEEE
// divide over the whole BF16 domain of the quantisers: block = one positive finite BF16 amax
// (0x0001 .. 0x7F7F), threads = every BF16 x with |x| <= amax, both signs
// (x and -x form one pair word).  counts[0] += values whose E4M3 codes
// differ, counts[1] += values whose single-precision quotients differ in
// value (Markstein path only; -0 and +0 count as equal).
__global__ void selftest_division_kernel(unsigned long long *counts)
{
    const uint32_t abits = blockIdx.x + 1;  // 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(abits << 16);
    const float s = tile_scale(amax);
    const bool fast = markstein_ok(s);
    const Markstein2 d(s, s);
    unsigned long long bad_code = 0, bad_quot = 0;
    for (uint32_t xb = threadIdx.x; xb <= abits; xb += blockDim.x) {
        const uint32_t w = xb | ((xb | 0x8000u) << 16);  // low: +x, high: -x
        const float i_lo = __fdiv_rn(bf16lo(w), s), i_hi = __fdiv_rn(bf16hi(w), s);
        const uint32_t icodes = e4m3x2(i_lo, i_hi);
        // the quantisers' path: Markstein's division, or the IEEE divide
        const uint32_t codes = fast ? d.codes(w) : codes_ieee(w, s, s);
        if (fast) {
            float q_lo, q_hi;
            d.quot(w, q_lo, q_hi);
            bad_quot += (q_lo != i_lo) + (q_hi != i_hi);
        }
        bad_code += ((codes & 0xFF) != (icodes & 0xFF)) + ((codes >> 8) != (icodes >> 8));
    }
    for (int o = 16; o >= 1; o >>= 1) {
        bad_code += __shfl_xor_sync(0xFFFFFFFFu, bad_code, o);
        bad_quot += __shfl_xor_sync(0xFFFFFFFFu, bad_quot, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (bad_code)
            atomicAdd(&counts[0], bad_code);
        if (bad_quot)
            atomicAdd(&counts[1], bad_quot);
    }
}

// Element-wise conversion with the quantisers' E4M3 rounding (diagnostic).
__global__ void encode_kernel(const float *__restrict__ x, uint8_t *__restrict__ q, int64_t n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 2;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 2; i < n; i += stride) {
        if (i + 1 < n) {
            const uint32_t c = e4m3x2(x[i], x[i + 1]);
            q[i] = static_cast<uint8_t>(c & 0xFF);
            q[i + 1] = static_cast<uint8_t>(c >> 8);
        } else {
            q[i] = static_cast<uint8_t>(e4m3x2(x[i], 0.0f) & 0xFF);
        }
    }
}

}  // namespace quant
}  // namespace fp8bs
