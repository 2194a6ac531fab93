// quant.cuh -- BF16 -> E4M3 tile quantisers (V3 report §6.1: 1x128 tiles
// for activations, 128x128 blocks for weights, scales computed online).
//
// Every kernel reads BF16 with 16-byte loads, takes the tile amax on the
// sign-cleared BF16 bit patterns (for finite inputs their unsigned order is
// the order of magnitudes, so the maximum is exact), forms the scale
// amax / 448 with an IEEE single-precision divide (1.0 for an all-zero tile)
// and each code as E4M3_RNE_sat(x / scale), with the codes identical to those
// of the IEEE single-precision quotient (see Quotient below).
// All grids are persistent: a CTA walks tiles with a stride of gridDim.x.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace quant {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max of the magnitudes held in a 16-byte group of 8 BF16 values, as a pair
// of 16-bit lanes (sign bits cleared).
__device__ __forceinline__ uint32_t amax8(const uint4 &v)
{
    uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
    return __vmaxu2(a, b);
}

__device__ __forceinline__ float pair_max_to_f32(uint32_t m2)
{
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    return __uint_as_float(m << 16);
}

__device__ __forceinline__ float tile_scale(float amax)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// x / s for the two values of a BF16 pair, by Markstein's division
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s)
// taken once per tile, q0 = RN(x r), the remainder e = x - s q0 (one fused
// multiply-add) and q = RN(q0 + e r) -- three floating-point operations per
// value, issued two values at a time (f32x2), instead of a full IEEE divide.
// q can differ from the IEEE quotient in its last bit (near underflow), but
// its E4M3 code never does: fp8bs_selftest_division encodes both for every
// BF16 amax and every BF16 x with |x| <= amax (about 2^31 pairs) and finds no
// difference.  The low and high value may have different scales (two
// columns of the transposed quantiser).  Scales below 2^-100 (reciprocal
// near overflow) take the IEEE divide.
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

struct QuotientPair {
    uint64_t r2, ns2;
    float s_lo, s_hi;
    bool fast;
    __device__ __forceinline__ QuotientPair(float scale_lo, float scale_hi)
    {
        s_lo = scale_lo;
        s_hi = scale_hi;
        fast = scale_lo >= 0x1p-100f && scale_hi >= 0x1p-100f;
        r2 = pack2(__frcp_rn(scale_lo), __frcp_rn(scale_hi));
        ns2 = pack2(-scale_lo, -scale_hi);
    }
    // quotients of the two values of BF16 pair word w (low half first)
    __device__ __forceinline__ void quot(uint32_t w, float &q_lo, float &q_hi) const
    {
        const float x_lo = bf16lo(w), x_hi = bf16hi(w);
        if (fast) {
            const uint64_t x2 = pack2(x_lo, x_hi);
            uint64_t q0, e, q;
            asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(r2));
            asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns2), "l"(x2));
            asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r2), "l"(q0));
            unpack2(q, q_lo, q_hi);
            // s > 0, so a quotient carries x's sign; the correction step
            // would turn -0 into +0, so the sign is restored explicitly
            q_lo = copysignf(q_lo, x_lo);
            q_hi = copysignf(q_hi, x_hi);
        } else {
            q_lo = __fdiv_rn(x_lo, s_lo);
            q_hi = __fdiv_rn(x_hi, s_hi);
        }
    }
    // E4M3 codes of the pair: low value in the low byte
    __device__ __forceinline__ uint32_t codes(uint32_t w) const
    {
        float lo, hi;
        quot(w, lo, hi);
        return e4m3x2(lo, hi);
    }
};

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
// Tile order: kb fastest, so neighbouring CTAs read neighbouring columns.
// ---------------------------------------------------------------------------
template <bool kBlock>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const uint16_t *__restrict__ x, int64_t M,
                                                              int64_t K, int64_t ldx,
                                                              uint8_t *__restrict__ q, int64_t ldq,
                                                              float *__restrict__ s, int64_t lds)
{
    __shared__ uint32_t red[kThreads / 32];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int j = lane & 3;                       // column-group phase within the row
    const int rw = (tid >> 5) * 8 + (lane >> 2);  // 0..63
    const int64_t nkb = K / 128;
    const int64_t ntiles = ((M + 127) / 128) * nkb;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t kb = tile % nkb;
        const int64_t m0 = (tile / nkb) * 128;
        uint4 v[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t m = m0 + rw + 64 * rr;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[rr][i] = (m < M) ? ldg_stream(x + m * ldx + kb * 128 + (j + 4 * i) * 8) : make_uint4(0, 0, 0, 0);
        }
        uint32_t am[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
            am[rr] = __vmaxu2(__vmaxu2(amax8(v[rr][0]), amax8(v[rr][1])), __vmaxu2(amax8(v[rr][2]), amax8(v[rr][3])));
        float sc[2];
        if constexpr (!kBlock) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                uint32_t a = am[rr];
                a = __vmaxu2(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
                a = __vmaxu2(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
                sc[rr] = tile_scale(pair_max_to_f32(a));
            }
        } else {
            uint32_t a = __vmaxu2(am[0], am[1]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                a = __vmaxu2(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            if (lane == 0)
                red[tid >> 5] = a;
            __syncthreads();
            uint32_t b = red[0];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w)
                b = __vmaxu2(b, red[w]);
            sc[0] = sc[1] = tile_scale(pair_max_to_f32(b));
            __syncthreads();  // red[] is rewritten by the next tile
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t m = m0 + rw + 64 * rr;
            if (m < M) {
                const QuotientPair qt(sc[rr], sc[rr]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint2 c;
                    c.x = qt.codes(v[rr][i].x) | (qt.codes(v[rr][i].y) << 16);
                    c.y = qt.codes(v[rr][i].z) | (qt.codes(v[rr][i].w) << 16);
                    *reinterpret_cast<uint2 *>(q + m * ldq + kb * 128 + (j + 4 * i) * 8) = c;
                }
                if (!kBlock && j == 0)
                    s[kb * lds + m] = sc[rr];
            }
        }
        if (kBlock && tid == 0)
            s[(m0 / 128) * lds + kb] = sc[0];
    }
}

// ---------------------------------------------------------------------------
// Tiles of 128 consecutive rows of one column (the token dimension of a
// weight-gradient operand), codes written transposed.  A CTA stages a
// 128-row x 128-column BF16 tile in shared memory (row pitch 65 words: the
// column reads of 32 consecutive rows hit 32 distinct banks), reduces each
// column, encodes into a [128 columns][128 rows] byte tile and writes it out
// with 16-byte coalesced stores.
//   x [T][ldx] (C columns); q [C][ldq] (row k holds the T codes of column k);
//   s [T/128][lds]: scale of tile (tb, k) at s[tb*lds + k].
// ---------------------------------------------------------------------------
constexpr int kColsPitch = 65;  // words per staged row (64 data words + 1)

struct ColsSmem {
    uint32_t xs[128 * kColsPitch];
    uint8_t qs[128 * 128];
    uint32_t red[4][64];
    float sc[128];
};

__global__ void __launch_bounds__(kThreads) quant_cols_kernel(const uint16_t *__restrict__ x, int64_t T,
                                                              int64_t C, int64_t ldx,
                                                              uint8_t *__restrict__ q, int64_t ldq,
                                                              float *__restrict__ s, int64_t lds)
{
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    ColsSmem &sm = *reinterpret_cast<ColsSmem *>(dyn_smem);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t ntb = T / 128;
    const int64_t ncb = (C + 127) / 128;
    const int64_t ntiles = ntb * ncb;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t cb = tile % ncb;
        const int64_t tb = tile / ncb;
        const int64_t t0 = tb * 128, c0 = cb * 128;

        // 1. load 128 rows x 256 bytes, 16 bytes per thread per row
        {
            const int c16 = tid & 15;
            const int rr = tid >> 4;
            uint4 v[8];
            const bool colok = c0 + c16 * 8 < C;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int64_t t = t0 + rr + 16 * p;
                v[p] = colok ? ldg_stream(x + t * ldx + c0 + c16 * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                uint32_t *dst = &sm.xs[(rr + 16 * p) * kColsPitch + c16 * 4];
                dst[0] = v[p].x;
                dst[1] = v[p].y;
                dst[2] = v[p].z;
                dst[3] = v[p].w;
            }
        }
        __syncthreads();

        // 2. column amax: thread -> word column w (2 columns), quarter of the rows
        {
            const int w = tid & 63;
            const int qr = tid >> 6;
            uint32_t a = 0;
#pragma unroll 8
            for (int r = 0; r < 32; ++r)
                a = __vmaxu2(a, sm.xs[(qr * 32 + r) * kColsPitch + w] & 0x7FFF7FFFu);
            sm.red[qr][w] = a;
        }
        __syncthreads();
        if (tid < 64) {
            uint32_t a = __vmaxu2(__vmaxu2(sm.red[0][tid], sm.red[1][tid]),
                                  __vmaxu2(sm.red[2][tid], sm.red[3][tid]));
            const float slo = tile_scale(__uint_as_float((a & 0xFFFFu) << 16));
            const float shi = tile_scale(__uint_as_float(a & 0xFFFF0000u));
            sm.sc[2 * tid] = slo;
            sm.sc[2 * tid + 1] = shi;
            if (c0 + 2 * tid < C) {
                s[tb * lds + c0 + 2 * tid] = slo;
                s[tb * lds + c0 + 2 * tid + 1] = shi;
            }
        }
        __syncthreads();

        // 3. encode: warp -> 8 word columns; lane -> rows lane + 32j
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            const int w = warp * 8 + i;
            const QuotientPair qp(sm.sc[2 * w], sm.sc[2 * w + 1]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = lane + 32 * j;
                const uint32_t word = sm.xs[r * kColsPitch + w];
                const uint32_t c2 = qp.codes(word);
                sm.qs[(2 * w) * 128 + r] = static_cast<uint8_t>(c2 & 0xFF);
                sm.qs[(2 * w + 1) * 128 + r] = static_cast<uint8_t>(c2 >> 8);
            }
        }
        __syncthreads();

        // 4. write the transposed code tile: 128 rows x 8 chunks of 16 bytes
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + kThreads * i;
            const int row = idx >> 3, ch = idx & 7;
            if (c0 + row < C) {
                const uint4 v = *reinterpret_cast<const uint4 *>(&sm.qs[row * 128 + ch * 16]);
                *reinterpret_cast<uint4 *>(q + (c0 + row) * ldq + t0 + ch * 16) = v;
            }
        }
        __syncthreads();
    }
}

// Exhaustive check of QuotientPair against the IEEE divide over the whole
// BF16 domain of the quantisers: block = one positive finite BF16 amax
// (0x0001 .. 0x7F7F), threads = every BF16 x with |x| <= amax, both signs
// (x and -x form one pair word).  counts[0] += values whose E4M3 codes
// differ, counts[1] += values whose single-precision quotients differ.
__global__ void selftest_division_kernel(unsigned long long *counts)
{
    const uint32_t abits = blockIdx.x + 1;  // 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(abits << 16);
    const float s = tile_scale(amax);
    const QuotientPair qp(s, s);
    unsigned long long bad_code = 0, bad_quot = 0;
    for (uint32_t xb = threadIdx.x; xb <= abits; xb += blockDim.x) {
        const uint32_t w = xb | ((xb | 0x8000u) << 16);  // low: +x, high: -x
        float q_lo, q_hi;
        qp.quot(w, q_lo, q_hi);
        const uint32_t codes = qp.codes(w);
        const float i_lo = __fdiv_rn(bf16lo(w), s), i_hi = __fdiv_rn(bf16hi(w), s);
        const uint32_t icodes = e4m3x2(i_lo, i_hi);
        bad_quot += (__float_as_uint(q_lo) != __float_as_uint(i_lo)) + (__float_as_uint(q_hi) != __float_as_uint(i_hi));
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
