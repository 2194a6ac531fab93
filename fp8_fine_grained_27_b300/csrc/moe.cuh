// moe.cuh -- the routed-expert (MoE) chain around the grouped GEMMs
// (V3 report §2 DeepSeekMoE: 256 routed experts, 8 per token, SwiGLU
// experts; §4 aux-loss-free balancing: a sigmoid affinity to each expert's
// centroid, selection by affinity + a per-expert bias, gates from the
// affinities normalised over the selected experts).
//
//   route_logits_kernel   l[t][e] = u_t . c_e in FP32 (CUDA cores)
//   route_select_kernel   top-k of sigmoid(l) + b per token, gates
//   route_group_kernel    rows grouped by expert, tokens in order
//   combine_kernel        y[t] = sum_j gate[t][j] * Y[row_of[t][j]]
//
// The routing decision (an integer) is taken from FP32 logits formed with
// one fused multiply-add per term in increasing k, then a double sigmoid and
// bias; that order is part of the definition, so the choice is reproducible
// bit for bit.  A tensor-core dot product would leave the accumulation order
// open and let near-ties flip.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopk = 16;

// ---------------------------------------------------------------------------
// Logits: a 64-token x 64-expert tile per CTA, 256 threads, 4 x 4 outputs per
// thread.  K advances 32 at a time through shared memory (tokens converted
// from BF16); every output accumulates its terms in increasing k with fmaf.
// Requires D % 32 == 0.
// ---------------------------------------------------------------------------
constexpr int kLT = 64, kLE = 64, kLK = 32, kLPad = 4;

__global__ void __launch_bounds__(256) route_logits_kernel(const uint16_t *__restrict__ x, int64_t T, int64_t D,
                                                           int64_t ldx, const float *__restrict__ cent,
                                                           int64_t ldc, int E, float *__restrict__ logits,
                                                           int *__restrict__ counts)
{
    __shared__ __align__(16) float xs[kLK][kLT + kLPad];
    __shared__ __align__(16) float cs[kLK][kLE + kLPad];
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kLT;
    const int e0 = blockIdx.y * kLE;
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int e = tid; e < E; e += 256)
            counts[e] = 0;  // the selection kernel, next on the stream, counts into it

    // loader mapping: tokens: row tid/4, 8 k from (tid%4)*8; centroids: expert
    // tid/8 (+32), 4 k from (tid%8)*4
    const int xr = tid >> 2, xk = (tid & 3) * 8;
    const int cr = tid >> 3, ck = (tid & 7) * 4;
    const bool xok = t0 + xr < T;
    const bool cok0 = e0 + cr < E, cok1 = e0 + cr + 32 < E;
    const uint16_t *xp = x + (t0 + xr) * ldx + xk;
    const float *cp0 = cent + static_cast<int64_t>(e0 + cr) * ldc + ck;
    const float *cp1 = cent + static_cast<int64_t>(e0 + cr + 32) * ldc + ck;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[i][j] = 0.0f;

    uint4 xv = xok ? *reinterpret_cast<const uint4 *>(xp) : make_uint4(0, 0, 0, 0);
    float4 c0 = cok0 ? *reinterpret_cast<const float4 *>(cp0) : make_float4(0, 0, 0, 0);
    float4 c1 = cok1 ? *reinterpret_cast<const float4 *>(cp1) : make_float4(0, 0, 0, 0);
    for (int64_t k0 = 0; k0 < D; k0 += kLK) {
        __syncthreads();  // the previous chunk's reads are done
        const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xs[xk + 2 * i][xr] = __uint_as_float(w[i] << 16);
            xs[xk + 2 * i + 1][xr] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        cs[ck + 0][cr] = c0.x;
        cs[ck + 1][cr] = c0.y;
        cs[ck + 2][cr] = c0.z;
        cs[ck + 3][cr] = c0.w;
        cs[ck + 0][cr + 32] = c1.x;
        cs[ck + 1][cr + 32] = c1.y;
        cs[ck + 2][cr + 32] = c1.z;
        cs[ck + 3][cr + 32] = c1.w;
        __syncthreads();
        if (k0 + kLK < D) {  // next chunk's loads overlap this chunk's FMAs
            xv = xok ? *reinterpret_cast<const uint4 *>(xp + k0 + kLK) : make_uint4(0, 0, 0, 0);
            c0 = cok0 ? *reinterpret_cast<const float4 *>(cp0 + k0 + kLK) : make_float4(0, 0, 0, 0);
            c1 = cok1 ? *reinterpret_cast<const float4 *>(cp1 + k0 + kLK) : make_float4(0, 0, 0, 0);
        }
#pragma unroll 8
        for (int kk = 0; kk < kLK; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4 *>(&cs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + ty * 4 + i;
        if (t >= T)
            continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E)
                logits[t * E + e] = acc[i][j];
        }
    }
}

// affinity of a logit: 1 / (1 + exp(-l)) in double
__device__ __forceinline__ double affinity(float l) { return 1.0 / (1.0 + exp(-static_cast<double>(l))); }

// ---------------------------------------------------------------------------
// Selection: one warp per token; lane i holds experts i, i + 32, ... (NJ per
// lane).  k rounds of a warp arg-max over (key desc, index asc) pick the
// experts; they are listed in increasing index order with their gates.
// ---------------------------------------------------------------------------
template <int NJ>
__global__ void __launch_bounds__(256) route_select_kernel(const float *__restrict__ logits, int64_t T, int E,
                                                           const float *__restrict__ bias, int topk,
                                                           int32_t *__restrict__ sel, float *__restrict__ gate,
                                                           int *__restrict__ counts)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (t >= T)
        return;
    const float *lt = logits + t * E;
    double key[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? affinity(lt[e]) + static_cast<double>(bias[e]) : -1.0e300;
    }
    uint32_t taken = 0;
    int chosen[kMaxTopk];
#pragma unroll 1
    for (int r = 0; r < topk; ++r) {
        double bk = -1.0e308;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && key[j] > bk) {
                bk = key[j];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const double ok = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        chosen[r] = bi;
    }
    if (lane == 0) {
        // increasing expert order (insertion sort of at most 16 indices)
        for (int i = 1; i < topk; ++i) {
            const int v = chosen[i];
            int j = i - 1;
            while (j >= 0 && chosen[j] > v) {
                chosen[j + 1] = chosen[j];
                --j;
            }
            chosen[j + 1] = v;
        }
        double sum = 0.0;
        for (int i = 0; i < topk; ++i)
            sum += affinity(lt[chosen[i]]);
        for (int i = 0; i < topk; ++i) {
            sel[t * topk + i] = chosen[i];
            gate[t * topk + i] = static_cast<float>(affinity(lt[chosen[i]]) / sum);
            atomicAdd(&counts[chosen[i]], 1);
        }
    }
}

// ---------------------------------------------------------------------------
// Grouping: block e owns expert e.  Its first row is the number of picks of
// lower experts; it scans the tokens in order, 256 at a time, and gives each
// token that picked e the next row (a block-wide prefix count of flags).
// offsets[e] is written by block e, offsets[E] by the last block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_group_kernel(const int32_t *__restrict__ sel, int64_t T, int topk,
                                                          int E, const int *__restrict__ counts,
                                                          int32_t *__restrict__ offsets,
                                                          int32_t *__restrict__ token_of_row,
                                                          int32_t *__restrict__ row_of)
{
    __shared__ int wsum[8];
    __shared__ int base_sh;
    const int e = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int part = 0;
    for (int i = tid; i < e; i += 256)
        part += counts[i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
    if (lane == 0)
        wsum[warp] = part;
    __syncthreads();
    if (tid == 0) {
        int b = 0;
        for (int w = 0; w < 8; ++w)
            b += wsum[w];
        base_sh = b;
        offsets[e] = b;
        if (e == E - 1)
            offsets[E] = b + counts[e];
    }
    __syncthreads();
    int base = base_sh;
    for (int64_t c0 = 0; c0 < T; c0 += 256) {
        const int64_t t = c0 + tid;
        int slot = -1;
        if (t < T)
            for (int j = 0; j < topk; ++j)
                if (sel[t * topk + j] == e)
                    slot = j;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, slot >= 0);
        __syncthreads();  // wsum of the previous chunk has been read
        if (lane == 0)
            wsum[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            before += (w < warp) ? wsum[w] : 0;
            total += wsum[w];
        }
        if (slot >= 0) {
            const int r = base + before + __popc(bal & ((1u << lane) - 1u));
            token_of_row[r] = static_cast<int32_t>(t);
            row_of[t * topk + slot] = r;
        }
        base += total;
    }
}

// ---------------------------------------------------------------------------
// Combine: one thread per 8 output columns of one token; FP32 fused
// multiply-adds over the token's experts in their listed order, BF16 out.
// Rows outside [0, R) contribute nothing (malformed maps cannot read out of
// bounds).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ Y, int64_t ldy, int64_t R,
                                                      const int32_t *__restrict__ row_of,
                                                      const float *__restrict__ gate, int64_t T, int topk,
                                                      int64_t N, uint16_t *__restrict__ out, int64_t ldo)
{
    const int64_t per_tok = N / 8;
    const int64_t total = T * per_tok;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / per_tok;
        const int64_t n = (idx - t * per_tok) * 8;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = 0.0f;
        for (int j = 0; j < topk; ++j) {
            const int32_t r = row_of[t * topk + j];
            if (r < 0 || r >= R)
                continue;
            const float g = gate[t * topk + j];
            const uint4 v = *reinterpret_cast<const uint4 *>(Y + static_cast<int64_t>(r) * ldy + n);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fmaf_rn(g, __uint_as_float(w[i] << 16), acc[2 * i]);
                acc[2 * i + 1] = __fmaf_rn(g, __uint_as_float(w[i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
        }
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)  // low half = even column
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed[i]) : "f"(acc[2 * i + 1]), "f"(acc[2 * i]));
        *reinterpret_cast<uint4 *>(out + t * ldo + n) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

}  // namespace moe
}  // namespace fp8bs
