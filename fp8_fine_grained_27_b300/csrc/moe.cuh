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
// bias.  A fixed order makes the choice reproducible from run to run, and it
// bounds each logit's distance from the exact product by the FP32 error of a
// sequential sum, so that only tokens whose key gap is inside that bound can
// differ from a choice made on exact logits.  A tensor-core dot product would
// leave the accumulation order open.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopk = 16;

// ---------------------------------------------------------------------------
// Logits: a 64-token x 64-expert tile per CTA of 64 threads; a thread owns 8
// tokens x 8 experts (two groups of four, 32 apart, so that every shared-
// memory read of a warp is one wavefront).  Every output accumulates its
// terms in increasing k, one fused multiply-add per term.  The multiply-adds
// run two outputs at a time (fma.rn.f32x2: each lane is an ordinary fmaf),
// pairing (t, e) with (t+1, e+1) and (t, e+1) with (t+1, e), so both
// operands are contiguous pairs in shared memory (one half-swap of the
// expert pair).  The problem gives few threads (one per 64 outputs), so each
// warp keeps 32 independent multiply-adds per step and reads the next
// step's operands during the current one.  K advances 32 at a time through
// double-buffered shared memory: the centroids (k-major) by cp.async, the
// tokens through registers, converted from BF16 and transposed.
// Requires D % 32 == 0.
// ---------------------------------------------------------------------------
constexpr int kLT = 64, kLE = 64, kLK = 32;
constexpr int kXP = kLT + 4;  // row pitch of the token tile (floats)
constexpr int kCP = kLE + 4;  // row pitch of the centroid tile

__device__ __forceinline__ uint64_t swap_halves(uint64_t v)
{
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(hi), "r"(lo));
    return r;
}

__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

__device__ __forceinline__ void lds2(uint64_t &a, uint64_t &b, uint32_t addr)
{
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr) : "memory");
}

__global__ void __launch_bounds__(64) route_logits_kernel(const uint16_t *__restrict__ x, int64_t T, int64_t D,
                                                          int64_t ldx, const float *__restrict__ centT, int64_t ldc,
                                                          int E, float *__restrict__ logits, int *__restrict__ counts)
{
    __shared__ __align__(16) float xs[2][kLK][kXP];
    __shared__ __align__(16) float cs[2][kLK][kCP];
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;  // experts {4tx, 32+4tx} + 0..3, tokens {4ty, 32+4ty} + 0..3
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kLT;
    const int e0 = blockIdx.y * kLE;
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int e = tid; e < E; e += 64)
            counts[e] = 0;  // the selection kernel, next on the stream, counts into it

    // token loader: row tid, 32 BF16 of K per chunk
    const bool xok = t0 + tid < T;
    const uint16_t *xp = x + (t0 + tid) * ldx;
    uint4 xv[4];
    auto fetch_x = [&](int64_t k0) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            xv[i] = xok ? *reinterpret_cast<const uint4 *>(xp + k0 + 8 * i) : make_uint4(0, 0, 0, 0);
    };
    auto stage_x = [&](int b) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xs[b][8 * i + 2 * j][tid] = __uint_as_float(w[j] << 16);
                xs[b][8 * i + 2 * j + 1][tid] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    };
    // centroid loader: 32 rows of K x 16 chunks of 16 bytes (4 experts) per chunk of K;
    // thread: chunk tid % 16 of rows tid / 16 + 4 i
    const int cc = tid & 15, cr = tid >> 4;
    const bool cok = e0 + 4 * cc < E;  // E % 4 == 0: a chunk is wholly in or out
    auto fetch_c = [&](int64_t k0, int b) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = cr + 4 * i;
            const float *src = centT + (k0 + r) * ldc + (cok ? e0 + 4 * cc : 0);
            cp_async16_zfill(smem_addr(&cs[b][r][4 * cc]), src, cok ? 16u : 0u);
        }
    };

    // accd[p][q] = {out(tp, eq), out(tp+1, eq+1)}, accx[p][q] = {out(tp, eq+1), out(tp+1, eq)}
    // for token pair p (tp = 4ty + 2p, p < 2; 32 + 4ty + 2(p-2), p >= 2) and expert pair q likewise
    uint64_t accd[4][4], accx[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            accd[p][q] = accx[p][q] = 0;

    fetch_c(0, 0);
    fetch_x(0);
    stage_x(0);
    cp_async_wait_all();
    __syncthreads();
    int b = 0;
    for (int64_t k0 = 0; k0 < D; k0 += kLK) {
        const bool more = k0 + kLK < D;
        if (more) {  // the next chunk lands while this one is multiplied
            fetch_c(k0 + kLK, b ^ 1);
            fetch_x(k0 + kLK);
        }
        const uint32_t xa = smem_addr(&xs[b][0][4 * ty]), ca = smem_addr(&cs[b][0][4 * tx]);
        uint64_t a[4], c[4];
        lds2(a[0], a[1], xa);
        lds2(a[2], a[3], xa + 128);
        lds2(c[0], c[1], ca);
        lds2(c[2], c[3], ca + 128);
#pragma unroll
        for (int kk = 0; kk < kLK; ++kk) {
            uint64_t an[4], cn[4];
            if (kk + 1 < kLK) {
                const uint32_t xo = xa + (kk + 1) * kXP * 4, co = ca + (kk + 1) * kCP * 4;
                lds2(an[0], an[1], xo);
                lds2(an[2], an[3], xo + 128);
                lds2(cn[0], cn[1], co);
                lds2(cn[2], cn[3], co + 128);
            }
            uint64_t cw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                cw[q] = swap_halves(c[q]);
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    fma2(accd[p][q], a[p], c[q]);
                    fma2(accx[p][q], a[p], cw[q]);
                }
            if (kk + 1 < kLK) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a[i] = an[i];
                    c[i] = cn[i];
                }
            }
        }
        if (more)
            stage_x(b ^ 1);
        cp_async_wait_all();
        __syncthreads();
        b ^= 1;
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float d0, d1, x0, x1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(accd[p][q]));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(accx[p][q]));
            const int64_t ta = t0 + (p < 2 ? 4 * ty + 2 * p : 32 + 4 * ty + 2 * (p - 2)), tb = ta + 1;
            const int ea = e0 + (q < 2 ? 4 * tx + 2 * q : 32 + 4 * tx + 2 * (q - 2)), eb = ea + 1;
            if (ta < T && ea < E)
                logits[ta * E + ea] = d0;
            if (tb < T && eb < E)
                logits[tb * E + eb] = d1;
            if (ta < T && eb < E)
                logits[ta * E + eb] = x0;
            if (tb < T && ea < E)
                logits[tb * E + ea] = x1;
        }
}

// affinity of a logit: 1 / (1 + exp(-l)) in double
__device__ __forceinline__ double affinity(float l) { return 1.0 / (1.0 + exp(-static_cast<double>(l))); }

// The selection key s + b is defined in double.  An FP32 screen decides
// almost every token: with CUDA's expf within 2 ulp, 1 + e and the divide
// correctly rounded and |b| < 4, the FP32 key is within 2^-20 of the exact
// key, so when the k-th and (k+1)-th FP32 keys are more than kScreenGap
// apart the FP32 top-k is the exact top-k (and the double one).  Tokens
// closer than that are decided again from the double keys.
constexpr float kScreenGap = 0x1p-16f;

// warp arg-max over (key desc, index asc)
template <typename F>
__device__ __forceinline__ void warp_argmax(F &bk, int &bi)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const F ok = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ok > bk || (ok == bk && oi < bi)) {
            bk = ok;
            bi = oi;
        }
    }
}

// k rounds of arg-max over this lane's NJ keys; returns the k-th key and the
// (k+1)-th (or -inf when every expert is chosen); chosen[] in pick order.
template <int NJ, typename F>
__device__ __forceinline__ void top_k(const F (&key)[NJ], int lane, int E, int topk, int *chosen, F &kth, F &next)
{
    uint32_t taken = 0;
    kth = next = -INFINITY;
#pragma unroll 1
    for (int r = 0; r <= topk && r < E; ++r) {
        F bk = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && (key[j] > bk || bi == 0x7FFFFFFF)) {
                bk = key[j];
                bi = e;
            }
        }
        warp_argmax(bk, bi);
        if (r == topk) {
            next = bk;
            break;
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        chosen[r] = bi;
        kth = bk;
    }
}

// ---------------------------------------------------------------------------
// Selection: one warp per token; lane i holds experts i, i + 32, ... (NJ per
// lane).  The chosen experts are listed in increasing index order with
// their gates (double affinities, summed in that order).
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
    int chosen[kMaxTopk];
    {
        float key[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            key[j] = (e < E) ? __fdiv_rn(1.0f, 1.0f + expf(-lt[e])) + bias[e] : -INFINITY;
        }
        float kth, next;
        top_k(key, lane, E, topk, chosen, kth, next);
        if (!(kth - next > kScreenGap)) {  // near tie: decide from the double keys
            double dkey[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int e = lane + 32 * j;
                dkey[j] = (e < E) ? affinity(lt[e]) + static_cast<double>(bias[e]) : -INFINITY;
            }
            double dk, dn;
            top_k(dkey, lane, E, topk, chosen, dk, dn);
        }
    }
    // lanes 0 .. topk-1 hold one chosen expert each, in increasing order
    int mine = 0x7FFFFFFF;
    for (int i = 0; i < topk; ++i) {  // rank of chosen[lane] among the chosen
        const int v = chosen[i];
        if (lane < topk) {
            int rank = 0;
            for (int q = 0; q < topk; ++q)
                rank += chosen[q] < v;
            if (rank == lane)
                mine = v;
        }
    }
    const double s_mine = (lane < topk) ? affinity(lt[mine]) : 0.0;
    double sum = 0.0;
    for (int i = 0; i < topk; ++i)
        sum += __shfl_sync(0xFFFFFFFFu, s_mine, i);
    if (lane < topk) {
        sel[t * topk + lane] = mine;
        gate[t * topk + lane] = static_cast<float>(s_mine / sum);
        atomicAdd(&counts[mine], 1);
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
            if (dbg_ok(r >= 0 && r < T * topk, DBG_MOE_GROUP)) {
                token_of_row[r] = static_cast<int32_t>(t);
                row_of[t * topk + slot] = r;
            }
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
            if (!dbg_ok(n + 8 <= ldy, DBG_MOE_COMBINE))
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
        if (dbg_ok(n + 8 <= ldo, DBG_MOE_COMBINE))
            *reinterpret_cast<uint4 *>(out + t * ldo + n) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

}  // namespace moe
}  // namespace fp8bs
