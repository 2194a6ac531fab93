// fp8bs.cu -- the C ABI of libfp8bs (declared in include/fp8bs.h): argument
// checks, TMA descriptors and kernel launches for the E4M3 quantisers and
// the block-scaled GEMMs.  Single translation unit; sm_103a only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <utility>

#include "../../include/fp8bs.h"
#include "gemm.cuh"
#include "moe.cuh"
#include "mx.cuh"
#include "ptx.cuh"
#include "quant.cuh"

// Library-owned scratch for fp8_moe_route_noalloc: the routing workspace of
// the largest expert count (1024 experts x 4 bytes).  One buffer per device;
// calls that use it on one device must be ordered (one stream, or events).
static constexpr long long kRouteScratchBytes = 4096;
static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];
static_assert(kRouteScratchBytes >= ((fp8bs::moe::kMaxExperts * 4 + 255) / 256) * 256,
              "the static routing scratch must hold the workspace of the largest expert count");

// Flags of the GEMM's K-split last round (one per CTA pair that shares a
// tile): a ring of kSplitRing slot groups of kSplitGroup flags.  Each launch
// takes the next group and its own flag value, so launches in flight at the
// same time on different streams do not share flags (unless more than
// kSplitRing of them are).
static constexpr int kSplitGroup = 256, kSplitRing = 256;
static __device__ uint32_t g_split_flags[kSplitGroup * kSplitRing];

namespace fp8bs {

// A barrier nothing completes, waited on with a short bound: exercises the
// timeout path of every kernel without faulting or hanging.
__global__ void selftest_timeout_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    const uint32_t a = smem_addr(&bar);
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(a, 1);
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(a, 0, ERR_TIMEOUT_SELFTEST, &s_abort, limit_ns);
    __syncthreads();
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    bool sm103 = false;
    int num_sms = 0;
    int quant_rows_ctas = 0;  // resident CTAs per SM, 1x128 and 128x128 kernels
    int quant_block_ctas = 0;
    int quant_cols_ctas = 0;
    int quant_blockt_ctas = 0;
    int quant_pair_ctas = 0;
    unsigned gemm_attr_set = 0;  // bit per GEMM instance: shared-memory attribute applied
    void *route_scratch = nullptr;  // device address of g_route_scratch
    unsigned mx_attr_set = 0;       // bit per block-scaled GEMM instance
    uint32_t *split_flags = nullptr;  // device address of g_split_flags
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8BS_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8BS_ECUDA;
        d.sm103 = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.sm103) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.quant_rows_ctas, quant::quant_rows_kernel<false>,
                                                              quant::kThreads, 0) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.quant_block_ctas, quant::quant_rows_kernel<true>,
                                                              quant::kThreads, 0) != cudaSuccess)
                return FP8BS_ECUDA;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.quant_pair_ctas, quant::quant_pair_kernel<false>,
                                                              quant::kThreads, 0) != cudaSuccess)
                return FP8BS_ECUDA;
            if (cudaFuncSetAttribute(quant::quant_t_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     quant::kQtDynSmem) != cudaSuccess ||
                cudaFuncSetAttribute(quant::quant_t_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     quant::kQtDynSmem) != cudaSuccess)
                return FP8BS_ECUDA;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.quant_cols_ctas, quant::quant_t_kernel<false>,
                                                              quant::kThreads, quant::kQtDynSmem) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.quant_blockt_ctas, quant::quant_t_kernel<true>,
                                                              quant::kThreads, quant::kQtDynSmem) != cudaSuccess)
                return FP8BS_ECUDA;
            if (!g_encode) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                        cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || !fn)
                    return FP8BS_ECUDA;
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
        }
        d.init = true;
    }
    if (!d.sm103)
        return FP8BS_EARCH;
    *out = &d;
    return FP8BS_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

quant::RowsArgs rows_args(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq, float *s,
                          int64_t lds, const int32_t *row_map = nullptr, int64_t src_rows = 0)
{
    return quant::RowsArgs{static_cast<const uint16_t *>(x), M, K, ldx, q, ldq, s, lds, row_map, src_rows};
}

int launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8BS_OK : FP8BS_ECUDA;
}

// 2D tensor map over a row-major matrix: `cols` contiguous elements per row,
// `rows` rows, row pitch `ld_bytes`; box = box_cols x box_rows.
int make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t cols, uint64_t rows,
             uint64_t ld_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_EINVAL;
}

// ------------------------------------------------------------------ GEMM
// The GEMM kernels are launched with programmatic stream serialisation: when
// the kernel before them is a quantiser (which signals early), their
// prologue (barriers, TMEM, descriptor prefetch) runs on SMs the quantiser has
// already left, and they wait on the device for its results.
template <typename... KArgs, typename... Args>
int launch_programmatic(void (*kern)(KArgs...), int grid, int threads, int smem, cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();  // clear it, as launch_status() does
        return FP8BS_ECUDA;
    }
    return launch_status();
}

template <int BN, int BMODE, bool OUT_F32, bool GROUPED, bool SWIGLU = false>
int launch_gemm(DeviceInfo *d, const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tSB,
                const gemm::Params &p, int grid, cudaStream_t st)
{
    using C = gemm::Cfg<BN, BMODE, GROUPED>;
    auto kern = gemm::gemm_kernel<BN, BMODE, OUT_F32, GROUPED, SWIGLU>;
    constexpr int inst_bit = SWIGLU ? 24 + (GROUPED ? 1 : 0)
                                    : (BN == 256 ? 0 : BN == 192 ? 1 : 2) * 8 + BMODE * 4 + (OUT_F32 ? 2 : 0) +
                                          (GROUPED ? 1 : 0);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!(d->gemm_attr_set & (1u << inst_bit))) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::ALLOC) != cudaSuccess)
                return FP8BS_ECUDA;
            d->gemm_attr_set |= (1u << inst_bit);
        }
    }
    return launch_programmatic(kern, grid, C::THREADS, C::ALLOC, st, tA, tB, tSB, p);
}

template <int BMODE, bool GROUPED>
int launch_gemm_bn(int bn, int out_dtype, DeviceInfo *d, const CUtensorMap &tA, const CUtensorMap &tB,
                   const CUtensorMap &tSB, const gemm::Params &p, int grid, cudaStream_t st)
{
    if (bn == 256)
        return out_dtype == 0 ? launch_gemm<256, BMODE, false, GROUPED>(d, tA, tB, tSB, p, grid, st)
                              : launch_gemm<256, BMODE, true, GROUPED>(d, tA, tB, tSB, p, grid, st);
    if (bn == 192)
        return out_dtype == 0 ? launch_gemm<192, BMODE, false, GROUPED>(d, tA, tB, tSB, p, grid, st)
                              : launch_gemm<192, BMODE, true, GROUPED>(d, tA, tB, tSB, p, grid, st);
    return out_dtype == 0 ? launch_gemm<128, BMODE, false, GROUPED>(d, tA, tB, tSB, p, grid, st)
                          : launch_gemm<128, BMODE, true, GROUPED>(d, tA, tB, tSB, p, grid, st);
}

std::atomic<int> g_tile_n{0};  // fp8bs_set_gemm_tile_n: 0 = automatic
std::atomic<int> g_split_k{1};  // fp8bs_set_gemm_split_last_round
std::atomic<uint32_t> g_split_epoch{0};

// The K-split last round for a dense GEMM with FP32 output whose tiles leave
// the last round of the persistent grid partly idle: the tiles from the
// second-to-last round on are shared out by K chunks (gemm.cuh, "The last
// round of tiles").  Sets p.sk_first, the launch's flag group and value.
int plan_split(DeviceInfo *d, gemm::Params &p, int64_t tiles, int grid, int out_dtype)
{
    const int64_t first = (tiles / grid - 1) * grid;
    if (out_dtype != 1 || g_split_k.load(std::memory_order_relaxed) == 0 || tiles <= grid || tiles % grid == 0 ||
        grid > kSplitGroup || (tiles - first) * (p.K / 128) >= (int64_t(1) << 31))
        return FP8BS_OK;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!d->split_flags &&
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d->split_flags), g_split_flags) != cudaSuccess)
            return FP8BS_ECUDA;
    }
    uint32_t e = g_split_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    if (e == 0)  // a flag value is never 0, the flags' initial value
        e = g_split_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    p.sk_first = static_cast<int>(first);
    p.sk_flags = d->split_flags + static_cast<int64_t>(e % kSplitRing) * kSplitGroup;
    p.sk_epoch = e;
    return FP8BS_OK;
}

template <int BN, bool OUT_F32>
int launch_mx(DeviceInfo *d, const CUtensorMap &tA, const CUtensorMap &tB, const mx::Params &p, int grid,
              cudaStream_t st)
{
    using C = mx::Cfg<BN>;
    auto kern = mx::mx_gemm_kernel<BN, OUT_F32>;
    constexpr unsigned bit = 1u << ((BN == 256 ? 2 : 0) + (OUT_F32 ? 1 : 0));
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!(d->mx_attr_set & bit)) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::ALLOC) != cudaSuccess)
                return FP8BS_ECUDA;
            d->mx_attr_set |= bit;
        }
    }
    return launch_programmatic(kern, grid, mx::THREADS, C::ALLOC, st, tA, tB, p);
}

// Output tile width: 128 when N <= 128; otherwise 256 with block scales and
// 192 with per-row B scales (b_scale_mode 1), whose promotion is the longer
// one: three promotion warpgroups of 64 columns keep more warps per
// scheduler busy than two of 128 (Wgrad GEMM 0.3420 -> 0.3195 ms, same box).
int pick_bn(int64_t M, int64_t N, int b_scale_mode, int num_sms)
{
    (void)M;
    (void)num_sms;
    const int forced = g_tile_n.load(std::memory_order_relaxed);
    if (forced)
        return forced;
    if (N <= 128)
        return 128;
    return b_scale_mode != 0 ? 192 : 256;
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

const char *fp8bs_version(void) { return "fp8bs 0.1 (sm_103a, tcgen05)"; }

const char *fp8bs_status_string(int status)
{
    switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_EINVAL: return "invalid argument";
    case FP8BS_EALIGN: return "pointer or pitch not 16-byte aligned";
    case FP8BS_EARCH: return "device is not sm_103";
    case FP8BS_ECUDA: return "CUDA error";
    case FP8BS_ETIMEOUT: return "kernel abandoned a bounded wait";
    default: return "unknown status";
    }
}

int fp8_quant_1x128(const void *x, int64_t M, int64_t K, int64_t ldx, int along, uint8_t *q, int64_t ldq, float *s,
                    int64_t lds, void *stream)
{
    if (M < 0 || K < 0 || (along != 0 && along != 1))
        return FP8BS_EINVAL;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!x || !q || !s || ldx < K)
        return FP8BS_EINVAL;
    if (M > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(x) || !aligned16(q) || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (along == 0) {
        if (K % 128 != 0 || ldq < K || lds < M)
            return FP8BS_EINVAL;
        const int64_t tiles = ((M + 127) / 128) * (K / 128);
        const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_rows_ctas);
        quant::quant_rows_kernel<false><<<static_cast<int>(grid), quant::kThreads, 0, st>>>(
            rows_args(x, M, K, ldx, q, ldq, s, lds));
    } else {
        if (M % 128 != 0 || K % 8 != 0 || ldq < M || lds < K)
            return FP8BS_EINVAL;
        const int64_t tiles = (M / 128) * ((K + 127) / 128);
        const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_cols_ctas);
        CUtensorMap tmX;
        if (make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
            return FP8BS_EINVAL;
        quant::quant_t_kernel<false><<<static_cast<int>(grid), quant::kThreads, quant::kQtDynSmem, st>>>(
            tmX, static_cast<const uint16_t *>(x), M, K, ldx, nullptr, 0, q, ldq, s, lds, nullptr, 0);
    }
    return launch_status();
}

int fp8_quant_128x128(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, float *s,
                      int64_t lds, void *stream)
{
    if (N < 0 || K < 0)
        return FP8BS_EINVAL;
    if (N == 0 || K == 0)
        return FP8BS_OK;
    if (!w || !q || !s || ldw < K || ldq < K || K % 128 != 0 || lds < K / 128)
        return FP8BS_EINVAL;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(w) || !aligned16(q) || (ldw * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t tiles = ((N + 127) / 128) * (K / 128);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_block_ctas);
    quant::quant_rows_kernel<true><<<static_cast<int>(grid), quant::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        rows_args(w, N, K, ldw, q, ldq, s, lds));
    return launch_status();
}

int fp8_quant_act_weight(const void *x, int64_t M, int64_t Kx, int64_t ldx, uint8_t *qx, int64_t ldqx, float *sx,
                         int64_t ldsx, const void *w, int64_t N, int64_t Kw, int64_t ldw, uint8_t *qw, int64_t ldqw,
                         float *sw, int64_t ldsw, int scale_rule, void *stream)
{
    if (M < 0 || Kx < 0 || N < 0 || Kw < 0 || (scale_rule != 0 && scale_rule != 1))
        return FP8BS_EINVAL;
    const bool do_x = M > 0 && Kx > 0, do_w = N > 0 && Kw > 0;
    if (!do_x && !do_w)
        return FP8BS_OK;
    if (do_x && (!x || !qx || !sx || ldx < Kx || Kx % 128 != 0 || ldqx < Kx || ldsx < M))
        return FP8BS_EINVAL;
    if (do_w && (!w || !qw || !sw || ldw < Kw || Kw % 128 != 0 || ldqw < Kw || ldsw < Kw / 128))
        return FP8BS_EINVAL;
    if (M > (int64_t(1) << 31) || Kx > (int64_t(1) << 31) || N > (int64_t(1) << 31) || Kw > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if ((do_x && (!aligned16(x) || !aligned16(qx) || (ldx * 2) % 16 != 0 || ldqx % 16 != 0)) ||
        (do_w && (!aligned16(w) || !aligned16(qw) || (ldw * 2) % 16 != 0 || ldqw % 16 != 0)))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    // an absent operand contributes no tiles
    const quant::RowsArgs ax = rows_args(x, do_x ? M : 0, do_x ? Kx : 128, ldx, qx, ldqx, sx, ldsx);
    const quant::RowsArgs aw = rows_args(w, do_w ? N : 0, do_w ? Kw : 128, ldw, qw, ldqw, sw, ldsw);
    const int64_t tiles = quant::rows_tiles(ax) + quant::rows_tiles(aw);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_pair_ctas);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (scale_rule == 0)
        quant::quant_pair_kernel<false><<<static_cast<int>(grid), quant::kThreads, 0, st>>>(ax, aw);
    else
        quant::quant_pair_kernel<true><<<static_cast<int>(grid), quant::kThreads, 0, st>>>(ax, aw);
    return launch_status();
}

int fp8_quant_1x128_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq, float *s,
                          int64_t lds, void *stream)
{
    if (M < 0 || K < 0)
        return FP8BS_EINVAL;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!x || !q || !s || ldx < K || K % 128 != 0 || ldq < K || lds < M)
        return FP8BS_EINVAL;
    if (M > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(x) || !aligned16(q) || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t tiles = ((M + 127) / 128) * (K / 128);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_rows_ctas);
    quant::quant_rows_kernel<false, true><<<static_cast<int>(grid), quant::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        rows_args(x, M, K, ldx, q, ldq, s, lds));
    return launch_status();
}

int fp8_quant_128x128_ue8m0(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, float *s,
                            int64_t lds, void *stream)
{
    if (N < 0 || K < 0)
        return FP8BS_EINVAL;
    if (N == 0 || K == 0)
        return FP8BS_OK;
    if (!w || !q || !s || ldw < K || ldq < K || K % 128 != 0 || lds < K / 128)
        return FP8BS_EINVAL;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(w) || !aligned16(q) || (ldw * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t tiles = ((N + 127) / 128) * (K / 128);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_block_ctas);
    quant::quant_rows_kernel<true, true><<<static_cast<int>(grid), quant::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        rows_args(w, N, K, ldw, q, ldq, s, lds));
    return launch_status();
}

int fp8_quant_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, float *s,
                        int64_t lds, uint8_t *qt, int64_t ldqt, float *st, int64_t ldst, void *stream)
{
    if (N < 0 || K < 0)
        return FP8BS_EINVAL;
    if (N == 0 || K == 0)
        return FP8BS_OK;
    if (!w || !qt || !st || (q == nullptr) != (s == nullptr))
        return FP8BS_EINVAL;
    if (ldw < K || K % 128 != 0 || N % 16 != 0 || ldqt < N || ldst < (N + 127) / 128)
        return FP8BS_EINVAL;
    if (q && (ldq < K || lds < K / 128))
        return FP8BS_EINVAL;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(w) || !aligned16(qt) || (ldw * 2) % 16 != 0 || ldqt % 16 != 0 ||
        (q && (!aligned16(q) || ldq % 16 != 0)))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t tiles = ((N + 127) / 128) * (K / 128);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_blockt_ctas);
    CUtensorMap tmW;
    if (make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, K, N, ldw * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
        return FP8BS_EINVAL;
    quant::quant_t_kernel<true><<<static_cast<int>(grid), quant::kThreads, quant::kQtDynSmem,
                                  static_cast<cudaStream_t>(stream)>>>(
        tmW, static_cast<const uint16_t *>(w), N, K, ldw, q, ldq, qt, ldqt, s, lds, st, ldst);
    return launch_status();
}

static int gemm_common_checks(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B,
                              const float *sb, void *C, int64_t ldc, int out_dtype, int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0 || (out_dtype != 0 && out_dtype != 1))
        return FP8BS_EINVAL;
    if (M == 0 || N == 0)
        return 1;  // nothing to do
    if (K == 0 || K % 128 != 0 || N % 8 != 0 || !A || !sa || !B || !sb || !C)
        return FP8BS_EINVAL;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (lda < K || ldsa < M || ldc < N)
        return FP8BS_EINVAL;
    const int esize = out_dtype == 0 ? 2 : 4;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 16 != 0 || (ldc * esize) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(sa) & 3) || (reinterpret_cast<uintptr_t>(sb) & 3))
        return FP8BS_EALIGN;
    return 0;
}

int fp8_gemm_blockscaled(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B, int64_t ldb,
                         const float *sb, int64_t ldsb, int b_scale_mode, void *C, int64_t ldc, int out_dtype,
                         int64_t M, int64_t N, int64_t K, void *stream)
{
    if (b_scale_mode != 0 && b_scale_mode != 1)
        return FP8BS_EINVAL;
    int rc = gemm_common_checks(A, lda, sa, ldsa, B, sb, C, ldc, out_dtype, M, N, K);
    if (rc < 0)
        return rc;
    if (rc == 1)
        return FP8BS_OK;
    if (ldb < K)
        return FP8BS_EINVAL;
    if (ldb % 16 != 0)
        return FP8BS_EALIGN;
    if (b_scale_mode == 0 && ldsb < K / 128)
        return FP8BS_EINVAL;
    if (b_scale_mode == 1) {
        if (ldsb < N)
            return FP8BS_EINVAL;
        if (ldsb % 4 != 0 || !aligned16(sb))
            return FP8BS_EALIGN;
    }
    DeviceInfo *d;
    rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;

    gemm::Params p;
    p.sa = sa;
    p.ldsa = ldsa;
    p.sb = sb;
    p.ldsb = ldsb;
    p.sb_estride = 0;
    p.C = C;
    p.ldc = ldc;
    p.s_out = nullptr;
    p.lds_out = 0;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.group_m = gemm::group_m_for(K);
    p.offs = nullptr;
    p.G = 0;

    const int BN = pick_bn(M, N, b_scale_mode, d->num_sms);
    p.tile_n = BN;
    p.b_rows = static_cast<int>(N);
    // per-row scales: the A row scales of a chunk are copied into shared
    // memory with its B scale row when that is a legal bulk copy (16-byte
    // aligned rows, a multiple of 16 bytes)
    p.sa_smem = (b_scale_mode == 1 && aligned16(sa) && ldsa % 4 == 0 && M % 4 == 0) ? 1 : 0;
    CUtensorMap tA, tB, tSB;
    std::memset(&tSB, 0, sizeof tSB);
    if (make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, lda, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, ldb, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8BS_EINVAL;
    if (b_scale_mode == 1 && make_map(&tSB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sb, N, K / 128, ldsb * 4, BN, 1,
                                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return FP8BS_EINVAL;
    const int64_t tiles = ((M + 127) / 128) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<int64_t>(tiles, d->num_sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = plan_split(d, p, tiles, grid, out_dtype);
    if (rc != FP8BS_OK)
        return rc;
    if (b_scale_mode == 0)
        return launch_gemm_bn<0, false>(BN, out_dtype, d, tA, tB, tSB, p, grid, st);
    return launch_gemm_bn<1, false>(BN, out_dtype, d, tA, tB, tSB, p, grid, st);
}

int fp8_grouped_gemm_moe(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B,
                         const float *sb, const int32_t *group_offsets, int G, int64_t M_total, void *C, int64_t ldc,
                         int out_dtype, int64_t N, int64_t K, void *stream)
{
    if (G < 1 || G > gemm::kMaxGroups || !group_offsets)
        return FP8BS_EINVAL;
    int rc = gemm_common_checks(A, lda, sa, ldsa, B, sb, C, ldc, out_dtype, M_total, N, K);
    if (rc < 0)
        return rc;
    if (rc == 1)
        return FP8BS_OK;
    if (int64_t(G) * N >= (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if ((reinterpret_cast<uintptr_t>(group_offsets) & 3))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;

    gemm::Params p;
    p.sa = sa;
    p.ldsa = ldsa;
    p.sb = sb;
    p.ldsb = K / 128;
    p.sb_estride = ((N + 127) / 128) * (K / 128);
    p.C = C;
    p.ldc = ldc;
    p.s_out = nullptr;
    p.lds_out = 0;
    p.M = static_cast<int>(M_total);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.group_m = gemm::group_m_for(K);
    p.offs = group_offsets;
    p.G = G;

    const int BN = pick_bn(M_total, N, 0, d->num_sms);
    p.tile_n = BN;
    p.b_rows = static_cast<int>(N);
    CUtensorMap tA, tB, tSB;
    std::memset(&tSB, 0, sizeof tSB);
    if (make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M_total, lda, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, int64_t(G) * N, K, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8BS_EINVAL;
    // upper bound on the tile count without reading the offsets on the host
    const int64_t max_tiles = ((M_total + 127) / 128 + G) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<int64_t>(max_tiles, d->num_sms));
    return launch_gemm_bn<0, true>(BN, out_dtype, d, tA, tB, tSB, p, grid, static_cast<cudaStream_t>(stream));
}

int fp8_gemm_ue8m0(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B, int64_t ldb,
                   const float *sb, int64_t ldsb, void *C, int64_t ldc, int out_dtype, int64_t M, int64_t N, int64_t K,
                   void *stream)
{
    int rc = gemm_common_checks(A, lda, sa, ldsa, B, sb, C, ldc, out_dtype, M, N, K);
    if (rc < 0)
        return rc;
    if (rc == 1)
        return FP8BS_OK;
    if (ldb < K || ldsb < K / 128)
        return FP8BS_EINVAL;
    if (ldb % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    mx::Params p;
    p.sa = sa;
    p.ldsa = ldsa;
    p.sb = sb;
    p.ldsb = ldsb;
    p.C = C;
    p.ldc = ldc;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    // This kernel keeps a tile longer than the promoted one and measured best
    // with 16 M tiles per raster group (FFN shape: 1737 us against 2182 with
    // 32), except when the whole M extent fits in one 32-tile group (MLA:
    // 67.6 against 69.7 us).
    p.group_m = ((M + mx::BM - 1) / mx::BM <= gemm::kGroupMLarge) ? gemm::kGroupMLarge : gemm::kGroupMSmall;
    const int forced = g_tile_n.load(std::memory_order_relaxed);
    const int BN = (forced == 192) ? 192 : 256;
    CUtensorMap tA, tB;
    if (make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, lda, 128, mx::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, ldb, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8BS_EINVAL;
    const int64_t tiles = ((M + mx::BM - 1) / mx::BM) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<int64_t>(tiles, d->num_sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (BN == 256)
        return out_dtype == 0 ? launch_mx<256, false>(d, tA, tB, p, grid, st) : launch_mx<256, true>(d, tA, tB, p, grid, st);
    return out_dtype == 0 ? launch_mx<192, false>(d, tA, tB, p, grid, st) : launch_mx<192, true>(d, tA, tB, p, grid, st);
}

int fp8_grouped_gemm_moe_swiglu(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B,
                                const float *sb, const int32_t *group_offsets, int G, int64_t M_total, uint8_t *Q,
                                int64_t ldq, float *s, int64_t lds, int64_t Nh, int64_t K, void *stream)
{
    if (G < 1 || G > gemm::kMaxGroups || !group_offsets || M_total < 0 || Nh < 0 || K < 0)
        return FP8BS_EINVAL;
    if (M_total == 0 || Nh == 0)
        return FP8BS_OK;
    if (K == 0 || K % 128 != 0 || Nh % 128 != 0 || !A || !sa || !B || !sb || !Q || !s)
        return FP8BS_EINVAL;
    if (M_total >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || int64_t(G) * 2 * Nh >= (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (lda < K || ldsa < M_total || ldq < Nh || lds < M_total)
        return FP8BS_EINVAL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(Q) || lda % 16 != 0 || ldq % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(sa) & 3) || (reinterpret_cast<uintptr_t>(sb) & 3) ||
        (reinterpret_cast<uintptr_t>(s) & 3) || (reinterpret_cast<uintptr_t>(group_offsets) & 3))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;

    gemm::Params p;
    p.sa = sa;
    p.ldsa = ldsa;
    p.sb = sb;
    p.ldsb = K / 128;
    p.sb_estride = (2 * Nh / 128) * (K / 128);
    p.C = Q;
    p.ldc = ldq;
    p.s_out = s;
    p.lds_out = lds;
    p.M = static_cast<int>(M_total);
    p.N = static_cast<int>(Nh);
    p.K = static_cast<int>(K);
    p.group_m = gemm::group_m_for(K);
    p.tile_n = 128;
    p.b_rows = static_cast<int>(2 * Nh);
    p.offs = group_offsets;
    p.G = G;

    CUtensorMap tA, tB, tSB;
    std::memset(&tSB, 0, sizeof tSB);
    if (make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M_total, lda, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, int64_t(G) * 2 * Nh, K, 128, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8BS_EINVAL;
    const int64_t max_tiles = ((M_total + 127) / 128 + G) * (Nh / 128);
    const int grid = static_cast<int>(std::min<int64_t>(max_tiles, d->num_sms));
    return launch_gemm<256, 0, false, true, true>(d, tA, tB, tSB, p, grid, static_cast<cudaStream_t>(stream));
}

int fp8_quant_1x128_gather(const void *x, int64_t T, int64_t K, int64_t ldx, const int32_t *row_map, int64_t R,
                           uint8_t *q, int64_t ldq, float *s, int64_t lds, void *stream)
{
    if (T < 0 || K < 0 || R < 0)
        return FP8BS_EINVAL;
    if (R == 0 || K == 0)
        return FP8BS_OK;
    if (!x || !row_map || !q || !s || ldx < K || K % 128 != 0 || ldq < K || lds < R)
        return FP8BS_EINVAL;
    if (T > (int64_t(1) << 31) || R > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if (!aligned16(x) || !aligned16(q) || (ldx * 2) % 16 != 0 || ldq % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(row_map) & 3))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t tiles = ((R + 127) / 128) * (K / 128);
    const int64_t grid = std::min<int64_t>(tiles, int64_t(d->num_sms) * d->quant_rows_ctas);
    quant::quant_rows_kernel<false><<<static_cast<int>(grid), quant::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        rows_args(x, R, K, ldx, q, ldq, s, lds, row_map, T));
    return launch_status();
}

int64_t fp8_moe_route_workspace_size(int E)
{
    if (E < 1 || E > moe::kMaxExperts)
        return -1;
    return (static_cast<int64_t>(E) * 4 + 255) / 256 * 256;
}

int fp8_moe_route(const void *x, int64_t T, int64_t D, int64_t ldx, const float *centroids, int64_t ldc,
                  const float *bias, int E, int topk, float *logits, int32_t *expert_idx, float *gate,
                  int32_t *offsets, int32_t *token_of_row, int32_t *row_of, void *workspace,
                  int64_t workspace_bytes, void *stream)
{
    if (T < 0 || D <= 0 || E < 1 || E > moe::kMaxExperts || E % 4 != 0 || topk < 1 || topk > moe::kMaxTopk ||
        topk > E)
        return FP8BS_EINVAL;
    if (D % 32 != 0 || ldx < D || ldc < E || !offsets || !workspace ||
        workspace_bytes < fp8_moe_route_workspace_size(E))
        return FP8BS_EINVAL;
    if (T > 0 && (!x || !centroids || !bias || !logits || !expert_idx || !gate || !token_of_row || !row_of))
        return FP8BS_EINVAL;
    if (T * topk >= (int64_t(1) << 31))
        return FP8BS_EINVAL;
    if ((T > 0 && (!aligned16(x) || !aligned16(centroids) || (ldx * 2) % 16 != 0 || (ldc * 4) % 16 != 0)) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *counts = static_cast<int *>(workspace);
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, st) != cudaSuccess)
            return FP8BS_ECUDA;
    } else {
        const dim3 lg(static_cast<unsigned>((T + moe::kLT - 1) / moe::kLT), (E + moe::kLE - 1) / moe::kLE);
        moe::route_logits_kernel<<<lg, 64, 0, st>>>(static_cast<const uint16_t *>(x), T, D, ldx, centroids, ldc, E,
                                                     logits, counts);
        const unsigned sg = static_cast<unsigned>((T + 7) / 8);
        if (E <= 256)
            moe::route_select_kernel<8><<<sg, 256, 0, st>>>(logits, T, E, bias, topk, expert_idx, gate, counts);
        else
            moe::route_select_kernel<32><<<sg, 256, 0, st>>>(logits, T, E, bias, topk, expert_idx, gate, counts);
    }
    moe::route_group_kernel<<<E, 256, 0, st>>>(expert_idx, T, topk, E, counts, offsets, token_of_row, row_of);
    return launch_status();
}

int fp8_moe_route_noalloc(const void *x, int64_t T, int64_t D, int64_t ldx, const float *centroids, int64_t ldc,
                          const float *bias, int E, int topk, float *logits, int32_t *expert_idx, float *gate,
                          int32_t *offsets, int32_t *token_of_row, int32_t *row_of, void *stream)
{
    const int64_t need = fp8_moe_route_workspace_size(E);
    if (need < 0 || need > kRouteScratchBytes)
        return FP8BS_EINVAL;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!d->route_scratch && cudaGetSymbolAddress(&d->route_scratch, g_route_scratch) != cudaSuccess)
            return FP8BS_ECUDA;
        scratch = d->route_scratch;
    }
    return fp8_moe_route(x, T, D, ldx, centroids, ldc, bias, E, topk, logits, expert_idx, gate, offsets,
                         token_of_row, row_of, scratch, kRouteScratchBytes, stream);
}

int fp8_moe_combine(const void *Y, int64_t ldy, int64_t R, const int32_t *row_of, const float *gate, int64_t T,
                    int topk, int64_t N, void *out, int64_t ldo, void *stream)
{
    if (T < 0 || N < 0 || R < 0 || topk < 1 || topk > moe::kMaxTopk)
        return FP8BS_EINVAL;
    if (T == 0 || N == 0)
        return FP8BS_OK;
    if (!Y || !row_of || !gate || !out || N % 8 != 0 || ldy < N || ldo < N)
        return FP8BS_EINVAL;
    if (!aligned16(Y) || !aligned16(out) || (ldy * 2) % 16 != 0 || (ldo * 2) % 16 != 0)
        return FP8BS_EALIGN;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t work = T * (N / 8);
    const int64_t grid = std::min<int64_t>((work + 255) / 256, int64_t(d->num_sms) * 8);
    moe::combine_kernel<<<static_cast<int>(grid), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(Y), ldy, R, row_of, gate, T, topk, N, static_cast<uint16_t *>(out), ldo);
    return launch_status();
}

int fp8bs_e4m3_encode(const float *x, uint8_t *q, int64_t n, void *stream)
{
    if (n < 0)
        return FP8BS_EINVAL;
    if (n == 0)
        return FP8BS_OK;
    if (!x || !q)
        return FP8BS_EINVAL;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    const int64_t blocks = std::min<int64_t>((n + 511) / 512, int64_t(d->num_sms) * 8);
    quant::encode_kernel<<<static_cast<int>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, q, n);
    return launch_status();
}

int fp8bs_selftest_division(unsigned long long *counts, void *stream)
{
    if (!counts)
        return FP8BS_EINVAL;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counts, 0, 2 * sizeof(unsigned long long), st) != cudaSuccess)
        return FP8BS_ECUDA;
    quant::selftest_division_kernel<<<0x7F7F, 256, 0, st>>>(counts);
    return launch_status();
}

int fp8bs_set_gemm_tile_n(int bn)
{
    if (bn != 0 && bn != 128 && bn != 192 && bn != 256)
        return FP8BS_EINVAL;
    g_tile_n.store(bn, std::memory_order_relaxed);
    return FP8BS_OK;
}

int fp8bs_set_gemm_split_last_round(int on)
{
    if (on != 0 && on != 1)
        return FP8BS_EINVAL;
    g_split_k.store(on, std::memory_order_relaxed);
    return FP8BS_OK;
}

int fp8bs_gemm_clock(double *mhz, long long *launches, int reset, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long h[3] = {0, 0, 0};
    const unsigned long long zero[3] = {0, 0, 0};
    if (cudaMemcpyFromSymbolAsync(h, g_fp8bs_clock, sizeof h, 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        (reset && cudaMemcpyToSymbolAsync(g_fp8bs_clock, zero, sizeof zero, 0, cudaMemcpyHostToDevice, st) !=
                      cudaSuccess) ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FP8BS_ECUDA;
    if (mhz)
        *mhz = h[1] ? 1e3 * static_cast<double>(h[0]) / static_cast<double>(h[1]) : 0.0;
    if (launches)
        *launches = static_cast<long long>(h[2]);
    return FP8BS_OK;
}

int fp8bs_debug_build(void)
{
#ifdef FP8BS_DEBUG
    return 1;
#else
    return 0;
#endif
}

int fp8bs_debug_site(void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_fp8bs_debug_site, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_fp8bs_debug_site, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FP8BS_ECUDA;
    return h;
}

int fp8bs_get_device_error(void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_fp8bs_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_fp8bs_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FP8BS_ECUDA;
    return h == 0 ? FP8BS_OK : FP8BS_ETIMEOUT;
}

int fp8bs_selftest_timeout(int64_t timeout_ns, void *stream)
{
    if (timeout_ns < 1 || timeout_ns > 1000000000)
        return FP8BS_EINVAL;
    DeviceInfo *d;
    int rc = current_device(&d);
    if (rc != FP8BS_OK)
        return rc;
    selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(timeout_ns));
    return launch_status();
}

}  // extern "C"
