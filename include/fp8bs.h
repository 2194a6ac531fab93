/*
 * fp8bs.h -- C ABI of libfp8bs: fine-grained FP8 (E4M3) quantisation and
 * block-scaled GEMM with FP32 promotion, for NVIDIA B300 (sm_103a).
 *
 * Method (web pages on DeepSeek-V3):
 *   "DeepSeek-V3 技术报告：从 671B MoE 到低成本训练系统" (xutianle.me):
 *     §6   the Fprop, Dgrad and Wgrad GEMMs of every Linear take FP8 inputs;
 *          their outputs stay in BF16 or FP32.
 *     §6.1 activations are scaled per 1x128 tile (one scale per token per 128
 *          channels), weights per 128x128 block, scales computed online.
 *     §6.2 after every 128 FP8 products the tensor-core partial sum is
 *          promoted and accumulated in FP32.
 *     §2   DeepSeekMoE: 256 routed experts, 8 chosen per token.
 *   51itzy.com infra commentary on DeepSeek-V3, FP8 paragraph: E4M3 in both
 *     the forward and the backward pass.
 * Readings where the pages are silent: OCP E4M3FN (max 448); scale =
 * amax / 448 as an IEEE FP32 divide (1.0 for an all-zero tile); code =
 * E4M3(x / scale) of the IEEE FP32 quotient, round-to-nearest-even,
 * saturating at +-448, sign kept.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers owned by the caller, except where a
 *     parameter says otherwise.  The library allocates no device memory per
 *     call.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Calls are asynchronous on `stream`; the library never synchronises,
 *     except fp8bs_get_device_error.
 *   - Argument errors are returned synchronously before any launch.  A failed
 *     launch returns FP8BS_ECUDA.  A kernel that gives up on a bounded
 *     internal wait records FP8BS_ETIMEOUT in a device error word read by
 *     fp8bs_get_device_error; the outputs of that launch are then incomplete.
 *     The word only reports: a launch gives up on its own waits alone, so an
 *     error left unread by an earlier launch does not affect later ones.
 *   - Leading dimensions (ld*) are in elements.  Code and BF16/FP32 matrices
 *     are row-major.  Base pointers must be 16-byte aligned and every row
 *     pitch a multiple of 16 bytes (FP8BS_EALIGN otherwise).
 *   - The device must be sm_103 (FP8BS_EARCH otherwise).
 *   - The GEMM calls are launched with programmatic stream serialisation:
 *     their on-chip set-up may start while the kernel before them in the
 *     stream is still running, but they wait on the device for that kernel
 *     to complete (and its writes to be visible) before touching global
 *     memory.  Stream order is therefore kept exactly as for an ordinary
 *     launch; the quantisers of this library let the next kernel start its
 *     set-up early.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_OK = 0,
    FP8BS_EINVAL = -1,   /* bad size, mode or null pointer */
    FP8BS_EALIGN = -2,   /* pointer or pitch not 16-byte aligned */
    FP8BS_EARCH = -3,    /* current device is not sm_103 */
    FP8BS_ECUDA = -4,    /* CUDA runtime/driver error at launch */
    FP8BS_ETIMEOUT = -5  /* a kernel gave up on a bounded wait */
} fp8bs_status;

/*
 * fp8_quant_1x128 -- per-tile 1x128 quantisation of a BF16 matrix
 * (V3 report §6.1: one scale per token per 128 channels; E4M3, online scale).
 *
 *   x      BF16 [M][ldx], K columns used.
 *   along  0: tiles run along the contiguous dimension: tile (m, kb) is
 *             x[m][128kb .. 128kb+127].
 *             q = codes [M][ldq] (ldq >= K); s = FP32 [K/128][lds], lds >= M
 *             (scale of tile (m, kb) at s[kb*lds + m]).
 *          1: tiles run along rows (used for the weight-gradient GEMM, whose
 *             reduction runs over tokens): tile (tb, k) is x[128tb .. 128tb+127][k].
 *             The codes come out transposed so that rows are contiguous:
 *             q = codes [K][ldq] (ldq >= M), q[k*ldq + m];
 *             s = FP32 [M/128][lds], lds >= K (scale of tile (tb, k) at s[tb*lds + k]).
 *   Requires K % 128 == 0 (along 0) or M % 128 == 0 (along 1), M, K > 0 or
 *   an empty matrix (M == 0 or K == 0 returns FP8BS_OK without a launch).
 *   Codes are uint8 E4M3 bit patterns.  Bit-exact with the reading above.
 */
int fp8_quant_1x128(const void *x, int64_t M, int64_t K, int64_t ldx, int along,
                    uint8_t *q, int64_t ldq, float *s, int64_t lds, void *stream);

/*
 * fp8_quant_128x128 -- per-block 128x128 quantisation of a BF16 weight
 * matrix (V3 report §6.1).
 *   w  BF16 [N][ldw], K columns used; q = codes [N][ldq];
 *   s  FP32 [ceil(N/128)][lds], lds >= K/128: scale of block (nb, kb) at
 *      s[nb*lds + kb].  A partial last block row (N % 128 != 0) takes its
 *      amax over the rows that exist.
 *   Requires K % 128 == 0.
 */
int fp8_quant_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                      uint8_t *q, int64_t ldq, float *s, int64_t lds, void *stream);

/*
 * fp8_quant_act_weight -- fp8_quant_1x128 (along 0) of an activation x and
 * fp8_quant_128x128 of a weight w in one launch (the two operands of a
 * Linear's forward GEMM, V3 report §6.1): the tiles of both tensors form one
 * work list, so that two small tensors keep the GPU busy together.
 *   x, M, Kx, ldx, qx, ldqx, sx, ldsx   as fp8_quant_1x128 (along 0);
 *   w, N, Kw, ldw, qw, ldqw, sw, ldsw   as fp8_quant_128x128;
 *   scale_rule 0: amax/448 scales; 1: power-of-two (UE8M0) scales, as the
 *   _ue8m0 quantisers below.  Results are bit-identical to the separate
 *   calls.  Either operand may be empty (M or Kx, N or Kw == 0).
 */
int fp8_quant_act_weight(const void *x, int64_t M, int64_t Kx, int64_t ldx, uint8_t *qx, int64_t ldqx, float *sx,
                         int64_t ldsx, const void *w, int64_t N, int64_t Kw, int64_t ldw, uint8_t *qw, int64_t ldqw,
                         float *sw, int64_t ldsw, int scale_rule, void *stream);

/*
 * fp8_quant_128x128_t -- per-block 128x128 quantisation of a BF16 weight
 * matrix that also writes the codes and block scales transposed, for the
 * Dgrad GEMM (V3 report §6: Dgrad takes the FP8 weights; §6.1: 128x128
 * weight blocks).  A 128x128 block is the same set of elements in W and in
 * W^T, so the transposed codes and scales are exactly the quantisation of
 * W^T: with them, dX = dY * W is fp8_gemm_blockscaled with A = codes of dY
 * (1x128 along its channels) and B = W^T codes, b_scale_mode 0.
 *   w   BF16 [N][ldw], K columns used (N = output channels of the layer).
 *   q   codes [N][ldq] and s FP32 [ceil(N/128)][lds] exactly as
 *       fp8_quant_128x128 writes them; both NULL to skip them.
 *   qt  codes [K][ldqt], ldqt >= N: qt[k*ldqt + n] = code of w[n][k].
 *   st  FP32 [K/128][ldst], ldst >= ceil(N/128): scale of block (nb, kb) at
 *       st[kb*ldst + nb].
 *   Requires K % 128 == 0 and N % 16 == 0; a partial last block row takes
 *   its amax over the rows that exist.  One pass over w.
 */
int fp8_quant_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw,
                        uint8_t *q, int64_t ldq, float *s, int64_t lds,
                        uint8_t *qt, int64_t ldqt, float *st, int64_t ldst, void *stream);

/* ------------------------------------------------------------------------
 * Power-of-two (UE8M0) scale variant.  The scale of a tile is 2^e with e the
 * smallest integer such that amax <= 448 * 2^e (so no code saturates), kept
 * >= -127 (the UE8M0 range); an all-zero tile has scale 1.  Codes are
 * E4M3_RNE(x * 2^-e), an exact scaling.  The scales are written as FP32
 * powers of two, in the layouts of fp8_quant_1x128 (along 0) and
 * fp8_quant_128x128, so both GEMM entry points take them; the UE8M0 byte
 * is the FP32 exponent field.  The pages' method uses amax/448 scales; the
 * power-of-two rule is the variant whose scales the tensor cores' block-
 * scaled MMA applies in hardware (it changes the numerics: at most one
 * binade of E4M3 range is given up per tile).
 * ------------------------------------------------------------------------ */
int fp8_quant_1x128_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq, float *s,
                          int64_t lds, void *stream);
int fp8_quant_128x128_ue8m0(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, float *s,
                            int64_t lds, void *stream);

/*
 * fp8_gemm_ue8m0 -- C = A * B^T for operands quantised with power-of-two
 * scales (fp8_quant_1x128_ue8m0, fp8_quant_128x128_ue8m0), on the tensor
 * cores' own block scaling (tcgen05 kind::mxf8f6f4, one UE8M0 scale per row
 * per 32 K): the products are scaled inside the MMA and the whole K is
 * accumulated in FP32 in tensor memory, with no promotion pass, so
 *     C[m][n] ~= sum_kb sa[kb][m] * sb(n, kb) * sum_k dec(A) dec(B)
 * up to the tensor core's FP32 accumulation.  Arguments and layouts as
 * fp8_gemm_blockscaled with b_scale_mode 0; every scale must be a power of
 * two within 2^-127 .. 2^127 (the _ue8m0 quantisers write nothing else; the
 * kernel takes the FP32 exponent field as the UE8M0 byte).
 */
int fp8_gemm_ue8m0(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa, const uint8_t *B, int64_t ldb,
                   const float *sb, int64_t ldsb, void *C, int64_t ldc, int out_dtype, int64_t M, int64_t N, int64_t K,
                   void *stream);

/*
 * fp8_gemm_blockscaled -- C = A * B^T from E4M3 codes with fine-grained
 * scales and FP32 promotion every 128 K (V3 report §6, §6.2).
 *
 *   A   codes [M][lda], K used;   sa FP32 [K/128][ldsa], ldsa >= M.
 *   B   codes [N][ldb], K used.
 *   b_scale_mode 0: sb FP32 [ceil(N/128)][ldsb], ldsb >= K/128: one scale per
 *                   128x128 block of B (weights; Fprop and Dgrad).
 *                1: sb FP32 [K/128][ldsb], ldsb >= N, ldsb % 4 == 0: one scale
 *                   per row of B per 128 K (both operands tiled 1x128 along
 *                   K, as in the weight-gradient GEMM).  When sa is 16-byte
 *                   aligned and ldsa and M are multiples of 4 (a dense
 *                   [K/128][M] scale array from fp8_quant_1x128 along=1
 *                   is, since that quantiser needs M % 8 == 0), the
 *                   kernel stages each chunk's row scales in shared memory
 *                   with a bulk copy; otherwise it reads them from global
 *                   memory.  The result is the same either way.
 *   C   [M][ldc]; out_dtype 0: BF16 (round to nearest even), 1: FP32.
 *   Result: for each 128-wide K chunk kb the tensor cores form the FP32
 *   partial P_kb of the E4M3 products, and
 *       C[m][n] = sum_kb  fl32(sa[kb][m] * sb(n, kb)) * P_kb[m][n]
 *   accumulated in FP32 (fused multiply-add), in order of kb.
 *   Requires K % 128 == 0, N % 8 == 0, M, N >= 0 (empty -> no launch).
 */
int fp8_gemm_blockscaled(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                         const uint8_t *B, int64_t ldb, const float *sb, int64_t ldsb,
                         int b_scale_mode, void *C, int64_t ldc, int out_dtype,
                         int64_t M, int64_t N, int64_t K, void *stream);

/*
 * fp8_grouped_gemm_moe -- per-expert block-scaled GEMMs over expert-sorted
 * rows (V3 report §2: routed experts; §6: FP8 GEMMs).
 *
 *   A   codes [M_total][lda], rows sorted by expert; sa FP32 [K/128][ldsa],
 *       ldsa >= M_total.
 *   B   codes [G][N][K] (contiguous); sb FP32 [G][ceil(N/128)][K/128]
 *       (contiguous): expert e's weights and 128x128 block scales.
 *   group_offsets  DEVICE int32 [G+1]: rows offs[e] .. offs[e+1]-1 belong to
 *       expert e; offs[0] == 0, non-decreasing, offs[G] <= M_total.  The
 *       offsets are read on the device only (no host synchronisation);
 *       malformed offsets make the kernel skip the offending experts.
 *   C   [M_total][ldc], out_dtype as above; rows of empty experts and rows
 *       past offs[G] are not written.
 *   Requires K % 128 == 0, N % 8 == 0, 1 <= G <= 1024.
 */
int fp8_grouped_gemm_moe(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                         const uint8_t *B, const float *sb, const int32_t *group_offsets,
                         int G, int64_t M_total, void *C, int64_t ldc, int out_dtype,
                         int64_t N, int64_t K, void *stream);

/* ------------------------------------------------------------------------
 * The routed-expert chain (V3 report §2 DeepSeekMoE: 256 routed experts, 8
 * per token, SwiGLU experts; §4 aux-loss-free balancing: sigmoid affinity to
 * each expert's centroid, top-k of affinity + bias, gates from the selected
 * affinities normalised to sum 1).  One layer forward:
 *   fp8_moe_route -> fp8_quant_1x128_gather -> fp8_grouped_gemm_moe_swiglu
 *   -> fp8_grouped_gemm_moe (down projection) -> fp8_moe_combine.
 * ------------------------------------------------------------------------ */

/* Bytes of device workspace fp8_moe_route needs for E experts (-1 if E is
 * outside 1 .. 1024). */
int64_t fp8_moe_route_workspace_size(int E);

/*
 * fp8_moe_route -- routing and grouping of T tokens over E experts.
 *   x          BF16 tokens [T][ldx], D used (D % 32 == 0).
 *   centroids  FP32, k-major: [D][ldc], ldc >= E (expert e's centroid is
 *              column e; a router weight stored once in the kernel's layout).
 *   bias       FP32 [E] (selection only).
 *   logits     out FP32 [T][E]: l[t][e] = sum_k x[t][k] * c[k][e], formed in
 *              FP32 with one fused multiply-add per term in increasing k (the
 *              decision below is taken from exactly these values).
 *   expert_idx out int32 [T][topk]: the topk experts with the largest
 *              1/(1+exp(-l)) + b (evaluated in double; a tie goes to the
 *              lower index), listed in increasing expert order.
 *   gate       out FP32 [T][topk]: s_e / (sum of the chosen s), s = the
 *              double affinity, the sum taken in the listed order.
 *   offsets    out int32 [E+1]: rows offsets[e] .. offsets[e+1]-1 belong to
 *              expert e; rows of one expert hold its tokens in increasing
 *              order.  token_of_row out int32 [T*topk]; row_of out int32
 *              [T][topk] (row of token t's j-th listed expert).
 *   workspace  device, >= fp8_moe_route_workspace_size(E) bytes, 256-byte
 *              aligned, owned by the caller; contents on return unspecified.
 *   Requires 1 <= E <= 1024, E % 4 == 0, 1 <= topk <= min(E, 16).  T == 0 writes zero
 *   offsets.  Deterministic: no result depends on launch timing.
 */
int fp8_moe_route(const void *x, int64_t T, int64_t D, int64_t ldx, const float *centroids, int64_t ldc,
                  const float *bias, int E, int topk, float *logits, int32_t *expert_idx, float *gate,
                  int32_t *offsets, int32_t *token_of_row, int32_t *row_of, void *workspace,
                  int64_t workspace_bytes, void *stream);

/*
 * fp8_moe_route_noalloc -- fp8_moe_route without a caller workspace: the
 * library uses its own static device scratch (4 KB per device, enough for
 * E <= 1024) and allocates nothing.  The method as the pages describe it has
 * no counterpart; this is a convenience of the interface.  Results are those
 * of fp8_moe_route.  The scratch is one buffer per device, so calls on one
 * device must be ordered (one stream, or events between streams).  An E
 * whose workspace would not fit returns FP8BS_EINVAL before any launch.
 */
int fp8_moe_route_noalloc(const void *x, int64_t T, int64_t D, int64_t ldx, const float *centroids, int64_t ldc,
                          const float *bias, int E, int topk, float *logits, int32_t *expert_idx, float *gate,
                          int32_t *offsets, int32_t *token_of_row, int32_t *row_of, void *stream);

/*
 * fp8_quant_1x128_gather -- fp8_quant_1x128 (along 0) of the rows
 * x[row_map[r]], r = 0 .. R-1: gathering and quantising in one pass (equal,
 * bit for bit, to quantising then gathering, since every scale belongs to
 * one row).  x BF16 [T][ldx]; row_map DEVICE int32 [R]; q codes [R][ldq];
 * s FP32 [K/128][lds], lds >= R.  A mapped row outside [0, T) quantises as
 * zeros (codes 0, scale 1).  Requires K % 128 == 0.
 */
int fp8_quant_1x128_gather(const void *x, int64_t T, int64_t K, int64_t ldx, const int32_t *row_map, int64_t R,
                           uint8_t *q, int64_t ldq, float *s, int64_t lds, void *stream);

/*
 * fp8_grouped_gemm_moe_swiglu -- per-expert up projection with the SwiGLU
 * and its 1x128 quantisation fused into the epilogue (the down projection
 * takes FP8 inputs, V3 report §6).
 *   A, sa, group_offsets, G, M_total as fp8_grouped_gemm_moe.
 *   B   codes [G][2*Nh][K]: rows 0 .. Nh-1 the gate projection, Nh .. 2Nh-1
 *       the up projection; sb FP32 [G][2*Nh/128][K/128] block scales.
 *   For each row and channel n < Nh, with g and u the FP32 results of the
 *   block-scaled GEMM (as fp8_gemm_blockscaled computes them) for rows n
 *   and Nh + n of B:  h = g / (1 + expf(-g)) * u  (FP32, IEEE divide), and
 *   h is quantised in 1x128 tiles along n: Q codes [M_total][ldq],
 *   s FP32 [Nh/128][lds], lds >= M_total (s = amax/448, codes of the IEEE
 *   quotient h / s).  Rows of empty experts and rows past offs[G] are not
 *   written.  Requires Nh % 128 == 0, K % 128 == 0, 1 <= G <= 1024.
 */
int fp8_grouped_gemm_moe_swiglu(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                                const uint8_t *B, const float *sb, const int32_t *group_offsets, int G,
                                int64_t M_total, uint8_t *Q, int64_t ldq, float *s, int64_t lds,
                                int64_t Nh, int64_t K, void *stream);

/*
 * fp8_moe_combine -- out[t][n] = BF16_RNE(sum_j gate[t][j] * Y[row_of[t][j]][n]),
 * the sum formed in FP32 with one fused multiply-add per listed expert, in
 * list order.  Y BF16 [R][ldy] (the down projection's rows); row_of int32
 * [T][topk]; gate FP32 [T][topk]; out BF16 [T][ldo].  A row index outside
 * [0, R) contributes nothing.  Requires N % 8 == 0.
 */
int fp8_moe_combine(const void *Y, int64_t ldy, int64_t R, const int32_t *row_of, const float *gate, int64_t T,
                    int topk, int64_t N, void *out, int64_t ldo, void *stream);

/*
 * fp8bs_e4m3_encode -- element-wise q[i] = E4M3_RNE_saturate(x[i]) with the
 * same conversion the quantisers use; x FP32 [n], q uint8 [n] (device).
 * A diagnostic for checking the conversion exhaustively.
 */
int fp8bs_e4m3_encode(const float *x, uint8_t *q, int64_t n, void *stream);

/*
 * fp8bs_selftest_division -- the quantisers divide by the tile scale with a
 * per-tile reciprocal and one Markstein correction instead of an IEEE divide.
 * This diagnostic encodes both quotients to E4M3 (the fast one exactly as
 * the quantisers form it, signs of zeros included) for every positive finite BF16 amax
 * and every BF16 x with |x| <= amax (about 2^31 values of each sign) and
 * writes counts[0] = values whose codes differ (0 means the fast path is
 * bit-exact on every BF16 input), counts[1] = values whose FP32 quotients
 * differ in value.
 * counts: DEVICE unsigned long long [2].
 */
int fp8bs_selftest_division(unsigned long long *counts, void *stream);

/*
 * fp8bs_set_gemm_tile_n -- output tile width (N per CTA tile) of the GEMM
 * entry points for block-scaled B: 128, 192 or 256, or 0 to let the library
 * choose from the problem shape (the default: 128 when N <= 128, else 256
 * with b_scale_mode 0 and 192 with b_scale_mode 1).  Process-wide; results
 * do not depend on it (every output element is computed the same way), only
 * speed.
 * fp8_gemm_ue8m0 uses 256 unless 192 is forced.
 */
int fp8bs_set_gemm_tile_n(int bn);

/*
 * fp8bs_set_gemm_split_last_round -- 1 (the default): when fp8_gemm_blockscaled
 * writes FP32 output and its output tiles leave the last round of the
 * persistent grid partly idle, the tiles from the second-to-last round on are
 * shared out by K chunks so that every CTA does the same number of chunks; a
 * tile shared by two CTAs is promoted by one of them over its first chunks
 * and by the other over the rest, continuing from the first one's FP32
 * accumulators (which pass through C), so every output element is still
 * promoted chunk by chunk in K order and the result is bit-identical to
 * whole tiles.  0: whole tiles only.  Process-wide; FP8BS_EINVAL for any
 * other value.  No counterpart on the pages (a scheduling choice).
 */
int fp8bs_set_gemm_split_last_round(int on);

/*
 * fp8bs_gemm_clock -- synchronise `stream` and report the SM clock the GEMM
 * kernels (fp8_gemm_blockscaled, fp8_grouped_gemm_moe(_swiglu),
 * fp8_gemm_ue8m0) ran at since the last reset: *mhz = the summed SM cycles
 * over the summed nanoseconds of one CTA per launch (from the end of its
 * set-up to its end), *launches = the launches counted.  Either pointer may
 * be NULL; reset != 0 clears the record after reading it.  Launches that
 * overlap on the GPU each count their own interval.  FP8BS_ECUDA on a CUDA
 * error.  No counterpart on the pages: a measurement aid (the clock drops
 * under the board's power cap, and sampling tools cannot resolve kernels of
 * a millisecond).
 */
int fp8bs_gemm_clock(double *mhz, long long *launches, int reset, void *stream);

/*
 * fp8bs_debug_build -- 1 if this library was compiled with FP8BS_DEBUG (the
 * bounds-checked build, libfp8bs_debug.so), else 0.
 *
 * fp8bs_debug_site -- synchronise `stream`, read and clear the bounds-check
 * record of the current device: 0 if no check has failed since the last
 * read, else the number of the first access site whose index fell outside
 * its extent (the kernel skipped that access; the site numbers are listed in
 * the library source beside the checks).  Always 0 in the release build,
 * which has no checks.  FP8BS_ECUDA on a CUDA error.
 * No counterpart on the pages: a test aid for the kernels' index arithmetic.
 */
int fp8bs_debug_build(void);
int fp8bs_debug_site(void *stream);

/* Human-readable text for a status code (static storage). */
const char *fp8bs_status_string(int status);

/*
 * fp8bs_get_device_error -- synchronise `stream`, read and clear the device
 * error word of the current device.  Returns FP8BS_OK, FP8BS_ETIMEOUT (some
 * kernel since the last read abandoned a bounded wait, and its outputs are
 * incomplete), or FP8BS_ECUDA.
 */
int fp8bs_get_device_error(void *stream);

/*
 * fp8bs_selftest_timeout -- launch one block that waits on a barrier nothing
 * will complete, with a wait bound of `timeout_ns` nanoseconds (1 .. 1e9),
 * so that callers can check the timeout path: the kernel records
 * FP8BS_ETIMEOUT and returns; nothing faults or hangs.
 */
int fp8bs_selftest_timeout(int64_t timeout_ns, void *stream);

/* Version string of the library build. */
const char *fp8bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
