/*
 * rlq.h — C ABI of librlq.so, the GB300 (sm_103a) FP8 quantized actor linear layer.
 *
 * The layer, as the pages on quantized RL rollout describe it:
 *   - fine-grained FP8 quantization: 1x128 per-group scales for activations and
 *     gradients, 128x128 per-block scales for weights, and a 128x1 grouping of
 *     the second WGrad operand fused with the first (Jet-RL notes, section
 *     "细粒度 GEMM 量化方案", Fig. 6);
 *   - FP8 GEMMs for the three training passes FProp, DGrad and WGrad on those
 *     operands (same section; DGrad takes FProp's configuration);
 *   - the one-time UAQ invariant-scaling fold WX = (W/s)(sX), s applied per
 *     column of W and per row of the previous activation (QuRL notes,
 *     关键设计 §1).
 *
 * Conventions for every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and never synchronises, except rlq_check.
 *   - Row-major storage: element (r, c) of a matrix with row pitch ld sits at
 *     base[r * ld + c].  All ld arguments count elements, not bytes.
 *   - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *   - "Codes" are FP8 E4M3 bytes (OCP "fn" variant: max 448, no infinities).
 *     Scales are fp32 dequantization multipliers: value ~= decode(code) * scale.
 *     A group's scale is fl32(amax / 448), or 1.0 when the group is all zero;
 *     a code is the round-to-nearest-even, saturating E4M3 encoding of
 *     fl32(x / scale) with IEEE fp32 division.
 *   - Alignment: every code and bf16 base pointer 16-byte aligned and every
 *     code / bf16 row pitch a multiple of 16 bytes; fp32 scale pointers 4-byte
 *     aligned.  Violations return RLQ_ERR_MISALIGNED.
 *   - Shapes: dimensions that carry 128-groups (K for activations, N and K for
 *     weights) must be multiples of 128, else RLQ_ERR_UNSUPPORTED.  The token
 *     dimension M may be any value >= 0.  A call with an empty extent returns
 *     RLQ_OK and launches nothing.
 *   - Errors: arguments are validated on the host before any launch (NULL
 *     pointers, negative sizes, ld smaller than the row, misalignment); on
 *     failure nothing is launched.  A failed launch returns RLQ_ERR_CUDA.  The
 *     GEMM kernels bound every wait on the GPU: a wait that runs out records
 *     an error word on the device, and the next rlq_check on that device
 *     returns RLQ_ERR_TIMEOUT.  rlq_last_error() describes the latest failure.
 *   - Inputs must be finite; NaN / Inf inputs are outside the contract.
 */
#ifndef RLQ_H
#define RLQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *rlq_stream_t; /* same type as cudaStream_t */

typedef enum {
    RLQ_OK = 0,
    RLQ_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, ld too small, bad flag */
    RLQ_ERR_UNSUPPORTED = 2, /* a 128-grouped dimension is not a multiple of 128 */
    RLQ_ERR_MISALIGNED = 3,  /* pointer or row pitch breaks the alignment rules */
    RLQ_ERR_CUDA = 4,        /* a CUDA call or launch failed */
    RLQ_ERR_TIMEOUT = 5      /* a bounded device-side wait ran out (rlq_check) */
} rlq_status;

/*
 * Activation / gradient quantization, 1x128 groups along K, with an optional
 * fused 128x1 grouping along M written transposed (one read of x).
 * Jet-RL notes, "细粒度 GEMM 量化方案": activations and gradients 1x128 per
 * group; the second WGrad operand 128x1, fused with the first to avoid
 * quantizing twice.
 *
 *   x   bf16 [M, K], pitch ldx >= K                      (input)
 *   q   E4M3 [M, K], pitch ldq >= K                      (output) row-wise codes
 *   s   f32, s[kb * lds + m], kb < K/128, lds >= M       (output) row-wise scales
 *   qT  E4M3, qT[k * ldqT + m] for k < K, m < M, ldqT >= M  (output, optional)
 *       column-wise codes: group (mb, k) = rows 128*mb .. min(M, 128*mb+128)-1
 *       of column k; positions m >= M are not written
 *   sc  f32, sc[mb * ldsc + k], mb < ceil(M/128), ldsc >= K (output; required
 *       exactly when qT is non-NULL)
 * K % 128 == 0.  Either both qT and sc are NULL (row-wise only) or neither.
 */
rlq_status rlq_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *q, int64_t ldq, float *s, int64_t lds,
                               uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc,
                               rlq_stream_t stream);

/*
 * RMSNorm fused with the activation quantization above, the UAQ scale carried
 * by the norm weight.  QuRL notes, 关键设计 §1: the per-channel s that
 * multiplies the previous activation can be folded straight into the norm's
 * scale (gamma' = gamma * s: rlq_uaq_fold with prev = gamma, R = 1).  Jet-RL
 * notes, 细粒度 GEMM 量化方案 / 实践建议: the forward activation is kept as its
 * 1x128 (and, for WGrad, 128x1) FP8 codes.  This call reads the hidden state
 * once from HBM, normalises it and quantizes the result, without writing the
 * bf16 activation; its codes and scales are exactly those of rlq_quant_act_1x128
 * applied to
 *
 *   x[m, k] = bf16_RN( fl32( fl32(h[m, k] * rstd[m]) * gamma[k] ) ),
 *   rstd[m] = fl32( 1 / fl32(sqrt( fl32( fl32(acc_m / K) + eps ) )) ),
 *   acc_m   = sum over k = 0 .. K-1, in index order, of h[m, k]^2 by fp32 fused
 *             multiply-adds from 0 (the order makes the result independent of
 *             the launch shape).
 *
 * The pages give no formula for the norm; this is the standard RMSNorm with
 * every step in fp32 and one rounding to bf16.
 *
 *   h      bf16 [M, K], pitch ldh >= K                   (input, the hidden state)
 *   gamma  bf16 [K], 16-byte aligned                     (input, the folded norm weight)
 *   eps    finite, >= 0; a row of zeros with eps == 0 is outside the contract
 *   rstd   f32 [M]                                        (output) rstd[m] above,
 *          also read back by the call's second kernel
 *   q, s, qT, ldqT, sc, ldsc: as in rlq_quant_act_1x128   (outputs)
 * K % 128 == 0.  Two launches on `stream`: the row factors, then the quantizer.
 */
rlq_status rlq_rmsnorm_quant_act_1x128(const uint16_t *h, int64_t M, int64_t K, int64_t ldh,
                                      const uint16_t *gamma, float eps, float *rstd,
                                      uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                      uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc,
                                      rlq_stream_t stream);

/*
 * Weight quantization, 128x128 blocks.  Jet-RL notes, "细粒度 GEMM 量化方案":
 * weights 128x128 per block; "系统实现": weights are quantized at the
 * parameter-update step.
 *
 *   w   bf16 [N, K], pitch ldw >= K                      (input)
 *   q   E4M3 [N, K], pitch ldq >= K                      (output)
 *   s   f32, s[nb * lds + kb], lds >= K/128              (output) block scales
 *   qT  E4M3 [K, N], pitch ldqT >= N                     (output, optional)
 *       the same codes transposed, the B operand of DGrad
 * N % 128 == 0 and K % 128 == 0.
 */
rlq_status rlq_quant_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                    uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                    uint8_t *qT, int64_t ldqT, rlq_stream_t stream);

/*
 * FProp: Y = X W^T with 1x128 X codes and 128x128 W codes.  Jet-RL notes,
 * "细粒度 GEMM 量化方案": the FProp input activation is 1x128-quantized
 * (row-major) and the weight 128x128-quantized.
 *
 *   Y[m, n] = bf16_RN( sum_kb xs[kb, m] * ws[n/128, kb] * sum_{k in kb} x[m,k] w[n,k] )
 *
 *   xq  E4M3 [M, K], pitch ldxq;   xs f32, xs[kb * ldxs + m], ldxs >= M
 *   wq  E4M3 [N, K], pitch ldwq;   ws f32, ws[nb * ldws + kb], ldws >= K/128
 *   y   bf16 [M, N], pitch ldy >= N (output, overwritten)
 * N % 128 == 0, K % 128 == 0.  Accumulation is fp32 (tensor-core partial sums
 * of each 128-K block, then the scale product applied in fp32).
 */
rlq_status rlq_gemm_fprop(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs,
                          const uint8_t *wq, int64_t ldwq, const float *ws, int64_t ldws,
                          uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                          rlq_stream_t stream);

/*
 * DGrad: dX = dY W with 1x128 dY codes (groups along N) and the FProp weight
 * blocks.  Jet-RL notes, "细粒度 GEMM 量化方案": DGrad is equivalent to FProp
 * and reuses its configuration.
 *
 *   dX[m, k] = bf16_RN( sum_nb dys[nb, m] * ws[nb, k/128] * sum_{n in nb} dy[m,n] w[n,k] )
 *
 *   dyq  E4M3 [M, N], pitch lddyq; dys f32, dys[nb * lddys + m], lddys >= M
 *   w    wq_is_transposed = 1: wqT E4M3 [K, N], pitch ldw >= N (from
 *        rlq_quant_weight_128x128's qT); wq_is_transposed = 0: wq E4M3 [N, K],
 *        pitch ldw >= K (the FProp operand itself)
 *   ws   f32 block scales of W as in FProp: ws[nb * ldws + kb], ldws >= K/128
 *   dx   bf16 [M, K], pitch lddx >= K (output, overwritten)
 * N % 128 == 0, K % 128 == 0.
 */
rlq_status rlq_gemm_dgrad(const uint8_t *dyq, int64_t lddyq, const float *dys, int64_t lddys,
                          const uint8_t *w, int64_t ldw, int wq_is_transposed,
                          const float *ws, int64_t ldws, uint16_t *dx, int64_t lddx,
                          int64_t M, int64_t N, int64_t K, rlq_stream_t stream);

/*
 * WGrad: dW = dY^T X with 128x1 groups along the M tokens on both operands
 * (the transposed outputs of rlq_quant_act_1x128).  Jet-RL notes,
 * "细粒度 GEMM 量化方案": WGrad takes a 1x128 first operand and a 128x1 second
 * operand; here both are grouped along the contraction (token) dimension,
 * which is what a 128-block promotion over the contraction needs.
 *
 *   dW[n, k] = bf16_RN( sum_mb dysc[mb, n] * xsc[mb, k] * sum_{m in mb} dy[m,n] x[m,k] )
 *
 *   dyqT E4M3, dyqT[n * lddyqT + m], lddyqT >= M; dysc f32, dysc[mb * lddysc + n], lddysc >= N
 *   xqT  E4M3, xqT[k * ldxqT + m],  ldxqT >= M;  xsc f32, xsc[mb * ldxsc + k],  ldxsc >= K,
 *        xsc 16-byte aligned and ldxsc % 4 == 0 (its rows are copied to shared memory in bulk)
 *   dw   bf16 [N, K], pitch lddw >= K (output, overwritten; M == 0 writes zeros)
 * N % 128 == 0, K % 128 == 0; the last token block may be partial.
 */
rlq_status rlq_gemm_wgrad(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc,
                          const uint8_t *xqT, int64_t ldxqT, const float *xsc, int64_t ldxsc,
                          uint16_t *dw, int64_t lddw, int64_t M, int64_t N, int64_t K,
                          rlq_stream_t stream);

/*
 * Per-token activations and per-channel weights, FP8.  QuRL notes, "损失函数 /
 * 训练策略": the rollout model runs with channel-wise weight quantization and
 * token-wise activation quantization (INT8 or FP8; the FP8 form is built here).
 *
 * rlq_quant_per_row: one group per row over all K columns, with the scale rule
 * and encoding of the 128-groups above (s = fl32(amax / 448), 1.0 for an
 * all-zero row; codes RN-even satfinite of fl32(x / s)).  Per-token
 * activations: x = X [M, K].  Per-channel weights: x = W [N, K] (one row per
 * output channel).
 *
 *   x      bf16 [M, K], pitch ldx >= K
 *   q      E4M3 [M, K], pitch ldq >= K
 *   s      f32 [M], s[m] = the row's scale (contiguous)
 *   s_rep  optional (NULL to skip): f32, s_rep[kb * ld_rep + m] = s[m] for every
 *          kb < K/128, ld_rep >= M — the layout rlq_gemm_fprop_per_channel reads
 * K % 128 == 0; M any value >= 0.
 *
 * rlq_gemm_fprop_per_channel: Y = diag(sx) (Qx Qw^T) diag(sw), i.e.
 *
 *   Y[m, n] = bf16_RN( sum_kb xs_rep[kb, m] * ws_rep[kb, n] * sum_{k in kb} x[m,k] w[n,k] )
 *
 * which with replicated scales (xs_rep[kb, m] = sx[m], ws_rep[kb, n] = sw[n])
 * equals sx[m] sw[n] sum_k x[m,k] w[n,k] up to the order of the fp32 sums.
 * The GEMM relies on that: it accumulates the whole contraction (or, split-K,
 * each split's range) in fp32 in the tensor cores and multiplies the sum once by
 * fl32(xs_rep[kb0, m] * ws_rep[kb0, n]), kb0 the first block of the range.
 *
 *   xq  E4M3 [M, K], pitch ldxq;  xs_rep f32, xs_rep[kb * ldxs + m], ldxs >= M
 *   wq  E4M3 [N, K], pitch ldwq;  ws_rep f32, ws_rep[kb * ldws + n], ldws >= N,
 *       ws_rep 16-byte aligned and ldws % 4 == 0
 *   y   bf16 [M, N], pitch ldy >= N (output, overwritten)
 * N % 128 == 0, K % 128 == 0.  Errors as for the other calls.
 */
rlq_status rlq_quant_per_row(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, int64_t ldq, float *s, float *s_rep, int64_t ld_rep,
                             rlq_stream_t stream);

rlq_status rlq_gemm_fprop_per_channel(const uint8_t *xq, int64_t ldxq, const float *xs_rep, int64_t ldxs,
                                      const uint8_t *wq, int64_t ldwq, const float *ws_rep, int64_t ldws,
                                      uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                      rlq_stream_t stream);

/*
 * Split-K form of rlq_gemm_fprop_per_channel, for decode-sized M (the rollout
 * case): workspace, workspace_bytes and the result's summation order as for
 * the split-K GEMMs below; rlq_gemm_splitk_workspace_bytes(RLQ_GEMM_FPROP, M,
 * N, K, ...) gives the size of its unconstrained plan.
 */
rlq_status rlq_gemm_fprop_per_channel_splitk(const uint8_t *xq, int64_t ldxq, const float *xs_rep, int64_t ldxs,
                                             const uint8_t *wq, int64_t ldwq, const float *ws_rep, int64_t ldws,
                                             uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                             void *workspace, int64_t workspace_bytes, rlq_stream_t stream);

/*
 * WGrad accumulated into an fp32 gradient, for micro-batch accumulation (the
 * pages' GEMMs write bf16; this keeps the sum over micro-batches in fp32):
 *
 *   dw_acc[n, k] += sum_mb dysc[mb, n] * xsc[mb, k] * sum_{m in mb} dy[m,n] x[m,k]
 *
 * with the operands of rlq_gemm_wgrad.  The product is formed as in
 * rlq_gemm_wgrad (fp32 promotion of each 128-token block) and the GEMM's
 * epilogue adds it to dw_acc in fp32; nothing is rounded to bf16.  Where the
 * library's split-K plan splits the contraction (outputs of few tiles) and the
 * workspace holds the plan, each split's fp32 sum goes to the workspace and a
 * reduction adds the splits, in split order, to dw_acc.
 *
 *   dw_acc     f32 [N, K], pitch ld_acc >= K, 16-byte aligned rows (pointer
 *              16-byte aligned, ld_acc % 4 == 0); read and written
 *   workspace  optional device scratch (NULL, or 16-byte aligned) for the split-K
 *              plan, sized as for rlq_gemm_wgrad_splitk; contents on entry do not
 *              matter; not to be used by anything else until the call has
 *              completed on `stream`
 * M == 0 adds nothing.  N % 128 == 0, K % 128 == 0.
 */
rlq_status rlq_gemm_wgrad_accumulate(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc,
                                     const uint8_t *xqT, int64_t ldxqT, const float *xsc, int64_t ldxsc,
                                     float *dw_acc, int64_t ld_acc, int64_t M, int64_t N, int64_t K,
                                     void *workspace, int64_t workspace_bytes, rlq_stream_t stream);

/*
 * NVFP4 weight quantization (QeRL news article: a hardware 4-bit float with
 * two-level scaling, FP8 E4M3 block scales and an FP32 tensor scale, used for
 * the policy weights).  The pages fix neither the block size nor the scale rule;
 * this call uses E2M1 elements, blocks of 16 consecutive elements along K and
 *
 *   st = fl32(amax(w) / (6 * 448)), or 1 for an all-zero w
 *   sb[n, kb] = E4M3_RNsat(fl32(fl32(amax of the block / 6) / st))
 *   q = E2M1_RNsat(fl32(x / fl32(decode(sb) * st)))  (+-0 when that scale is 0)
 *
 * so that x ~= e2m1(q) * e4m3(sb) * st.  E2M1 rounding is to nearest, ties to
 * the even code, saturating at +-6; the sign of zero is kept.
 *
 *   w   bf16 [N, K], pitch ldw >= K (elements, a multiple of 8)
 *   q   packed E2M1 codes, two per byte: byte b of row n holds element 2b in its
 *       low nibble and 2b + 1 in its high nibble; pitch ldq >= K/2 bytes, rows
 *       8-byte aligned (ldq % 8 == 0)
 *   sb  E4M3 block-scale codes [N, K/16], pitch ldsb >= K/16 bytes
 *   st  one fp32 in device memory (written; used as scratch during the call)
 * K % 16 == 0; N any value >= 0.
 */
rlq_status rlq_quant_nvfp4(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                           uint8_t *sb, int64_t ldsb, float *st, rlq_stream_t stream);

/*
 * NVFP4 weight-only GEMM: BF16 activations times NVFP4 weights, the FP4 x BF16
 * rollout GEMM of the QeRL news article (NVFP4 with two-level scaling, FP8 E4M3
 * block scales and an FP32 tensor scale, run by FP4 x BF16 kernels).
 *
 *   Y[m, n] = bf16_RN( st * sum_k x[m, k] * e2m1(q[n, k]) * e4m3(sb[n, k / 16]) )
 *
 * with the operands rlq_quant_nvfp4 writes.  Each weight value e2m1 * e4m3 is exact
 * in bf16 (at most 6 significant bits, within [2^-10, 2688] or 0); the products with
 * x and their sum over K are accumulated in fp32 by the tensor cores, then multiplied
 * once by st and rounded to bf16.  The activations are not quantized.  Batches of
 * up to 4 tokens run on the CUDA cores instead (fp32 FMAs of the same exact products,
 * summed in a fixed order): the result is the same up to the order of the fp32
 * additions, and repeats bit for bit from call to call.
 *
 *   x    bf16 [M, K], pitch ldx >= K (elements, a multiple of 8), 16-byte aligned
 *   wq   packed E2M1 codes [N, K/2] as rlq_quant_nvfp4 writes them (low nibble =
 *        even element), pitch ldwq >= K/2 bytes, a multiple of 16, 16-byte aligned
 *   wsb  E4M3 block-scale codes [N, K/16], pitch ldwsb >= K/16 bytes, a multiple of
 *        16, 16-byte aligned
 *   wst  the fp32 tensor scale, one value in device memory
 *   y    bf16 [M, N], pitch ldy >= N (output, overwritten)
 * N % 128 == 0 and K % 64 == 0, else RLQ_ERR_UNSUPPORTED.  M any value >= 0.
 * Errors as for the other GEMMs (bounded device waits report at rlq_check).
 */
rlq_status rlq_gemm_nvfp4_weight_only(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq,
                                      const uint8_t *wsb, int64_t ldwsb, const float *wst, uint16_t *y,
                                      int64_t ldy, int64_t M, int64_t N, int64_t K, rlq_stream_t stream);

/*
 * Split-K form of the NVFP4 weight-only GEMM, for decode-sized M, where the
 * output has fewer 128 x 256 tiles than the GPU has SMs (a layer with few
 * output channels and a long contraction leaves most SMs idle otherwise).  A
 * scheduling choice of this library; the pages prescribe no tiling.  Each
 * split sums a contiguous range of K (a multiple of 256 elements) in fp32 on
 * the tensor cores, multiplies its sum by st, and the split results are added
 * in split order in fp32 and rounded to bf16 once:
 *
 *   Y[m, n] = bf16_RN( sum over splits s, in order, of fl32(st * S_s[m, n]) )
 *
 * Deterministic (no atomics); it may differ from the single-pass call in the
 * last bits of the fp32 sum.  workspace and workspace_bytes as for the FP8
 * split-K calls (caller-owned, 16-byte aligned or NULL for one pass; the plan
 * is lowered until splits * M * N * 4 bytes fit); the unconstrained plan's
 * size comes from rlq_gemm_splitk_workspace_bytes(RLQ_GEMM_NVFP4_WEIGHT_ONLY,
 * M, N, K), which is 0 for M <= 2: one or two tokens run the single-pass CUDA-core
 * path whatever the workspace, with the bits of rlq_gemm_nvfp4_weight_only.  Other arguments, shapes and errors as for
 * rlq_gemm_nvfp4_weight_only.
 */
rlq_status rlq_gemm_nvfp4_weight_only_splitk(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq,
                                            const uint8_t *wsb, int64_t ldwsb, const float *wst, uint16_t *y,
                                            int64_t ldy, int64_t M, int64_t N, int64_t K, void *workspace,
                                            int64_t workspace_bytes, rlq_stream_t stream);

/*
 * AQN, adaptive quantization noise (QeRL news article: channel-wise Gaussian
 * perturbations mapped into the LayerNorm scale parameters, decaying on an
 * exponential schedule).  The pages give no formula; the one used here:
 *
 *   rlq_aqn_sigma:   *sigma = sigma_start * (sigma_end / sigma_start)^(t / (T - 1))
 *                    for step t of T (0 <= t < T): sigma_start at t = 0, sigma_end
 *                    at t = T - 1, geometric in between (computed in double,
 *                    rounded once to fp32).  T == 1 or equal levels give
 *                    sigma_start.  Levels must be finite and >= 0, and > 0 for a
 *                    decaying schedule.  Host-only: no stream, no GPU.
 *   rlq_aqn_perturb: gamma[k] = bf16_RN(fl32(gamma[k] + fl32(sigma * z[k]))), in
 *                    place, for k < K: gamma the norm scale (bf16 [K], 2-byte
 *                    aligned device memory), z one standard-normal draw per
 *                    channel (f32 [K] device memory, drawn by the caller), sigma
 *                    finite.  The product and the sum round separately.
 */
rlq_status rlq_aqn_sigma(float sigma_start, float sigma_end, int64_t t, int64_t T, float *sigma);

rlq_status rlq_aqn_perturb(uint16_t *gamma, int64_t K, const float *z, float sigma, rlq_stream_t stream);

/*
 * Split-K forms of the three GEMMs, for outputs too small to occupy every SM
 * (decode-sized M in FProp and DGrad, a narrow layer's WGrad).  The pages'
 * GEMMs do not prescribe a tiling; this is a scheduling choice of this
 * library.  The result follows the same formula as the single-pass call, with
 * the sum over contraction blocks taken in two levels: each split sums a
 * contiguous range of 128-blocks in fp32 (as the single-pass kernel does over
 * all of them), the split sums are added in split order in fp32, and the total
 * is rounded to bf16 once.  Results are deterministic (no atomics) but may
 * differ from the single-pass call in the last bits of the fp32 sum.
 *
 *   workspace        device scratch owned by the caller, 16-byte aligned, or
 *                    NULL (then the call is the single-pass GEMM); the kernels
 *                    write it before they read it, so its contents on entry
 *                    do not matter.  It must not be used by anything else
 *                    until the call has completed on `stream`.
 *   workspace_bytes  its size.  The library picks the number of splits from
 *                    the shape and the device's SM count, then lowers it until
 *                    the fp32 partials (splits * rows * cols * 4 bytes) fit;
 *                    with too little room it runs one pass.
 * Other arguments, shapes and errors are those of the single-pass call.
 *
 * rlq_gemm_splitk_workspace_bytes writes to *bytes the workspace size the
 * unconstrained plan uses on the current device for that GEMM and shape
 * (0 when the plan is one pass).
 */
typedef enum {
    RLQ_GEMM_FPROP = 0,
    RLQ_GEMM_DGRAD = 1,
    RLQ_GEMM_WGRAD = 2,
    RLQ_GEMM_NVFP4_WEIGHT_ONLY = 3 /* rlq_gemm_nvfp4_weight_only_splitk; M, N, K as in that call */
} rlq_gemm_kind;

rlq_status rlq_gemm_splitk_workspace_bytes(rlq_gemm_kind kind, int64_t M, int64_t N, int64_t K,
                                           int64_t *bytes);

rlq_status rlq_gemm_fprop_splitk(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs,
                                 const uint8_t *wq, int64_t ldwq, const float *ws, int64_t ldws,
                                 uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                 void *workspace, int64_t workspace_bytes, rlq_stream_t stream);

rlq_status rlq_gemm_dgrad_splitk(const uint8_t *dyq, int64_t lddyq, const float *dys, int64_t lddys,
                                 const uint8_t *w, int64_t ldw, int wq_is_transposed,
                                 const float *ws, int64_t ldws, uint16_t *dx, int64_t lddx,
                                 int64_t M, int64_t N, int64_t K,
                                 void *workspace, int64_t workspace_bytes, rlq_stream_t stream);

rlq_status rlq_gemm_wgrad_splitk(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc,
                                 const uint8_t *xqT, int64_t ldxqT, const float *xsc, int64_t ldxsc,
                                 uint16_t *dw, int64_t lddw, int64_t M, int64_t N, int64_t K,
                                 void *workspace, int64_t workspace_bytes, rlq_stream_t stream);

/*
 * Split-K FProp that allocates nothing: the workspace is a static scratch
 * array inside the library.  The pages have no counterpart to this call; it
 * serves callers that cannot allocate device memory: a host program that keeps
 * all device memory in its own pools and hands this library no allocator (an
 * inference engine that reserves HBM for weights and the KV cache at start-up,
 * or a plug-in inside one), or a real-time loop that must not call cudaMalloc
 * because of its implicit synchronisation.  The caller still owns and passes
 * every input and output.
 *
 *   Arguments and shapes are those of rlq_gemm_fprop_splitk.  The call runs
 *   the library's unconstrained split-K plan for (M, N, K) (the one
 *   rlq_gemm_splitk_workspace_bytes sizes), so its result is that of
 *   rlq_gemm_fprop_splitk given a workspace of at least that size.  When that
 *   plan needs more than RLQ_STATIC_SCRATCH_BYTES, the call returns
 *   RLQ_ERR_UNSUPPORTED and launches nothing; it does not fall back to a
 *   smaller plan (rlq_gemm_fprop_splitk with a caller's workspace of that
 *   size would).  A plan of one pass uses no scratch.
 *   The scratch (RLQ_STATIC_SCRATCH_BYTES, 16 MiB, in device memory) is held
 *   on every device that loads the library until the process exits.  The
 *   call itself calls no cudaMalloc, cudaFree or other allocating routine.
 *   The first call on a device in each CUDA context looks up the scratch's
 *   device address (cudaGetSymbolAddress, with that device current) and
 *   remembers it with the context; a call under a different context (after
 *   cudaDeviceReset, or under a context made current with the driver API)
 *   looks it up again.  Make the first call in a context before any stream
 *   capture.
 *   All calls on a device share the one scratch, which keeps whatever the
 *   last call left there; each call writes every scratch element it reads, so
 *   nothing needs clearing.  Calls whose executions overlap on the GPU (other
 *   streams, other host threads) race on the scratch and give wrong results:
 *   order them, for example on one stream.
 */
#define RLQ_STATIC_SCRATCH_BYTES 16777216

rlq_status rlq_gemm_fprop_splitk_static(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs,
                                        const uint8_t *wq, int64_t ldwq, const float *ws, int64_t ldws,
                                        uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                        rlq_stream_t stream);

/*
 * UAQ invariant-scaling fold, in place.  QuRL notes, 关键设计 §1: WX = (W/s)(sX)
 * with s > 1 applied per column of W and per row of the previous activation
 * (foldable into a LayerNorm / RMSNorm scale); run once before RL.
 *
 *   w     bf16 [N, K], pitch ldw >= K: w[n,k] <- bf16_RN(fl32(w[n,k] / s[k]))
 *   s     f32 [K], 16-byte aligned, every entry > 0 and finite (not checked on the device)
 *   prev  bf16 [R, K], pitch ldp >= K, nullable: prev[r,k] <- bf16_RN(fl32(prev[r,k] * s[k]))
 *         (the previous activation, R = M rows, or a norm weight, R = 1)
 * K % 8 == 0 (16-byte vectors); w / prev 16-byte aligned with pitches % 8 == 0.
 */
rlq_status rlq_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s,
                        uint16_t *prev, int64_t R, int64_t ldp, rlq_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns RLQ_ERR_TIMEOUT if a bounded wait ran out in an
 * earlier launch, RLQ_ERR_CUDA if CUDA reports an error, else RLQ_OK.
 */
rlq_status rlq_check(rlq_stream_t stream);

/*
 * Diagnostic for the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing will ever arrive on, for at most timeout_us microseconds
 * (1 .. 10^7), then records a timeout and exits.  The following rlq_check
 * returns RLQ_ERR_TIMEOUT and the context stays usable.
 */
rlq_status rlq_diag_bounded_wait(int64_t timeout_us, rlq_stream_t stream);

/*
 * Diagnostic for the block-scaled GEMM's own abort path: arms, for the calling
 * host thread, a one-shot fault in the next GEMM call it makes (any of the
 * FProp / DGrad / WGrad entry points).  That launch runs on single CTAs, and
 * the TMA producer of every CTA withholds the loads of its first pipeline
 * stage, so nothing ever arrives on that stage's barrier: the MMA warp's
 * bounded wait runs out (RLQ_WAIT_TIMEOUT_MS, 1 s by default), it records a
 * timeout and raises the CTA's abort flag, and the CTA drains its copies in
 * flight, frees its tensor memory and exits.  The output of that call is
 * undefined; the following rlq_check returns RLQ_ERR_TIMEOUT, and later calls
 * run normally.  Nothing faults, traps or hangs.  Host-only; always RLQ_OK.
 */
rlq_status rlq_diag_arm_gemm_stall(void);

/* Static description of a status code. */
const char *rlq_status_string(rlq_status status);

/* Description of the latest failure in the calling thread ("" if none). */
const char *rlq_last_error(void);

/* Library version, "major.minor.patch". */
const char *rlq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RLQ_H */
