// Internal declarations shared by the translation units of librlq.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rlq.h"

namespace rlq {

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialization allowed and begins with pdl_begin(), which
// first waits until the grids it depends on (the previous kernels in the stream)
// have completed and their memory is visible, and then lets the next kernel in
// the stream be scheduled as soon as every block of this grid has started.  The
// next kernel's blocks can then be resident and waiting when this grid ends,
// instead of being launched only afterwards.  No kernel touches global memory
// before the wait, so the ordering of the stream is unchanged.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records a failure description for rlq_last_error() and returns `st`.
rlq_status fail(rlq_status st, const char *fmt, ...);

// Text of the latest failure in the calling thread.
const char *last_error_text();

// Maps a CUDA error (if any) to RLQ_ERR_CUDA with a description.
rlq_status cuda_status(cudaError_t err, const char *what);

// ---- quantizers and fold (rlq_quant.cu); arguments already validated ----
// With rstd and gamma set, x is a hidden state normalised on the fly
// (x = bf16_RN(fl32(fl32(h * rstd[m]) * gamma[k]))) before quantization.
cudaError_t launch_quant_rows(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                              int64_t ldq, float *s, int64_t lds, cudaStream_t st,
                              const float *rstd = nullptr, const uint16_t *gamma = nullptr);
cudaError_t launch_quant_dual(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                              int64_t ldq, float *s, int64_t lds, uint8_t *qT, int64_t ldqT,
                              float *sc, int64_t ldsc, cudaStream_t st,
                              const float *rstd = nullptr, const uint16_t *gamma = nullptr);
// rstd[m] = fl32(1 / sqrt(fl32(fl32(sum_k h[m,k]^2 / K) + eps))), the sum in index order.
cudaError_t launch_rms_rstd(const uint16_t *h, int64_t M, int64_t K, int64_t ldh, float eps, float *rstd,
                            cudaStream_t st);
cudaError_t launch_quant_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q,
                                int64_t ldq, float *s, int64_t lds, uint8_t *qT, int64_t ldqT,
                                cudaStream_t st);
cudaError_t launch_quant_per_row(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                                 int64_t ldq, float *s, float *s_rep, int64_t ld_rep, cudaStream_t st);
cudaError_t launch_quant_nvfp4(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                               uint8_t *sb, int64_t ldsb, float *st, cudaStream_t st_stream);
cudaError_t launch_aqn_perturb(uint16_t *gamma, int64_t K, const float *z, float sigma, cudaStream_t st);
cudaError_t launch_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s,
                            uint16_t *prev, int64_t R, int64_t ldp, cudaStream_t st);

// ---- block-scaled GEMM (rlq_gemm.cu) ----
//
// out[r, c] = bf16( sum_b sa(b, r) * sb(b, c) * sum_{j in block b} A[r, j] * B[c, j] )
// A: E4M3 [R rows][L contraction], pitch lda bytes; B: E4M3 [C rows][L], pitch ldb.
// sa(b, r) = sa[b * ld_sa + r].
// B is [C rows][L] (K-major) or, with b_mn_major, [L rows][C] (the FProp weight
// codes read as DGrad's operand without a transposed copy); pitch ldb bytes.
// Block-scaled B (per_col_sb == false): sb(b, c) = sb[b * sb_bstride + (c / 128) * sb_cstride].
// Column-scaled B (per_col_sb == true):  sb(b, c) = sb[b * sb_bstride + c], rows 16-byte aligned.
struct GemmArgs {
    const uint8_t *A;
    int64_t lda;
    const uint8_t *B;
    int64_t ldb;
    const float *sa;
    int64_t ld_sa;
    const float *sb;
    int64_t sb_bstride;
    int64_t sb_cstride;
    bool per_col_sb;
    bool b_mn_major;
    // sa(b, r) and sb(b, c) equal for every contraction block b (per-token x
    // per-channel scales, sb column-scaled): the contraction is accumulated in
    // the tensor cores and scaled once
    bool scale_once;
    uint16_t *out;
    int64_t ldo;
    int64_t R, C, L;
    // split-K workspace (16-byte aligned fp32), or NULL for the single-pass GEMM
    float *ws;
    int64_t ws_bytes;
    // accumulate mode: acc[r * ld_acc + c] += the fp32 result (out is not written),
    // from the GEMM's epilogue, or from the split-K partials where the plan splits
    float *acc;
    int64_t ld_acc;
};
rlq_status launch_gemm(const GemmArgs &a, cudaStream_t st);

// ---- NVFP4 weight-only GEMM (rlq_gemm_nvfp4.cu); arguments already validated ----
// Y[M, N] = bf16(st * X W^T), X bf16 [M, K] (pitch ldx elements), W from packed
// E2M1 codes wq [N, K/2] (pitch ldwq bytes) and E4M3 block scales wsb [N, K/16]
// (pitch ldwsb bytes), st one fp32 in device memory.  K % 64 == 0, K > 0.
// workspace (16-byte aligned, or NULL for one pass) holds the split plan's fp32
// partials; the plan is lowered until they fit workspace_bytes.
rlq_status launch_gemm_nvfp4w(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq, const uint8_t *wsb,
                              int64_t ldwsb, const float *st, uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                              void *workspace, int64_t workspace_bytes, cudaStream_t stream);
// Split count and workspace bytes (splits * M * N * 4, or 0 for one pass) of the
// NVFP4 GEMM's split plan on the current device; ws_cap limits the workspace
// (-1: no limit).
rlq_status plan_nvfp4_splitk(int64_t M, int64_t N, int64_t K, int64_t ws_cap, int *splits, int64_t *ws_bytes);
// out[r, c] = bf16_RN(sum over s < splits, in order, of ws[(s * R + r) * C + c]),
// C % 8 == 0, on `sms` SMs' worth of blocks at most.
rlq_status launch_splitk_reduce(const float *ws, int splits, int64_t R, int64_t C, uint16_t *out, int64_t ldo, int sms,
                                cudaStream_t st);

// Number of contraction splits the split-K GEMM uses for an [R x C] output
// with contraction length L on the current device, and the workspace bytes
// (splits * R * C * 4, or 0 for one split) it needs.  ws_cap limits the
// workspace (-1: no limit).
rlq_status plan_splitk(int64_t R, int64_t C, int64_t L, int64_t ws_cap, int *splits, int64_t *ws_bytes);

// Reads and clears the device error words of the current device (after syncing st).
rlq_status check_device_errors(cudaStream_t st);
// The NVFP4 GEMM's translation unit's error word, read and cleared (0: none).
cudaError_t take_nvfp4_error_word(cudaStream_t st, unsigned long long *word);
rlq_status launch_diag_wait(int64_t timeout_us, cudaStream_t st);

// Arms, for the calling thread, a one-shot stall of the next block-scaled GEMM
// launch: it runs on single CTAs and its producer withholds the first stage's
// loads, so the MMA warp's bounded wait runs out and the CTA takes its abort path.
void arm_gemm_stall();

}  // namespace rlq
