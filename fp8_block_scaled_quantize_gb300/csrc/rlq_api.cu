// C ABI of librlq.so: host-side argument validation and dispatch to the
// kernels.  Every check runs before any launch; a failing call launches
// nothing and leaves a description for rlq_last_error().
#include <cmath>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "rlq_internal.h"

namespace rlq {

namespace {
thread_local char g_last_error[512] = "";
}

rlq_status fail(rlq_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

const char *last_error_text() { return g_last_error; }

rlq_status cuda_status(cudaError_t err, const char *what)
{
    if (err == cudaSuccess)
        return RLQ_OK;
    return fail(RLQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

}  // namespace rlq

using namespace rlq;

namespace {

constexpr int64_t G = 128;
constexpr int64_t MAX_DIM = (int64_t)1 << 31;  // TMA coordinates and tile indices are 32-bit

bool al(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

#define RLQ_REQUIRE(cond, code, ...)        \
    do {                                    \
        if (!(cond))                        \
            return fail((code), __VA_ARGS__); \
    } while (0)

// Code matrix [rows][cols] with pitch ld (bytes): TMA-ready.
rlq_status check_codes(const char *name, const void *p, int64_t ld, int64_t cols)
{
    RLQ_REQUIRE(p, RLQ_ERR_INVALID_ARG, "%s is NULL", name);
    RLQ_REQUIRE(ld >= cols, RLQ_ERR_INVALID_ARG, "%s: pitch %lld < row length %lld", name, (long long)ld, (long long)cols);
    RLQ_REQUIRE(al(p, 16), RLQ_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    RLQ_REQUIRE(ld % 16 == 0, RLQ_ERR_MISALIGNED, "%s: pitch %lld bytes is not a multiple of 16", name, (long long)ld);
    return RLQ_OK;
}

// bf16 matrix with pitch ld (elements).
rlq_status check_bf16(const char *name, const void *p, int64_t ld, int64_t cols)
{
    RLQ_REQUIRE(p, RLQ_ERR_INVALID_ARG, "%s is NULL", name);
    RLQ_REQUIRE(ld >= cols, RLQ_ERR_INVALID_ARG, "%s: pitch %lld < row length %lld", name, (long long)ld, (long long)cols);
    RLQ_REQUIRE(al(p, 16), RLQ_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    RLQ_REQUIRE(ld % 8 == 0, RLQ_ERR_MISALIGNED, "%s: pitch %lld elements is not a multiple of 8 (16 bytes)", name,
                (long long)ld);
    return RLQ_OK;
}

// fp32 scale array, s[b * ld + i] for i < extent.
rlq_status check_scales(const char *name, const void *p, int64_t ld, int64_t extent)
{
    RLQ_REQUIRE(p, RLQ_ERR_INVALID_ARG, "%s is NULL", name);
    RLQ_REQUIRE(ld >= extent, RLQ_ERR_INVALID_ARG, "%s: pitch %lld < %lld", name, (long long)ld, (long long)extent);
    RLQ_REQUIRE(al(p, 4), RLQ_ERR_MISALIGNED, "%s is not 4-byte aligned", name);
    return RLQ_OK;
}

#define RLQ_TRY(expr)                  \
    do {                               \
        const rlq_status _st = (expr); \
        if (_st != RLQ_OK)             \
            return _st;                \
    } while (0)

cudaStream_t cs(rlq_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

rlq_status rlq_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq, float *s,
                               int64_t lds, uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size (M=%lld, K=%lld)", (long long)M, (long long)K);
    RLQ_REQUIRE(K % G == 0, RLQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 128", (long long)K);
    RLQ_REQUIRE((qT == nullptr) == (sc == nullptr), RLQ_ERR_INVALID_ARG,
                "qT and sc must be both NULL (row-wise only) or both set (fused 128x1)");
    RLQ_REQUIRE(M < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("x", x, ldx, K));
    RLQ_TRY(check_codes("q", q, ldq, K));
    RLQ_TRY(check_scales("s", s, lds, M));
    if (qT) {
        RLQ_TRY(check_codes("qT", qT, ldqT, M));
        RLQ_TRY(check_scales("sc", sc, ldsc, K));
        return cuda_status(launch_quant_dual(x, M, K, ldx, q, ldq, s, lds, qT, ldqT, sc, ldsc, cs(stream)),
                           "1x128 + 128x1 quantizer launch");
    }
    return cuda_status(launch_quant_rows(x, M, K, ldx, q, ldq, s, lds, cs(stream)), "1x128 quantizer launch");
}

rlq_status rlq_rmsnorm_quant_act_1x128(const uint16_t *h, int64_t M, int64_t K, int64_t ldh, const uint16_t *gamma,
                                      float eps, float *rstd, uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                      uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size (M=%lld, K=%lld)", (long long)M, (long long)K);
    RLQ_REQUIRE(K % G == 0, RLQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 128", (long long)K);
    RLQ_REQUIRE((qT == nullptr) == (sc == nullptr), RLQ_ERR_INVALID_ARG,
                "qT and sc must be both NULL (row-wise only) or both set (fused 128x1)");
    RLQ_REQUIRE(M < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    RLQ_REQUIRE(std::isfinite(eps) && eps >= 0.0f, RLQ_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (M == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("h", h, ldh, K));
    RLQ_REQUIRE(gamma, RLQ_ERR_INVALID_ARG, "gamma is NULL");
    RLQ_REQUIRE(al(gamma, 16), RLQ_ERR_MISALIGNED, "gamma is not 16-byte aligned");
    RLQ_TRY(check_scales("rstd", rstd, M, M));
    RLQ_TRY(check_codes("q", q, ldq, K));
    RLQ_TRY(check_scales("s", s, lds, M));
    if (qT) {
        RLQ_TRY(check_codes("qT", qT, ldqT, M));
        RLQ_TRY(check_scales("sc", sc, ldsc, K));
    }
    RLQ_TRY(cuda_status(launch_rms_rstd(h, M, K, ldh, eps, rstd, cs(stream)), "RMSNorm row-factor launch"));
    if (qT)
        return cuda_status(launch_quant_dual(h, M, K, ldh, q, ldq, s, lds, qT, ldqT, sc, ldsc, cs(stream), rstd, gamma),
                           "RMSNorm + 1x128 + 128x1 quantizer launch");
    return cuda_status(launch_quant_rows(h, M, K, ldh, q, ldq, s, lds, cs(stream), rstd, gamma),
                       "RMSNorm + 1x128 quantizer launch");
}

rlq_status rlq_quant_per_row(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq, float *s,
                             float *s_rep, int64_t ld_rep, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size (M=%lld, K=%lld)", (long long)M, (long long)K);
    RLQ_REQUIRE(K % G == 0, RLQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 128", (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("x", x, ldx, K));
    RLQ_TRY(check_codes("q", q, ldq, K));
    RLQ_TRY(check_scales("s", s, M, M));
    if (s_rep)
        RLQ_TRY(check_scales("s_rep", s_rep, ld_rep, M));
    return cuda_status(launch_quant_per_row(x, M, K, ldx, q, ldq, s, s_rep, ld_rep, cs(stream)),
                       "per-row quantizer launch");
}

rlq_status rlq_quant_nvfp4(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, uint8_t *sb,
                           int64_t ldsb, float *st, rlq_stream_t stream)
{
    RLQ_REQUIRE(N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size (N=%lld, K=%lld)", (long long)N, (long long)K);
    RLQ_REQUIRE(K % 16 == 0, RLQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 16", (long long)K);
    RLQ_REQUIRE(N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    RLQ_REQUIRE(st, RLQ_ERR_INVALID_ARG, "st is NULL");
    RLQ_REQUIRE(al(st, 4), RLQ_ERR_MISALIGNED, "st is not 4-byte aligned");
    if (N == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("w", w, ldw, K));
    RLQ_REQUIRE(q, RLQ_ERR_INVALID_ARG, "q is NULL");
    RLQ_REQUIRE(ldq >= K / 2, RLQ_ERR_INVALID_ARG, "q: pitch %lld < %lld bytes", (long long)ldq, (long long)(K / 2));
    RLQ_REQUIRE(al(q, 8) && ldq % 8 == 0, RLQ_ERR_MISALIGNED, "q rows must be 8-byte aligned");
    RLQ_REQUIRE(sb, RLQ_ERR_INVALID_ARG, "sb is NULL");
    RLQ_REQUIRE(ldsb >= K / 16, RLQ_ERR_INVALID_ARG, "sb: pitch %lld < %lld", (long long)ldsb, (long long)(K / 16));
    return cuda_status(launch_quant_nvfp4(w, N, K, ldw, q, ldq, sb, ldsb, st, cs(stream)), "NVFP4 quantizer launch");
}

rlq_status rlq_quant_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                    float *s, int64_t lds, uint8_t *qT, int64_t ldqT, rlq_stream_t stream)
{
    RLQ_REQUIRE(N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size (N=%lld, K=%lld)", (long long)N, (long long)K);
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (N == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("w", w, ldw, K));
    RLQ_TRY(check_codes("q", q, ldq, K));
    RLQ_TRY(check_scales("s", s, lds, K / G));
    if (qT)
        RLQ_TRY(check_codes("qT", qT, ldqT, N));
    return cuda_status(launch_quant_weight(w, N, K, ldw, q, ldq, s, lds, qT, ldqT, cs(stream)),
                       "128x128 quantizer launch");
}

}  // extern "C"

namespace {

rlq_status check_workspace(const void *workspace, int64_t workspace_bytes)
{
    RLQ_REQUIRE(workspace_bytes >= 0, RLQ_ERR_INVALID_ARG, "workspace_bytes is negative");
    RLQ_REQUIRE(al(workspace, 16), RLQ_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    return RLQ_OK;
}

rlq_status gemm_fprop(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs, const uint8_t *wq, int64_t ldwq,
                      const float *ws, int64_t ldws, uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                      void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || N == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("y", y, ldy, N));
    if (K > 0) {
        RLQ_TRY(check_codes("xq", xq, ldxq, K));
        RLQ_TRY(check_codes("wq", wq, ldwq, K));
        RLQ_TRY(check_scales("xs", xs, ldxs, M));
        RLQ_TRY(check_scales("ws", ws, ldws, K / G));
    }
    GemmArgs a{};
    a.A = xq;
    a.lda = ldxq;
    a.B = wq;
    a.ldb = ldwq;
    a.sa = xs;
    a.ld_sa = ldxs;
    a.sb = ws;
    a.sb_bstride = 1;      // contraction block kb
    a.sb_cstride = ldws;   // output column block nb
    a.per_col_sb = false;
    a.out = y;
    a.ldo = ldy;
    a.R = M;
    a.C = N;
    a.L = K;
    a.ws = static_cast<float *>(workspace);
    a.ws_bytes = workspace_bytes;
    return launch_gemm(a, cs(stream));
}

rlq_status gemm_dgrad(const uint8_t *dyq, int64_t lddyq, const float *dys, int64_t lddys, const uint8_t *w, int64_t ldw,
                      int wq_is_transposed, const float *ws, int64_t ldws, uint16_t *dx, int64_t lddx, int64_t M,
                      int64_t N, int64_t K, void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(wq_is_transposed == 0 || wq_is_transposed == 1, RLQ_ERR_INVALID_ARG,
                "wq_is_transposed must be 0 or 1");
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("dx", dx, lddx, K));
    if (N > 0) {
        RLQ_TRY(check_codes("dyq", dyq, lddyq, N));
        RLQ_TRY(check_scales("dys", dys, lddys, M));
        RLQ_TRY(check_scales("ws", ws, ldws, K / G));
        if (wq_is_transposed)
            RLQ_TRY(check_codes("wqT", w, ldw, N));
        else
            RLQ_TRY(check_codes("wq", w, ldw, K));
    }
    GemmArgs a{};
    a.A = dyq;
    a.lda = lddyq;
    a.B = w;  // wqT [K rows][N] (output column k, contraction n), or wq [N rows][K] read MN-major
    a.ldb = ldw;
    a.b_mn_major = (wq_is_transposed == 0);
    a.sa = dys;
    a.ld_sa = lddys;
    a.sb = ws;             // scale of contraction block nb, output block kb: ws[nb * ldws + kb]
    a.sb_bstride = ldws;
    a.sb_cstride = 1;
    a.per_col_sb = false;
    a.out = dx;
    a.ldo = lddx;
    a.R = M;
    a.C = K;
    a.L = N;
    a.ws = static_cast<float *>(workspace);
    a.ws_bytes = workspace_bytes;
    return launch_gemm(a, cs(stream));
}

rlq_status gemm_wgrad(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc, const uint8_t *xqT,
                      int64_t ldxqT, const float *xsc, int64_t ldxsc, uint16_t *dw, int64_t lddw, int64_t M, int64_t N,
                      int64_t K, void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (N == 0 || K == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("dw", dw, lddw, K));
    if (M > 0) {
        RLQ_TRY(check_codes("dyqT", dyqT, lddyqT, M));
        RLQ_TRY(check_codes("xqT", xqT, ldxqT, M));
        RLQ_TRY(check_scales("dysc", dysc, lddysc, N));
        RLQ_TRY(check_scales("xsc", xsc, ldxsc, K));
        RLQ_REQUIRE(al(xsc, 16) && ldxsc % 4 == 0, RLQ_ERR_MISALIGNED,
                    "xsc rows must be 16-byte aligned (pointer 16-byte aligned, pitch a multiple of 4)");
    }
    GemmArgs a{};
    a.A = dyqT;
    a.lda = lddyqT;
    a.B = xqT;
    a.ldb = ldxqT;
    a.sa = dysc;
    a.ld_sa = lddysc;
    a.sb = xsc;
    a.sb_bstride = ldxsc;
    a.sb_cstride = 0;
    a.per_col_sb = true;
    a.out = dw;
    a.ldo = lddw;
    a.R = N;
    a.C = K;
    a.L = M;
    a.ws = static_cast<float *>(workspace);
    a.ws_bytes = workspace_bytes;
    return launch_gemm(a, cs(stream));
}

rlq_status gemm_fprop_per_channel(const uint8_t *xq, int64_t ldxq, const float *xs_rep, int64_t ldxs, const uint8_t *wq,
                                  int64_t ldwq, const float *ws_rep, int64_t ldws, uint16_t *y, int64_t ldy, int64_t M,
                                  int64_t N, int64_t K, void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || N == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("y", y, ldy, N));
    if (K > 0) {
        RLQ_TRY(check_codes("xq", xq, ldxq, K));
        RLQ_TRY(check_codes("wq", wq, ldwq, K));
        RLQ_TRY(check_scales("xs_rep", xs_rep, ldxs, M));
        RLQ_TRY(check_scales("ws_rep", ws_rep, ldws, N));
        RLQ_REQUIRE(al(ws_rep, 16) && ldws % 4 == 0, RLQ_ERR_MISALIGNED,
                    "ws_rep rows must be 16-byte aligned (pointer 16-byte aligned, pitch a multiple of 4)");
    }
    GemmArgs a{};
    a.A = xq;
    a.lda = ldxq;
    a.B = wq;
    a.ldb = ldwq;
    a.sa = xs_rep;
    a.ld_sa = ldxs;
    a.sb = ws_rep;
    a.sb_bstride = ldws;
    a.sb_cstride = 0;
    a.per_col_sb = true;
    a.scale_once = true;  // the scales are the same for every K-block: scale the whole sum once
    a.out = y;
    a.ldo = ldy;
    a.R = M;
    a.C = N;
    a.L = K;
    a.ws = static_cast<float *>(workspace);
    a.ws_bytes = workspace_bytes;
    return launch_gemm(a, cs(stream));
}

}  // namespace

extern "C" {

rlq_status rlq_gemm_fprop(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs, const uint8_t *wq,
                          int64_t ldwq, const float *ws, int64_t ldws, uint16_t *y, int64_t ldy, int64_t M, int64_t N,
                          int64_t K, rlq_stream_t stream)
{
    return gemm_fprop(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, nullptr, 0, stream);
}

rlq_status rlq_gemm_dgrad(const uint8_t *dyq, int64_t lddyq, const float *dys, int64_t lddys, const uint8_t *w,
                          int64_t ldw, int wq_is_transposed, const float *ws, int64_t ldws, uint16_t *dx, int64_t lddx,
                          int64_t M, int64_t N, int64_t K, rlq_stream_t stream)
{
    return gemm_dgrad(dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx, M, N, K, nullptr, 0,
                      stream);
}

rlq_status rlq_gemm_wgrad(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc, const uint8_t *xqT,
                          int64_t ldxqT, const float *xsc, int64_t ldxsc, uint16_t *dw, int64_t lddw, int64_t M,
                          int64_t N, int64_t K, rlq_stream_t stream)
{
    return gemm_wgrad(dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K, nullptr, 0, stream);
}

rlq_status rlq_gemm_fprop_per_channel(const uint8_t *xq, int64_t ldxq, const float *xs_rep, int64_t ldxs,
                                      const uint8_t *wq, int64_t ldwq, const float *ws_rep, int64_t ldws, uint16_t *y,
                                      int64_t ldy, int64_t M, int64_t N, int64_t K, rlq_stream_t stream)
{
    return gemm_fprop_per_channel(xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N, K, nullptr, 0, stream);
}

rlq_status rlq_gemm_splitk_workspace_bytes(rlq_gemm_kind kind, int64_t M, int64_t N, int64_t K, int64_t *bytes)
{
    RLQ_REQUIRE(bytes, RLQ_ERR_INVALID_ARG, "bytes is NULL");
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    int64_t R, C, L;
    switch (kind) {
    case RLQ_GEMM_FPROP:
        R = M, C = N, L = K;
        break;
    case RLQ_GEMM_DGRAD:
        R = M, C = K, L = N;
        break;
    case RLQ_GEMM_WGRAD:
        R = N, C = K, L = M;
        break;
    case RLQ_GEMM_NVFP4_WEIGHT_ONLY: {
        int splits = 1;
        return plan_nvfp4_splitk(M, N, K, -1, &splits, bytes);
    }
    default:
        return fail(RLQ_ERR_INVALID_ARG, "unknown GEMM kind %d", (int)kind);
    }
    int splits = 1;
    return plan_splitk(R, C, L, -1, &splits, bytes);
}

rlq_status rlq_gemm_fprop_splitk(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs, const uint8_t *wq,
                                 int64_t ldwq, const float *ws, int64_t ldws, uint16_t *y, int64_t ldy, int64_t M,
                                 int64_t N, int64_t K, void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    return gemm_fprop(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, workspace, workspace_bytes, stream);
}

rlq_status rlq_gemm_wgrad_accumulate(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc,
                                     const uint8_t *xqT, int64_t ldxqT, const float *xsc, int64_t ldxsc, float *dw_acc,
                                     int64_t ld_acc, int64_t M, int64_t N, int64_t K, void *workspace,
                                     int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % G == 0, RLQ_ERR_UNSUPPORTED, "N=%lld and K=%lld must be multiples of 128",
                (long long)N, (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (N == 0 || K == 0 || M == 0)
        return RLQ_OK;  // nothing to add
    RLQ_REQUIRE(dw_acc, RLQ_ERR_INVALID_ARG, "dw_acc is NULL");
    RLQ_REQUIRE(ld_acc >= K, RLQ_ERR_INVALID_ARG, "dw_acc: pitch %lld < %lld", (long long)ld_acc, (long long)K);
    RLQ_REQUIRE(al(dw_acc, 16) && ld_acc % 4 == 0, RLQ_ERR_MISALIGNED,
                "dw_acc rows must be 16-byte aligned (pointer 16-byte aligned, pitch a multiple of 4)");
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    RLQ_TRY(check_codes("dyqT", dyqT, lddyqT, M));
    RLQ_TRY(check_codes("xqT", xqT, ldxqT, M));
    RLQ_TRY(check_scales("dysc", dysc, lddysc, N));
    RLQ_TRY(check_scales("xsc", xsc, ldxsc, K));
    RLQ_REQUIRE(al(xsc, 16) && ldxsc % 4 == 0, RLQ_ERR_MISALIGNED,
                "xsc rows must be 16-byte aligned (pointer 16-byte aligned, pitch a multiple of 4)");
    GemmArgs a{};
    a.A = dyqT;
    a.lda = lddyqT;
    a.B = xqT;
    a.ldb = ldxqT;
    a.sa = dysc;
    a.ld_sa = lddysc;
    a.sb = xsc;
    a.sb_bstride = ldxsc;
    a.sb_cstride = 0;
    a.per_col_sb = true;
    // the epilogue adds into dw_acc (or, where the split-K plan splits, writes
    // fp32 partials that a reduction adds); no bf16 output
    a.out = nullptr;
    a.ldo = 0;
    a.R = N;
    a.C = K;
    a.L = M;
    a.ws = static_cast<float *>(workspace);
    a.ws_bytes = workspace_bytes;
    a.acc = dw_acc;
    a.ld_acc = ld_acc;
    return launch_gemm(a, cs(stream));
}

rlq_status rlq_gemm_fprop_per_channel_splitk(const uint8_t *xq, int64_t ldxq, const float *xs_rep, int64_t ldxs,
                                             const uint8_t *wq, int64_t ldwq, const float *ws_rep, int64_t ldws,
                                             uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                             void *workspace, int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    return gemm_fprop_per_channel(xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N, K, workspace,
                                  workspace_bytes, stream);
}

rlq_status rlq_gemm_dgrad_splitk(const uint8_t *dyq, int64_t lddyq, const float *dys, int64_t lddys, const uint8_t *w,
                                 int64_t ldw, int wq_is_transposed, const float *ws, int64_t ldws, uint16_t *dx,
                                 int64_t lddx, int64_t M, int64_t N, int64_t K, void *workspace,
                                 int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    return gemm_dgrad(dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx, M, N, K, workspace,
                      workspace_bytes, stream);
}

rlq_status rlq_gemm_wgrad_splitk(const uint8_t *dyqT, int64_t lddyqT, const float *dysc, int64_t lddysc,
                                 const uint8_t *xqT, int64_t ldxqT, const float *xsc, int64_t ldxsc, uint16_t *dw,
                                 int64_t lddw, int64_t M, int64_t N, int64_t K, void *workspace,
                                 int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    return gemm_wgrad(dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K, workspace,
                      workspace_bytes, stream);
}

rlq_status rlq_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s, uint16_t *prev, int64_t R,
                        int64_t ldp, rlq_stream_t stream)
{
    RLQ_REQUIRE(N >= 0 && K >= 0 && R >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(K % 8 == 0, RLQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 8", (long long)K);
    if (K == 0 || (N == 0 && (prev == nullptr || R == 0)))
        return RLQ_OK;
    RLQ_REQUIRE(s, RLQ_ERR_INVALID_ARG, "s is NULL");
    RLQ_REQUIRE(al(s, 16), RLQ_ERR_MISALIGNED, "s is not 16-byte aligned");
    if (N > 0)
        RLQ_TRY(check_bf16("w", w, ldw, K));
    if (prev && R > 0)
        RLQ_TRY(check_bf16("prev", prev, ldp, K));
    return cuda_status(launch_uaq_fold(w, N, K, ldw, s, prev, R, ldp, cs(stream)), "UAQ fold launch");
}

}  // extern "C"

namespace {

rlq_status gemm_nvfp4(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq, const uint8_t *wsb, int64_t ldwsb,
                      const float *wst, uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K, void *workspace,
                      int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_REQUIRE(M >= 0 && N >= 0 && K >= 0, RLQ_ERR_INVALID_ARG, "negative size");
    RLQ_REQUIRE(N % G == 0 && K % 64 == 0, RLQ_ERR_UNSUPPORTED,
                "N=%lld must be a multiple of 128 and K=%lld a multiple of 64", (long long)N, (long long)K);
    RLQ_REQUIRE(M < MAX_DIM && N < MAX_DIM && K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    if (M == 0 || N == 0)
        return RLQ_OK;
    RLQ_TRY(check_bf16("y", y, ldy, N));
    if (K == 0)  // empty contraction: the sum is zero
        return cuda_status(cudaMemset2DAsync(y, (size_t)ldy * 2, 0, (size_t)N * 2, (size_t)M, cs(stream)),
                           "cudaMemset2DAsync (empty contraction)");
    RLQ_TRY(check_bf16("x", x, ldx, K));
    RLQ_TRY(check_codes("wq", wq, ldwq, K / 2));
    RLQ_TRY(check_codes("wsb", wsb, ldwsb, K / 16));
    RLQ_REQUIRE(wst, RLQ_ERR_INVALID_ARG, "wst is NULL");
    RLQ_REQUIRE(al(wst, 4), RLQ_ERR_MISALIGNED, "wst is not 4-byte aligned");
    return launch_gemm_nvfp4w(x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, workspace, workspace_bytes,
                              cs(stream));
}

}  // namespace

extern "C" {

rlq_status rlq_gemm_nvfp4_weight_only(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq,
                                     const uint8_t *wsb, int64_t ldwsb, const float *wst, uint16_t *y, int64_t ldy,
                                     int64_t M, int64_t N, int64_t K, rlq_stream_t stream)
{
    return gemm_nvfp4(x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, nullptr, 0, stream);
}

rlq_status rlq_gemm_nvfp4_weight_only_splitk(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq,
                                            const uint8_t *wsb, int64_t ldwsb, const float *wst, uint16_t *y,
                                            int64_t ldy, int64_t M, int64_t N, int64_t K, void *workspace,
                                            int64_t workspace_bytes, rlq_stream_t stream)
{
    RLQ_TRY(check_workspace(workspace, workspace_bytes));
    return gemm_nvfp4(x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, workspace, workspace_bytes, stream);
}

rlq_status rlq_aqn_sigma(float sigma_start, float sigma_end, int64_t t, int64_t T, float *sigma)
{
    RLQ_REQUIRE(sigma, RLQ_ERR_INVALID_ARG, "sigma is NULL");
    RLQ_REQUIRE(T >= 1 && t >= 0 && t < T, RLQ_ERR_INVALID_ARG, "step t=%lld outside 0 .. T-1 (T=%lld)", (long long)t,
                (long long)T);
    RLQ_REQUIRE(std::isfinite(sigma_start) && std::isfinite(sigma_end) && sigma_start >= 0.0f && sigma_end >= 0.0f,
                RLQ_ERR_INVALID_ARG, "noise levels must be finite and >= 0");
    if (T == 1 || sigma_start == sigma_end || t == 0) {
        *sigma = sigma_start;
        return RLQ_OK;
    }
    if (t == T - 1) {
        *sigma = sigma_end;
        return RLQ_OK;
    }
    RLQ_REQUIRE(sigma_start > 0.0f && sigma_end > 0.0f, RLQ_ERR_INVALID_ARG,
                "a decaying schedule needs sigma_start > 0 and sigma_end > 0");
    // geometric: sigma_start * (sigma_end / sigma_start)^(t / (T - 1)), in double, rounded once
    const double frac = (double)t / (double)(T - 1);
    *sigma = (float)((double)sigma_start * std::exp(frac * std::log((double)sigma_end / (double)sigma_start)));
    return RLQ_OK;
}

rlq_status rlq_aqn_perturb(uint16_t *gamma, int64_t K, const float *z, float sigma, rlq_stream_t stream)
{
    RLQ_REQUIRE(K >= 0, RLQ_ERR_INVALID_ARG, "negative size K=%lld", (long long)K);
    RLQ_REQUIRE(K < MAX_DIM, RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    RLQ_REQUIRE(std::isfinite(sigma), RLQ_ERR_INVALID_ARG, "sigma is not finite");
    if (K == 0)
        return RLQ_OK;
    RLQ_REQUIRE(gamma && z, RLQ_ERR_INVALID_ARG, "gamma or z is NULL");
    RLQ_REQUIRE(al(gamma, 2) && al(z, 4), RLQ_ERR_MISALIGNED, "gamma must be 2-byte and z 4-byte aligned");
    return cuda_status(launch_aqn_perturb(gamma, K, z, sigma, cs(stream)), "AQN launch");
}

rlq_status rlq_check(rlq_stream_t stream) { return check_device_errors(cs(stream)); }

rlq_status rlq_diag_bounded_wait(int64_t timeout_us, rlq_stream_t stream)
{
    RLQ_REQUIRE(timeout_us >= 1 && timeout_us <= 10000000, RLQ_ERR_INVALID_ARG, "timeout_us must be in 1 .. 10^7");
    return launch_diag_wait(timeout_us, cs(stream));
}

rlq_status rlq_diag_arm_gemm_stall(void)
{
    arm_gemm_stall();
    return RLQ_OK;
}

const char *rlq_status_string(rlq_status status)
{
    switch (status) {
    case RLQ_OK:
        return "RLQ_OK";
    case RLQ_ERR_INVALID_ARG:
        return "RLQ_ERR_INVALID_ARG: invalid argument";
    case RLQ_ERR_UNSUPPORTED:
        return "RLQ_ERR_UNSUPPORTED: unsupported shape";
    case RLQ_ERR_MISALIGNED:
        return "RLQ_ERR_MISALIGNED: pointer or pitch breaks the alignment rules";
    case RLQ_ERR_CUDA:
        return "RLQ_ERR_CUDA: CUDA call or launch failed";
    case RLQ_ERR_TIMEOUT:
        return "RLQ_ERR_TIMEOUT: a bounded device-side wait ran out";
    }
    return "unknown rlq_status";
}

const char *rlq_last_error(void) { return last_error_text(); }

const char *rlq_version(void) { return "0.1.0"; }

}  // extern "C"
