// Split-K FProp on scratch memory that the library owns, for callers that
// cannot allocate device memory.
//
// Who needs it: a host program that hands this library no allocator and keeps
// every byte of device memory in its own pools (an inference engine that
// reserves HBM for weights and the KV cache at start-up), a plug-in that runs
// inside such a program, or a real-time loop that must not call cudaMalloc,
// whose implicit synchronisation would stall the other streams.  These callers
// can pass inputs and outputs they already own, but cannot obtain the split-K
// workspace that rlq_gemm_fprop_splitk wants.
//
// The scratch is a file-scope __device__ array of RLQ_STATIC_SCRATCH_BYTES;
// every device that loads the library holds it until the process exits.  In
// host code `g_static_scratch` is only a host-side stand-in for the symbol:
// its device address comes from cudaGetSymbolAddress, with the device current,
// on the first call made on that device in a given CUDA context.  The address
// is remembered per device together with the context it was looked up in: a
// call under another context (after cudaDeviceReset rebuilt the primary
// context, or under a context the caller made current with the driver API)
// looks it up again, since the module, and with it the array, may then sit
// elsewhere.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "rlq_internal.h"

namespace rlq {
namespace {

static_assert(RLQ_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte granularity");

static __device__ __align__(256) float g_static_scratch[RLQ_STATIC_SCRATCH_BYTES / sizeof(float)];

constexpr int MAX_DEVICES = 64;

struct ScratchTable {
    std::mutex mu;
    void *ptr[MAX_DEVICES] = {};
    CUcontext ctx[MAX_DEVICES] = {};  // context each address was looked up in
};

ScratchTable &scratch_table()
{
    static ScratchTable t;
    return t;
}

// The calling thread's current CUDA context (NULL if none), through the
// driver entry point the runtime exposes; no library beyond the runtime is
// linked for it.
CUcontext current_context()
{
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    });
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS)
        return nullptr;
    return c;
}

// Device address of the static scratch on the current device, looked up on
// the first call in each context.
rlq_status static_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES)
        return fail(RLQ_ERR_UNSUPPORTED, "device ordinal %d is beyond the %d devices the static scratch tracks", dev,
                    MAX_DEVICES);
    ScratchTable &t = scratch_table();
    std::lock_guard<std::mutex> g(t.mu);
    CUcontext ctx = current_context();
    if (t.ptr[dev] == nullptr || ctx == nullptr || ctx != t.ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaGetSymbolAddress(static split-K scratch)");
        if (p == nullptr || ((uintptr_t)p & 255u) != 0)
            return fail(RLQ_ERR_CUDA, "static split-K scratch has an unexpected device address %p", p);
        // the lookup made the device's primary context current if none was
        ctx = current_context();
        t.ptr[dev] = p;
        t.ctx[dev] = ctx;
    }
    *out = t.ptr[dev];
    return RLQ_OK;
}

}  // namespace
}  // namespace rlq

extern "C" rlq_status rlq_gemm_fprop_splitk_static(const uint8_t *xq, int64_t ldxq, const float *xs, int64_t ldxs,
                                                   const uint8_t *wq, int64_t ldwq, const float *ws, int64_t ldws,
                                                   uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                                   rlq_stream_t stream)
{
    using namespace rlq;
    if (M < 0 || N < 0 || K < 0)
        return fail(RLQ_ERR_INVALID_ARG, "negative size");
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31))
        return fail(RLQ_ERR_UNSUPPORTED, "dimension beyond 2^31");
    void *scratch = nullptr;
    rlq_status st = static_scratch(&scratch);
    if (st != RLQ_OK)
        return st;
    int64_t need = 0;
    st = rlq_gemm_splitk_workspace_bytes(RLQ_GEMM_FPROP, M, N, K, &need);
    if (st != RLQ_OK)
        return st;
    if (need > (int64_t)RLQ_STATIC_SCRATCH_BYTES)
        return fail(RLQ_ERR_UNSUPPORTED,
                    "split-K FProp of M=%lld N=%lld K=%lld needs %lld bytes of scratch, beyond the %lld-byte static "
                    "scratch; call rlq_gemm_fprop_splitk with a workspace, or rlq_gemm_fprop",
                    (long long)M, (long long)N, (long long)K, (long long)need, (long long)RLQ_STATIC_SCRATCH_BYTES);
    // With a cap at least as large as the plan's workspace, the plan (and so
    // the result) is the one rlq_gemm_fprop_splitk makes with any workspace
    // of `need` bytes or more.  Every partial the reduction reads is written
    // first by the same call, so the scratch needs no clearing.
    return rlq_gemm_fprop_splitk(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, scratch,
                                 (int64_t)RLQ_STATIC_SCRATCH_BYTES, stream);
}
