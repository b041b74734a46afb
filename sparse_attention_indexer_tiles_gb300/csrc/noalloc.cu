// idx_score_topk_noalloc: the fused score + exact top-k for callers that
// cannot allocate device memory.
//
// Some callers only ever receive pointers to memory that someone else owns: a
// plugin inside a host framework that manages all device memory and offers its
// extensions no allocator, or a latency-critical serving loop that must not
// call cudaMalloc (which may synchronize the device and fragments the heap).
// Such a caller cannot provide idx_score_topk's workspace.  This entry point
// runs the same launch sequence on a scratch array compiled into the library
// instead, and allocates nothing itself.
#include <cstddef>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/idx.h"

namespace {

// The scratch every call uses.  A __device__ array lives in the module image:
// each GPU that loads this library holds IDX_NOALLOC_SCRATCH_BYTES of it until
// the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[IDX_NOALLOC_SCRATCH_BYTES];

// In host code the array's name is only a host-side stand-in, so its device
// address is looked up (cudaGetSymbolAddress, with the device current) the
// first time a device calls, and cached together with the CUDA context it
// belongs to: after cudaDeviceReset the device gets a new primary context and
// a new copy of the array, and the next call looks the address up again.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrent = CUresult (*)(CUcontext*);

CtxGetCurrent ctx_get_current() {
    static std::once_flag once;
    static CtxGetCurrent fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrent>(p);
    });
    return fn;
}

idx_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return IDX_ECUDA;
    }
    CtxGetCurrent get = ctx_get_current();
    if (!get) return IDX_ECUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return IDX_ECUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        // the lookup also makes the device's primary context current when no
        // context was yet
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return IDX_ECUDA;
        }
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return IDX_ECUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return IDX_OK;
}

}  // namespace

extern "C" idx_status idx_score_topk_noalloc(const void* q, const void* k, const float* k_scale,
                                              const float* w, const int* ks, const int* ke,
                                              int rows, long long keys, long long max_len, int H,
                                              int D, int topk, idx_dtype dt, int* out_idx,
                                              const idx_options* opt, void* stream) {
    // no rows: idx_score_topk validates the other arguments and launches nothing
    if (rows <= 0)
        return idx_score_topk(q, k, k_scale, w, ks, ke, rows, keys, max_len, H, D, topk, dt,
                              out_idx, nullptr, 0, opt, stream);
    // the workspace this problem needs must fit in the built-in scratch array
    const size_t need = idx_score_topk_workspace(rows, keys, max_len, H, D, topk, dt, opt);
    if (need > (size_t)IDX_NOALLOC_SCRATCH_BYTES) return IDX_EWORKSPACE;
    void* scratch = nullptr;
    const idx_status st = scratch_for_current_device(&scratch);
    if (st != IDX_OK) return st;
    // Every word of the workspace that the launch sequence reads is written
    // earlier in the same call, so nothing needs clearing between calls.
    return idx_score_topk(q, k, k_scale, w, ks, ke, rows, keys, max_len, H, D, topk, dt, out_idx,
                          scratch, (size_t)IDX_NOALLOC_SCRATCH_BYTES, opt, stream);
}
