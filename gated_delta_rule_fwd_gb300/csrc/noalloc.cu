// lr_fwd_chunked_noalloc: the chunked forward for callers that cannot
// allocate device memory.
//
// The bf16 chunked forward needs scratch memory between its two kernels
// (lr_fwd_chunked takes it as a caller-owned workspace).  Some callers cannot
// provide one: code running inside a host framework that owns every byte of
// device memory and offers no allocator to its plug-ins, and code on a path
// where cudaMalloc is not allowed because it may synchronise the device or
// fail at an unpredictable moment.  This entry point takes the scratch from a
// fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library is loaded holds LR_STATIC_WORKSPACE_BYTES for it until the process
// exits.  In host code the array's name only stands in for it (it is not a
// device address), so its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, the first time the entry
// point runs there, and kept for the life of the process (the device must not
// be reset while the library is loaded).  That first call should therefore
// come before any stream capture.  All calls share the one array: calls whose kernels may overlap on
// the GPU (different streams, or several host threads) race on it and must be
// serialised by the caller.  Each call rewrites every byte of scratch it
// reads, so nothing has to be cleared between calls.
#include <mutex>

#include "lr_internal.cuh"

namespace lr {
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[LR_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_workspace_ptr[kMaxDevices] = {};

// Device address of the static workspace on the current device (set up on
// first use).  Returns nullptr if it cannot be obtained.
void *static_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_workspace_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess) {
            cudaGetLastError();  // consume the error, so later launches do not report it
            return nullptr;
        }
        g_workspace_ptr[dev] = ptr;
    }
    return g_workspace_ptr[dev];
}

}  // namespace
}  // namespace lr

extern "C" lr_status lr_fwd_chunked_noalloc(const void *q, const void *k, const void *v,
                                            const float *alpha, const float *beta,
                                            const float *S0, void *o, float *S_T, int B, int H,
                                            int T, int dk, int dv, int chunk, lr_dtype dt,
                                            lr_mode mode, cudaStream_t stream) {
    const size_t need = lr_fwd_chunked_workspace_size(B, H, T, dk, dv, chunk, dt, mode);
    if (need > LR_STATIC_WORKSPACE_BYTES) return LR_ERR_TOO_LARGE;
    void *ws = nullptr;
    if (need > 0) {
        ws = lr::static_workspace();
        if (!ws) return LR_ERR_CUDA;
    }
    return lr_fwd_chunked(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, chunk, dt, mode, ws,
                          need > 0 ? (size_t)LR_STATIC_WORKSPACE_BYTES : 0, stream);
}
