// Internal declarations shared by the CUDA translation units of liblr.
// Nothing here is part of the C ABI (include/lr.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lr.h"

namespace lr {

// ---------------------------------------------------------------- conversions
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Four consecutive elements widened to fp32 (16-byte aligned for float,
// 8-byte aligned for bf16).
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    float4 r;
    r.x = __uint_as_float(raw.x << 16);
    r.y = __uint_as_float(raw.x & 0xffff0000u);
    r.z = __uint_as_float(raw.y << 16);
    r.w = __uint_as_float(raw.y & 0xffff0000u);
    return r;
}

// Mode flags as compile-time properties.
struct ModeBits {
    bool alpha;  // the state decays by alpha_t
    bool delta;  // the write is the corrected (delta-rule) pseudo-value
};
__host__ __device__ constexpr ModeBits mode_bits(int mode) {
    return ModeBits{mode == LR_MODE_DECAY || mode == LR_MODE_GATED_DELTA,
                    mode == LR_MODE_DELTA || mode == LR_MODE_GATED_DELTA};
}

// ------------------------------------------------------------------ launchers
// Every launcher assumes arguments already validated by lr_api.cu and returns
// the cudaError_t of the launch.

// Decode step (decode.cu).
cudaError_t launch_step(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                        lr_dtype dt, lr_mode mode, cudaStream_t stream);

// Chunked forward on CUDA cores in fp32 (chunked_simt.cu).
cudaError_t launch_chunked_simt(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *S_T, int B,
                                int H, int T, int dk, int dv, lr_dtype dt, lr_mode mode,
                                cudaStream_t stream);

// Chunked forward on the tensor cores, bf16 (chunked_tc.cu).
cudaError_t launch_chunked_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *S_T, int B,
                              int H, int T, int dk, int dv, lr_mode mode, void *ws,
                              cudaStream_t stream);
// Workspace bytes the tensor-core path needs.
size_t chunked_tc_workspace_bytes(int B, int H, int T, int dk);

// Returns and clears the tensor-core kernel's bounded-wait error word
// (1 if set, 0 if clear, -1 if the device could not be read).
int read_and_clear_tc_error();

// Set the dynamic shared-memory limit of `fn` once per device.
cudaError_t ensure_smem_attr(const void *fn, int bytes, int slot);

}  // namespace lr
