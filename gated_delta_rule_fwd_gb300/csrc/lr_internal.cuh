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

// fp32 -> bf16, rounded to nearest even, through the paired conversion
// instruction (same bits as the single-value conversion, which is slower on
// this target).
__device__ __forceinline__ __nv_bfloat16 bf16_rn(float x) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(x));
    return __ushort_as_bfloat16((unsigned short)(r & 0xffffu));
}

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return bf16_rn(x);
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
    return ModeBits{mode == LR_MODE_DECAY || mode == LR_MODE_GATED_DELTA ||
                        mode == LR_MODE_DIAG_DECAY,
                    mode == LR_MODE_DELTA || mode == LR_MODE_GATED_DELTA};
}

// ------------------------------------------------- maps around the recurrence
// The lr_fuse options as the kernels receive them (validated on the host).
struct Fuse {
    unsigned flags = 0;
    const float *ascale = nullptr;  // [H], c_h of the softplus gate
    const float *norm_w = nullptr;  // [dv] or NULL for ones
    float norm_eps = 0.f;
};

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }
// ln(1 + e^x) without overflow
__device__ __forceinline__ float softplus_f(float x) {
    return fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x)));
}
// x sigmoid(x)
__device__ __forceinline__ float silu_f(float x) { return x / (1.f + __expf(-x)); }
// 1 / max(sqrt(ss), 1e-12): the scale that L2-normalises a vector with sum of squares ss
__device__ __forceinline__ float inv_l2(float ss) { return rsqrtf(fmaxf(ss, 1e-24f)); }

// ln alpha from the value read from memory: ln a without a gate map,
// ln sigmoid(a) = -softplus(-a), -c softplus(a), or c ln sigmoid(a).
__device__ __forceinline__ float log_gate(unsigned fl, float a, float c) {
    if (fl & LR_FUSE_ALPHA_SIGMOID) return -softplus_f(-a);
    if (fl & LR_FUSE_ALPHA_SOFTPLUS) return -c * softplus_f(a);
    if (fl & LR_FUSE_ALPHA_SIGMOID_POW) return -c * softplus_f(-a);
    return __logf(a);
}
// alpha itself (decode, and the products of the diagonal gate)
__device__ __forceinline__ float gate(unsigned fl, float a, float c) {
    if (fl & LR_FUSE_ALPHA_SIGMOID) return sigmoid_f(a);
    if (fl & LR_FUSE_ALPHA_SOFTPLUS) return __expf(-c * softplus_f(a));
    if (fl & LR_FUSE_ALPHA_SIGMOID_POW) return __expf(-c * softplus_f(-a));
    return a;
}
// the alpha maps that take c_h from alpha_scale
constexpr unsigned kScaledAlphaMaps = LR_FUSE_ALPHA_SOFTPLUS | LR_FUSE_ALPHA_SIGMOID_POW;
constexpr unsigned kAlphaMaps = LR_FUSE_ALPHA_SIGMOID | kScaledAlphaMaps;
__device__ __forceinline__ float write_strength(unsigned fl, float b) {
    return (fl & LR_FUSE_BETA_SIGMOID) ? sigmoid_f(b) : b;
}

// ------------------------------------------------------------------ launchers
// Every launcher assumes arguments already validated by lr_api.cu and returns
// the cudaError_t of the launch.

// Decode step (decode.cu).
cudaError_t launch_step(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                        lr_dtype dt, lr_mode mode, const Fuse &fz, cudaStream_t stream);

// Chunked forward on CUDA cores in fp32 (chunked_simt.cu).
cudaError_t launch_chunked_simt(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *S_T, int B,
                                int H, int T, int dk, int dv, lr_dtype dt, lr_mode mode,
                                const Fuse &fz, cudaStream_t stream);

// Chunked forward on the tensor cores, bf16 (chunked_tc.cu).
cudaError_t launch_chunked_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *S_T, int B,
                              int H, int T, int dk, int dv, lr_mode mode, const Fuse &fz,
                              void *ws, cudaStream_t stream);
// Workspace bytes the tensor-core path needs (with the transformed q and k
// for the diagonal gate or when the flags ask for SiLU + L2).
size_t chunked_tc_workspace_bytes(int B, int H, int T, int dk, lr_mode mode, unsigned flags);

// mLSTM (mlstm.cu).  Workspace of the bf16 path, and the launchers.
size_t mlstm_workspace_bytes(int B, int H, int T, int dk);
cudaError_t launch_mlstm_chunked(const void *q, const void *k, const void *v, const float *fgate,
                                 const float *igate, const float *C0, const float *n0,
                                 const float *m0, void *h, float *C_T, float *n_T, float *m_T,
                                 int B, int H, int T, int dk, int dv, lr_dtype dt, void *ws,
                                 cudaStream_t stream);
cudaError_t launch_mlstm_step(const void *q, const void *k, const void *v, const float *fgate,
                              const float *igate, float *C, float *n, float *m, void *h, int N,
                              int H, int dk, int dv, lr_dtype dt, cudaStream_t stream);

// The bf16 mLSTM on the tensor cores (chunked_tc.cu).  phase 0: the per-block
// pass, records for the scan without delta (stage layout of lr_fwd_chunked)
// plus, per block, the fp32 aux values [row sums 64][m_t 64][g'_t 64][g_C]
// [Delta n dk] at `aux`; m_prev [B*H][nblk] is the stabiliser at every block
// start.  phase 1: the scan, h = numerator times the token's factor, which the
// caller has written into the records (mlstm_factor_slot), and C_T.
cudaError_t launch_mlstm_tc(const void *q, const void *k, const void *v, const float *fgate,
                            const float *igate, const float *m_prev, const float *C0, void *h,
                            float *C_T, float *aux, int phase, int B, int H, int T, int dk, int dv,
                            void *ws, cudaStream_t stream);
// The record slot of the mLSTM's per-token factors (see launch_mlstm_tc).
void mlstm_factor_slot(int dk, size_t *rec_bytes, size_t *offset);
size_t records_bytes_tc(int B, int H, int T, int dk);
// Whether launch_chunked_tc applies LR_FUSE_O_RMSNORM itself (in the scan) for
// this mode and these sizes; otherwise the caller runs the norm pass after it.
bool chunked_tc_applies_norm(lr_mode mode, int B, int H, int dv);

// Generalised delta rule of RWKV-7 (gen_delta.cu): the fp32 chunked kernel and
// the decode step (fp32 or bf16).
cudaError_t launch_gen_delta_chunked(const void *q, const void *kw, const void *v, const float *w,
                                     const float *kappa, const float *a, const float *S0, void *o,
                                     float *S_T, int B, int H, int T, int dk, int dv, lr_dtype dt,
                                     cudaStream_t stream);
cudaError_t launch_gen_delta_step(const void *q, const void *kw, const void *v, const float *w,
                                  const float *kappa, const float *a, float *S, void *o, int N,
                                  int H, int dk, int dv, lr_dtype dt, cudaStream_t stream);
// The bf16 path on the tensor cores (gen_delta_tc.cu): the per-block pass over
// 32-token blocks, then the scan of scan_tc.cuh; workspace of
// gen_delta_tc_workspace_bytes(...) bytes.
size_t gen_delta_tc_workspace_bytes(int B, int H, int T, int dk);
cudaError_t launch_gen_delta_tc(const void *q, const void *kw, const void *v, const float *w,
                                const float *kappa, const float *a, const float *S0, void *o,
                                float *S_T, int B, int H, int T, int dk, int dv, void *ws,
                                cudaStream_t stream);

// In-place RMSNorm of `rows` rows of dv channels (norm.cu).
cudaError_t launch_rmsnorm(void *o, const float *w, float eps, size_t rows, int dv, lr_dtype dt,
                           cudaStream_t stream);

// Return and clear the bounded-wait error word of the tensor-core kernels of
// chunked_tc.cu and of gen_delta_tc.cu (each has its own): 1 if set, 0 if
// clear, -1 if the device could not be read.
int read_and_clear_tc_error();
// The failure-detection test hook of the chunked forward's scan (0 = off).
cudaError_t set_scan_fault_tc(unsigned on);
int read_and_clear_gd_tc_error();

// Set the dynamic shared-memory limit of `fn` once per device.
cudaError_t ensure_smem_attr(const void *fn, int bytes, int slot);

}  // namespace lr
