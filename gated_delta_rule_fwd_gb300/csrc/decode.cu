// Decode step: one token for N x H independent states, streamed from HBM.
//
// Page "Le architetture lineari: RetNet, RWKV, xLSTM", section "RetNet: la
// retention e le sue tre forme", recurrent form: a fixed-size memory updated
// once per token at O(d^2) cost.  Each value channel r (a row of S) evolves
// on its own given k, alpha and beta:
//
//     u_r = beta (v_r - a S[r,:].k)  (delta rows)   or   v_r  (others)
//     S[r,:] <- a S[r,:] + u_r k ;   o_r = a S[r,:].q + u_r (k.q)
//
// The kernel is bound by HBM bandwidth (fp32 state read once and written
// once, 0.75 flop per byte).  Mapping: one CTA of 128 threads per (n, h); 8
// lanes share a row, each lane owning DK/32 float4 columns interleaved so
// that the 8 lanes of a row read 128 contiguous bytes per instruction; a
// warp covers 4 rows per pass, the CTA 16 rows.  Each thread keeps UNROLL
// rows of loads in flight.  Row dot products reduce over the 8 lanes with
// three xor shuffles.
#include "lr_internal.cuh"

namespace lr {
namespace {

constexpr int kStepThreads = 128;
constexpr int kLanesPerRow = 8;
constexpr int kRowsPerPass = kStepThreads / kLanesPerRow;  // 16

__device__ __forceinline__ float4 ld_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}

__device__ __forceinline__ float sum8(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

template <int DK, typename Tin, bool ALPHA, bool DELTA, int UNROLL>
__global__ void __launch_bounds__(kStepThreads)
step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
            const float *__restrict__ alpha, const float *__restrict__ beta,
            float *__restrict__ S, Tin *__restrict__ o, int dv) {
    constexpr int NV = DK / (4 * kLanesPerRow);  // float4 per lane per row
    static_assert(NV >= 1 && NV * 4 * kLanesPerRow == DK, "DK must be 32, 64 or 128");

    const int head = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane & (kLanesPerRow - 1);
    const int rg = lane / kLanesPerRow;

    const Tin *qh = q + (size_t)head * DK;
    const Tin *kh = k + (size_t)head * DK;
    const Tin *vh = v + (size_t)head * dv;
    float *Sh = S + (size_t)head * dv * DK;
    Tin *oh = o + (size_t)head * dv;

    float4 kr[NV], qr[NV];
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
        const int col = 4 * (kLanesPerRow * m + sub);
        kr[m] = load4(kh + col);
        qr[m] = load4(qh + col);
        kq += kr[m].x * qr[m].x + kr[m].y * qr[m].y + kr[m].z * qr[m].z + kr[m].w * qr[m].w;
    }
    kq = sum8(kq);
    const float a = ALPHA ? alpha[head] : 1.f;
    const float b = DELTA ? beta[head] : 1.f;

    const int passes = dv / kRowsPerPass;
    for (int p0 = 0; p0 < passes; p0 += UNROLL) {
        float4 s[UNROLL][NV];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = (p0 + u) * kRowsPerPass + warp * 4 + rg;
#pragma unroll
            for (int m = 0; m < NV; ++m)
                s[u][m] = ld_stream(Sh + (size_t)r * DK + 4 * (kLanesPerRow * m + sub));
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = (p0 + u) * kRowsPerPass + warp * 4 + rg;
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                sk += s[u][m].x * kr[m].x + s[u][m].y * kr[m].y + s[u][m].z * kr[m].z +
                      s[u][m].w * kr[m].w;
                sq += s[u][m].x * qr[m].x + s[u][m].y * qr[m].y + s[u][m].z * qr[m].z +
                      s[u][m].w * qr[m].w;
            }
            sk = sum8(sk);
            sq = sum8(sq);
            const float vr = to_f(vh[r]);
            const float ur = DELTA ? b * (vr - a * sk) : vr;
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                float4 t;
                t.x = a * s[u][m].x + ur * kr[m].x;
                t.y = a * s[u][m].y + ur * kr[m].y;
                t.z = a * s[u][m].z + ur * kr[m].z;
                t.w = a * s[u][m].w + ur * kr[m].w;
                st_stream(Sh + (size_t)r * DK + 4 * (kLanesPerRow * m + sub), t);
            }
            if (sub == 0) oh[r] = from_f<Tin>(a * sq + ur * kq);
        }
    }
}

template <int DK, typename Tin, bool ALPHA, bool DELTA>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, float *S, void *o, int NH, int dv,
                         cudaStream_t stream) {
    // dv in {32, 64, 128}: 2, 4 or 8 passes of 16 rows; UNROLL 2 divides all.
    step_kernel<DK, Tin, ALPHA, DELTA, 2><<<NH, kStepThreads, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, S, static_cast<Tin *>(o), dv);
    return cudaGetLastError();
}

template <int DK, typename Tin>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int NH, int dv, lr_mode mode,
                        cudaStream_t stream) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, Tin, false, false>(q, k, v, alpha, beta, S, o, NH, dv, stream);
    case LR_MODE_DECAY:
        return launch_typed<DK, Tin, true, false>(q, k, v, alpha, beta, S, o, NH, dv, stream);
    case LR_MODE_DELTA:
        return launch_typed<DK, Tin, false, true>(q, k, v, alpha, beta, S, o, NH, dv, stream);
    default:
        return launch_typed<DK, Tin, true, true>(q, k, v, alpha, beta, S, o, NH, dv, stream);
    }
}

template <typename Tin>
cudaError_t launch_dk(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, float *S, void *o, int NH, int dk, int dv,
                      lr_mode mode, cudaStream_t stream) {
    switch (dk) {
    case 32: return launch_mode<32, Tin>(q, k, v, alpha, beta, S, o, NH, dv, mode, stream);
    case 64: return launch_mode<64, Tin>(q, k, v, alpha, beta, S, o, NH, dv, mode, stream);
    default: return launch_mode<128, Tin>(q, k, v, alpha, beta, S, o, NH, dv, mode, stream);
    }
}

}  // namespace

cudaError_t launch_step(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                        lr_dtype dt, lr_mode mode, cudaStream_t stream) {
    const int NH = N * H;
    if (dt == LR_DT_F32)
        return launch_dk<float>(q, k, v, alpha, beta, S, o, NH, dk, dv, mode, stream);
    return launch_dk<__nv_bfloat16>(q, k, v, alpha, beta, S, o, NH, dk, dv, mode, stream);
}

}  // namespace lr
