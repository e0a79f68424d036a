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
//
// With the lr_fuse maps (page "Scrivere meglio nella memoria: gate e delta
// rule"): SiLU of q and k is taken once per element for the CTA, shared
// through shared memory, and the two L2 norms are one CTA-wide sum; the gates
// are mapped on load, and with the output RMSNorm the d_v outputs of the head
// are kept in shared memory, normalised together and stored once.
//
// Diagonal gate (GLA row, same page, gates section): alpha is a vector over the
// key channels, so each lane loads the gates of its own columns and the row
// update is S[r,:] <- alpha * S[r,:] + v_r k (element-wise), o_r = S_new[r,:] . q.
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

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
__device__ __forceinline__ float4 scale4(float4 a, float s) {
    return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}

template <int DK, typename Tin, bool ALPHA, bool DELTA, bool DIAG, int UNROLL>
__global__ void __launch_bounds__(kStepThreads)
step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
            const float *__restrict__ alpha, const float *__restrict__ beta,
            float *__restrict__ S, Tin *__restrict__ o, int H, int dv, const Fuse fz) {
    __shared__ float o_sh[128];  // the head's outputs, with the output RMSNorm
    __shared__ float ss_sh[kStepThreads / 32];
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

    const unsigned fl = fz.flags;
    float4 kr[NV], qr[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) {
        const int col = 4 * (kLanesPerRow * m + sub);
        kr[m] = load4(kh + col);
        qr[m] = load4(qh + col);
    }
    if (fl & LR_FUSE_QK_SILU_L2) {
        // Every row group holds the same columns, so SiLU is taken once per
        // element for the CTA (thread i: element i of k and of q) and shared;
        // the two squared norms are one CTA-wide sum.
        __shared__ __align__(16) float qk_sh[2 * DK];
        __shared__ float nn_sh[2][kStepThreads / 32];
        float kk = 0.f, qq = 0.f;
        for (int i = threadIdx.x; i < DK; i += kStepThreads) {
            const float ks = silu_f(to_f(kh[i])), qs = silu_f(to_f(qh[i]));
            qk_sh[i] = ks;
            qk_sh[DK + i] = qs;
            kk += ks * ks;
            qq += qs * qs;
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, d);
            qq += __shfl_xor_sync(0xffffffffu, qq, d);
        }
        if (lane == 0) {
            nn_sh[0][warp] = kk;
            nn_sh[1][warp] = qq;
        }
        __syncthreads();
        kk = 0.f;
        qq = 0.f;
#pragma unroll
        for (int w = 0; w < kStepThreads / 32; ++w) {
            kk += nn_sh[0][w];
            qq += nn_sh[1][w];
        }
        const float ik = inv_l2(kk), iq = inv_l2(qq);
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int col = 4 * (kLanesPerRow * m + sub);
            kr[m] = scale4(*reinterpret_cast<const float4 *>(qk_sh + col), ik);
            qr[m] = scale4(*reinterpret_cast<const float4 *>(qk_sh + DK + col), iq);
        }
    }
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) kq += dot4(kr[m], qr[m]);
    kq = sum8(kq);
    const float ac = (fl & kScaledAlphaMaps) ? fz.ascale[head % H] : 0.f;
    const float a = (ALPHA && !DIAG) ? gate(fl, alpha[head], ac) : 1.f;
    float4 ar[NV];  // the diagonal gate of this lane's columns
    if (DIAG) {
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            float4 g = *reinterpret_cast<const float4 *>(alpha + (size_t)head * DK +
                                                        4 * (kLanesPerRow * m + sub));
            if (fl & kAlphaMaps)
                g = make_float4(gate(fl, g.x, ac), gate(fl, g.y, ac), gate(fl, g.z, ac),
                                gate(fl, g.w, ac));
            ar[m] = g;
        }
    }
    const float b = DELTA ? write_strength(fl, beta[head]) : 1.f;
    const bool norm = (fl & LR_FUSE_O_RMSNORM) != 0;
    float oss = 0.f;  // sum of squares of the outputs this lane produced

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
        if (DIAG) {  // decay first: the row update and read-out use alpha * s
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
#pragma unroll
                for (int m = 0; m < NV; ++m)
                    s[u][m] = make_float4(s[u][m].x * ar[m].x, s[u][m].y * ar[m].y,
                                          s[u][m].z * ar[m].z, s[u][m].w * ar[m].w);
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
            if (sub == 0) {
                const float orow = a * sq + ur * kq;
                if (norm) {
                    o_sh[r] = orow;
                    oss += orow * orow;
                } else {
                    oh[r] = from_f<Tin>(orow);
                }
            }
        }
    }
    if (norm) {  // one barrier: per-warp partial sums, then every thread finishes the sum
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) oss += __shfl_xor_sync(0xffffffffu, oss, d);
        if (lane == 0) ss_sh[warp] = oss;
        __syncthreads();
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kStepThreads / 32; ++w) ss += ss_sh[w];
        const float inv = rsqrtf(ss / (float)dv + fz.norm_eps);
        const int r = threadIdx.x;
        if (r < dv) oh[r] = from_f<Tin>(o_sh[r] * inv * (fz.norm_w ? fz.norm_w[r] : 1.f));
    }
}

template <int DK, typename Tin, bool ALPHA, bool DELTA, bool DIAG = false>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, float *S, void *o, int NH, int H, int dv,
                         const Fuse &fz, cudaStream_t stream) {
    // dv in {32, 64, 128}: 2, 4 or 8 passes of 16 rows; UNROLL 2 divides all.
    step_kernel<DK, Tin, ALPHA, DELTA, DIAG, 2><<<NH, kStepThreads, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, S, static_cast<Tin *>(o), H, dv, fz);
    return cudaGetLastError();
}

template <int DK, typename Tin>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int NH, int H, int dv,
                        lr_mode mode, const Fuse &fz, cudaStream_t stream) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, Tin, false, false>(q, k, v, alpha, beta, S, o, NH, H, dv, fz, stream);
    case LR_MODE_DECAY:
        return launch_typed<DK, Tin, true, false>(q, k, v, alpha, beta, S, o, NH, H, dv, fz, stream);
    case LR_MODE_DELTA:
        return launch_typed<DK, Tin, false, true>(q, k, v, alpha, beta, S, o, NH, H, dv, fz, stream);
    case LR_MODE_DIAG_DECAY:
        return launch_typed<DK, Tin, true, false, true>(q, k, v, alpha, beta, S, o, NH, H, dv, fz,
                                                        stream);
    default:
        return launch_typed<DK, Tin, true, true>(q, k, v, alpha, beta, S, o, NH, H, dv, fz, stream);
    }
}

template <typename Tin>
cudaError_t launch_dk(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, float *S, void *o, int NH, int H, int dk, int dv,
                      lr_mode mode, const Fuse &fz, cudaStream_t stream) {
    switch (dk) {
    case 32: return launch_mode<32, Tin>(q, k, v, alpha, beta, S, o, NH, H, dv, mode, fz, stream);
    case 64: return launch_mode<64, Tin>(q, k, v, alpha, beta, S, o, NH, H, dv, mode, fz, stream);
    default: return launch_mode<128, Tin>(q, k, v, alpha, beta, S, o, NH, H, dv, mode, fz, stream);
    }
}

}  // namespace

cudaError_t launch_step(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                        lr_dtype dt, lr_mode mode, const Fuse &fz, cudaStream_t stream) {
    const int NH = N * H;
    if (dt == LR_DT_F32)
        return launch_dk<float>(q, k, v, alpha, beta, S, o, NH, H, dk, dv, mode, fz, stream);
    return launch_dk<__nv_bfloat16>(q, k, v, alpha, beta, S, o, NH, H, dk, dv, mode, fz, stream);
}

}  // namespace lr
