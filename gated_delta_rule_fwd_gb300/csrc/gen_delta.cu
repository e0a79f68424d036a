// Generalised delta rule of RWKV-7 (page "Le architetture lineari: RetNet,
// RWKV, xLSTM", RWKV section; the extracted page lost the equation, read from
// its prose in the chapter's convention):
//
//     S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) + v_t kw_t^T,   o_t = S_t q_t,
//
// w_t a per-channel decay, kappa_t the removal key, a_t the per-channel rate,
// kw_t the write key.  Per value row r with s = S[r,:]: u = s . kappa,
// s <- s * w - u (a * kappa) + v_r kw.
//
// Chunked form (CUDA cores, fp32 arithmetic, 32-token blocks).  With u_t =
// S_{t-1} kappa_t and L the per-channel cumulative log decay of the block,
// unrolling the block gives a unit-lower-triangular system for U (the
// pseudo-values of the WY representation, first page, delta-rule section,
// here with per-channel decays):
//   (I + A) U = Kdec S0^T + Bk V,   A_ts = (b_s e^{L_{t-1} - L_s}) . kappa_t,
//                                   Bk_ts = (kw_s e^{L_{t-1} - L_s}) . kappa_t   (s < t)
//   O = (Q e^L) S0^T + Qk V - Qb U,  Qk_ts = (kw_s e^{L_t - L_s}) . q_t,
//                                    Qb_ts = (b_s e^{L_t - L_s}) . q_t           (s <= t)
//   S <- S0 Diag(e^{L_last}) + V^T (kw e^{L_last - L}) - U^T (b e^{L_last - L}),
// with b = a * kappa and Kdec_t = kappa_t e^{L_{t-1}}.  Every decay factor is
// e^{L_t - L_s} with t >= s, at most 1, so no rescaling is needed.  This is
// the fp32 path; bf16 runs on the tensor cores (gen_delta_tc.cu).
#include "lr_internal.cuh"

namespace lr {
namespace {

constexpr int C2 = 32;   // tokens per block
constexpr int DVS = 32;  // value channels per CTA
constexpr int NT = 512;

template <int DK>
struct GdSmem {
    static constexpr int KP = DK + 1, PP = C2 + 1, UP = DVS + 1;
    static constexpr int kQ = 0, kKw = kQ + C2 * KP, kKp = kKw + C2 * KP, kB = kKp + C2 * KP;
    static constexpr int kL = kB + C2 * KP, kS = kL + C2 * KP, kV = kS + DVS * KP;
    static constexpr int kU = kV + C2 * DVS, kQk = kU + C2 * UP, kQb = kQk + C2 * PP;
    static constexpr int kBk = kQb + C2 * PP, kA = kBk + C2 * PP;
    static constexpr int floats = kA + C2 * PP;
    static constexpr int bytes = floats * 4;
};

template <int DK, typename Tin>
__global__ void __launch_bounds__(NT)
chunk_gd_kernel(const Tin *__restrict__ q, const Tin *__restrict__ kw, const Tin *__restrict__ v,
                const float *__restrict__ w, const float *__restrict__ kappa,
                const float *__restrict__ ar, const float *__restrict__ S0, Tin *__restrict__ o,
                float *__restrict__ ST, int H, int T, int dv) {
    using L = GdSmem<DK>;
    constexpr int KP = L::KP, PP = L::PP, UP = L::UP;
    extern __shared__ float sm[];
    float *Qs = sm + L::kQ, *Kw = sm + L::kKw, *Kp = sm + L::kKp, *Bv = sm + L::kB;
    float *Ls = sm + L::kL, *Ss = sm + L::kS, *Vs = sm + L::kV, *Us = sm + L::kU;
    float *Qk = sm + L::kQk, *Qb = sm + L::kQb, *Bk = sm + L::kBk, *Am = sm + L::kA;
    const int tid = threadIdx.x;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;

    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        Ss[c * KP + j] = S0 ? S0[(bh * dv + c0 + c) * DK + j] : 0.f;
    }
    for (int t0 = 0; t0 < T; t0 += C2) {
        const int n = min(C2, T - t0);
        __syncthreads();
        // ---- stage (padded tokens: zero keys and queries, w = 1, a = 0)
        for (int idx = tid; idx < C2 * DK; idx += NT) {
            const int r = idx / DK, j = idx % DK;
            const bool ok = r < n;
            const size_t g = (bh * T + t0 + r) * DK + j;
            Qs[r * KP + j] = ok ? to_f(q[g]) : 0.f;
            Kw[r * KP + j] = ok ? to_f(kw[g]) : 0.f;
            const float kp = ok ? kappa[g] : 0.f;
            Kp[r * KP + j] = kp;
            Bv[r * KP + j] = ok ? ar[g] * kp : 0.f;
            Ls[r * KP + j] = ok ? logf(w[g]) : 0.f;
        }
        for (int idx = tid; idx < C2 * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            Vs[r * DVS + c] = r < n ? to_f(v[(bh * T + t0 + r) * dv + c0 + c]) : 0.f;
        }
        __syncthreads();
        if (tid < DK) {  // cumulative log decay per channel
            float acc = 0.f;
            for (int r = 0; r < C2; ++r) {
                acc += Ls[r * KP + tid];
                Ls[r * KP + tid] = acc;
            }
        }
        __syncthreads();
        // ---- the four decayed score matrices over the pairs s <= t (p enumerates
        //      the lower triangle row by row: t = the largest with t(t+1)/2 <= p)
        for (int idx = tid; idx < C2 * C2; idx += NT) {  // zero the upper triangle
            const int t = idx / C2, s = idx % C2;
            if (s > t) Qk[t * PP + s] = Qb[t * PP + s] = Bk[t * PP + s] = Am[t * PP + s] = 0.f;
        }
        for (int p = tid; p < C2 * (C2 + 1) / 2; p += NT) {
            int t = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
            if ((t + 1) * (t + 2) / 2 <= p) ++t;
            if (t * (t + 1) / 2 > p) --t;
            const int s = p - t * (t + 1) / 2;
            float qk = 0.f, qb = 0.f, bk = 0.f, aa = 0.f;
            {
                for (int j = 0; j < DK; ++j) {
                    const float Lt = Ls[t * KP + j], Ls_ = Ls[s * KP + j];
                    const float d1 = __expf(Lt - Ls_);
                    const float kwj = Kw[s * KP + j], bj = Bv[s * KP + j];
                    qk += Qs[t * KP + j] * kwj * d1;
                    qb += Qs[t * KP + j] * bj * d1;
                    if (s < t) {
                        const float d0 = __expf(Ls[(t - 1) * KP + j] - Ls_);
                        bk += Kp[t * KP + j] * kwj * d0;
                        aa += Kp[t * KP + j] * bj * d0;
                    }
                }
            }
            Qk[t * PP + s] = qk;
            Qb[t * PP + s] = qb;
            Bk[t * PP + s] = bk;
            Am[t * PP + s] = aa;
        }
        __syncthreads();
        // ---- Q e^{L_t} and Kdec = kappa e^{L_{t-1}} in place (the scores are done)
        for (int idx = tid; idx < C2 * DK; idx += NT) {
            const int t = idx / DK, j = idx % DK;
            Qs[t * KP + j] *= __expf(Ls[t * KP + j]);
            Kp[t * KP + j] *= t > 0 ? __expf(Ls[(t - 1) * KP + j]) : 1.f;
        }
        __syncthreads();
        // ---- right-hand side Kdec S0^T + Bk V
        for (int idx = tid; idx < C2 * DVS; idx += NT) {
            const int t = idx / DVS, c = idx % DVS;
            float acc = 0.f;
            for (int j = 0; j < DK; ++j) acc += Kp[t * KP + j] * Ss[c * KP + j];
            for (int s = 0; s < t; ++s) acc += Bk[t * PP + s] * Vs[s * DVS + c];
            Us[t * UP + c] = acc;
        }
        __syncthreads();
        // ---- forward substitution (I + A) U = rhs: one thread per value channel
        if (tid < DVS) {
            for (int t = 1; t < C2; ++t) {
                float acc = Us[t * UP + tid];
                for (int s = 0; s < t; ++s) acc -= Am[t * PP + s] * Us[s * UP + tid];
                Us[t * UP + tid] = acc;
            }
        }
        __syncthreads();
        // ---- outputs O = (Q e^L) S0^T + Qk V - Qb U
        for (int idx = tid; idx < C2 * DVS; idx += NT) {
            const int t = idx / DVS, c = idx % DVS;
            if (t >= n) continue;
            float acc = 0.f;
            for (int j = 0; j < DK; ++j) acc += Qs[t * KP + j] * Ss[c * KP + j];
            for (int s = 0; s <= t; ++s)
                acc += Qk[t * PP + s] * Vs[s * DVS + c] - Qb[t * PP + s] * Us[s * UP + c];
            o[(bh * T + t0 + t) * dv + c0 + c] = from_f<Tin>(acc);
        }
        __syncthreads();
        // ---- state S <- S0 Diag(e^{L_last}) + V^T (kw e^{L_last - L}) - U^T (b e^{L_last - L})
        for (int idx = tid; idx < C2 * DK; idx += NT) {
            const int r = idx / DK, j = idx % DK;
            const float f = __expf(Ls[(C2 - 1) * KP + j] - Ls[r * KP + j]);
            Kw[r * KP + j] *= f;
            Bv[r * KP + j] *= f;
        }
        __syncthreads();
        for (int idx = tid; idx < DVS * DK; idx += NT) {
            const int c = idx / DK, j = idx % DK;
            float acc = 0.f;
            for (int s = 0; s < C2; ++s)
                acc += Vs[s * DVS + c] * Kw[s * KP + j] - Us[s * UP + c] * Bv[s * KP + j];
            Ss[c * KP + j] = __expf(Ls[(C2 - 1) * KP + j]) * Ss[c * KP + j] + acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        ST[(bh * dv + c0 + c) * DK + j] = Ss[c * KP + j];
    }
}

// ----------------------------------------------------------------- decode
constexpr int kStepThreads = 128, kLanesPerRow = 8, kRowsPerPass = 16;

__device__ __forceinline__ float sum8(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}
__device__ __forceinline__ float4 ld4f(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float dot4(float4 x, float4 y) {
    return x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kStepThreads)
gd_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ kw, const Tin *__restrict__ v,
               const float *__restrict__ w, const float *__restrict__ kappa,
               const float *__restrict__ ar, float *__restrict__ S, Tin *__restrict__ o, int dv) {
    constexpr int NV = DK / (4 * kLanesPerRow);
    const int head = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, rg = lane >> 3;
    float4 qr[NV], kr[NV], wr[NV], cr[NV], br[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int col = 4 * (kLanesPerRow * u + sub);
        const size_t g = (size_t)head * DK + col;
        qr[u] = load4(q + g);
        kr[u] = load4(kw + g);
        wr[u] = ld4f(w + g);
        cr[u] = ld4f(kappa + g);
        const float4 a4 = ld4f(ar + g);
        br[u] = make_float4(a4.x * cr[u].x, a4.y * cr[u].y, a4.z * cr[u].z, a4.w * cr[u].w);
    }
    float *Sh = S + (size_t)head * dv * DK;
    for (int p = 0; p < dv / kRowsPerPass; ++p) {
        const int r = p * kRowsPerPass + warp * 4 + rg;
        float4 s[NV];
        float uu = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            s[u] = ld4f(Sh + (size_t)r * DK + 4 * (kLanesPerRow * u + sub));
            uu += dot4(s[u], cr[u]);
        }
        uu = sum8(uu);
        const float vr = to_f(v[(size_t)head * dv + r]);
        float oo = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            float4 t;
            t.x = s[u].x * wr[u].x - uu * br[u].x + vr * kr[u].x;
            t.y = s[u].y * wr[u].y - uu * br[u].y + vr * kr[u].y;
            t.z = s[u].z * wr[u].z - uu * br[u].z + vr * kr[u].z;
            t.w = s[u].w * wr[u].w - uu * br[u].w + vr * kr[u].w;
            *reinterpret_cast<float4 *>(Sh + (size_t)r * DK + 4 * (kLanesPerRow * u + sub)) = t;
            oo += dot4(t, qr[u]);
        }
        oo = sum8(oo);
        if (sub == 0) o[(size_t)head * dv + r] = from_f<Tin>(oo);
    }
}

template <typename Tin>
cudaError_t chunked_typed(const void *q, const void *kw, const void *v, const float *w,
                          const float *kappa, const float *a, const float *S0, void *o, float *S_T,
                          int B, int H, int T, int dk, int dv, cudaStream_t stream, int slot) {
    auto go = [&](auto kern, int bytes) {
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), bytes, slot);
        if (e != cudaSuccess) return e;
        kern<<<dim3(dv / DVS, H, B), NT, bytes, stream>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(kw), static_cast<const Tin *>(v),
            w, kappa, a, S0, static_cast<Tin *>(o), S_T, H, T, dv);
        return cudaGetLastError();
    };
    switch (dk) {
    case 32: return go(chunk_gd_kernel<32, Tin>, GdSmem<32>::bytes);
    case 64: return go(chunk_gd_kernel<64, Tin>, GdSmem<64>::bytes);
    default: return go(chunk_gd_kernel<128, Tin>, GdSmem<128>::bytes);
    }
}

}  // namespace

// Attribute slots 148..150 belong to this file (the fp32 chunked kernel).
cudaError_t launch_gen_delta_chunked(const void *q, const void *kw, const void *v, const float *w,
                                     const float *kappa, const float *a, const float *S0, void *o,
                                     float *S_T, int B, int H, int T, int dk, int dv, lr_dtype dt,
                                     cudaStream_t stream) {
    if (dt != LR_DT_F32) return cudaErrorInvalidValue;  // bf16 runs on the tensor cores
    const int s = 148 + (dk == 32 ? 0 : dk == 64 ? 1 : 2);
    return chunked_typed<float>(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dk, dv, stream, s);
}

cudaError_t launch_gen_delta_step(const void *q, const void *kw, const void *v, const float *w,
                                  const float *kappa, const float *a, float *S, void *o, int N,
                                  int H, int dk, int dv, lr_dtype dt, cudaStream_t stream) {
    const int NH = N * H;
    auto go = [&](auto kern, auto tin) {
        using Tin = decltype(tin);
        kern<<<NH, kStepThreads, 0, stream>>>(static_cast<const Tin *>(q),
                                              static_cast<const Tin *>(kw),
                                              static_cast<const Tin *>(v), w, kappa, a, S,
                                              static_cast<Tin *>(o), dv);
        return cudaGetLastError();
    };
    if (dt == LR_DT_F32) {
        switch (dk) {
        case 32: return go(gd_step_kernel<32, float>, float{});
        case 64: return go(gd_step_kernel<64, float>, float{});
        default: return go(gd_step_kernel<128, float>, float{});
        }
    }
    using bf = __nv_bfloat16;
    switch (dk) {
    case 32: return go(gd_step_kernel<32, bf>, bf{});
    case 64: return go(gd_step_kernel<64, bf>, bf{});
    default: return go(gd_step_kernel<128, bf>, bf{});
    }
}

}  // namespace lr
