// mLSTM memory (page "Le architetture lineari: RetNet, RWKV, xLSTM", xLSTM
// section, the matrix-memory cell), stabilised as the page gives it:
//
//   m_t = max(log f_t + m_{t-1}, igate_t),
//   C~_t = e^{log f_t + m_{t-1} - m_t} C~_{t-1} + e^{igate_t - m_t} v_t k_t^T   (n~ likewise with k_t),
//   h_t = C~_t q_t / max(|n~_t^T q_t|, e^{-m_t}).
//
// The stabiliser depends on the gates only, so the bf16 path computes it for
// every block start first (mlstm_stab_kernel), then runs the per-block pass
// (chunked_tc.cu), the normaliser n~ at every block start
// (mlstm_nscan_kernel) and every token's factor 1 / max(|denominator|,
// e^{-m_t}) (mlstm_den_kernel), and last the scan without delta, which
// multiplies each token's numerator by its factor before the one rounding to
// bf16.  The fp32 path and the decode step do it all in one kernel each.
#include <math.h>

#include <type_traits>

#include "lr_internal.cuh"

namespace lr {
namespace {

constexpr int C = 64;
constexpr int DVS = 32;
// aux record of a block (written by the per-block pass): row sums, m_t, g'_t,
// g_C, Delta n -- the offsets used there
constexpr int kMlstmAux = 384, kAuxRs = 0, kAuxM = 64, kAuxG = 128, kAuxGC = 192, kAuxDn = 256;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct MlstmWs {
    size_t recs, mprev, aux, nst, total;
};
MlstmWs mlstm_ws(int B, int H, int T, int dk) {
    const size_t nblk = (size_t)((T + C - 1) / C), bh = (size_t)B * H;
    MlstmWs w;
    w.recs = 0;
    w.mprev = align256(records_bytes_tc(B, H, T, dk));
    w.aux = align256(w.mprev + bh * nblk * 4);
    w.nst = align256(w.aux + bh * nblk * kMlstmAux * 4);
    w.total = w.nst + bh * nblk * (size_t)dk * 4;
    return w;
}

// --------------------------------------------------------------- stabiliser
// One CTA per (b, h).  Each thread summarises blocks (F_C = sum of log f,
// X = max_s (F_C - F_s + igate_s)); thread 0 then walks them in order:
// m_end = max(F_C + m_start, X).  Writes m at every block start and the final m.
constexpr int kStabThreads = 256;

__global__ void __launch_bounds__(kStabThreads)
mlstm_stab_kernel(const float *__restrict__ fgate, const float *__restrict__ igate,
                  const float *__restrict__ m0, float *__restrict__ m_prev,
                  float *__restrict__ mT, int T, int nblk) {
    __shared__ float sF[kStabThreads], sX[kStabThreads];
    __shared__ float carry;
    const size_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) carry = m0 ? m0[bh] : -INFINITY;
    for (int g0 = 0; g0 < nblk; g0 += kStabThreads) {
        const int j = g0 + tid;
        float F = 0.f, X = -INFINITY;
        if (j < nblk) {
            const int t0 = j * C, n = min(C, T - t0);
            for (int s = 0; s < n; ++s) {
                F += __logf(fgate[bh * T + t0 + s]);
                X = fmaxf(X, igate[bh * T + t0 + s] - F);
            }
            X += F;
        }
        sF[tid] = F;
        sX[tid] = X;
        __syncthreads();
        if (tid == 0) {
            float m = carry;
            const int cnt = min(kStabThreads, nblk - g0);
            for (int i = 0; i < cnt; ++i) {
                m_prev[bh * nblk + g0 + i] = m;
                m = fmaxf(sF[i] + m, sX[i]);
            }
            carry = m;
        }
        __syncthreads();
    }
    if (tid == 0) mT[bh] = carry;
}

// ---------------------------------------------------------------- normaliser
// One warp per (b, h): n~ at every block start, n~ <- g_C n~ + Delta n.
template <int DK>
__global__ void __launch_bounds__(32)
mlstm_nscan_kernel(const float *__restrict__ aux, const float *__restrict__ n0,
                   float *__restrict__ nst, float *__restrict__ nT, int nblk) {
    constexpr int E = DK / 32;
    const size_t bh = blockIdx.x;
    const int lane = threadIdx.x;
    float nv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) nv[e] = n0 ? n0[bh * DK + lane + 32 * e] : 0.f;
#pragma unroll 4
    for (int j = 0; j < nblk; ++j) {
        const float *a = aux + (bh * nblk + j) * kMlstmAux;
        const float gc = a[kAuxGC];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            nst[(bh * nblk + j) * DK + lane + 32 * e] = nv[e];
            nv[e] = gc * nv[e] + a[kAuxDn + lane + 32 * e];
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) nT[bh * DK + lane + 32 * e] = nv[e];
}

// One CTA of 4 warps per (block, b, h); a warp takes four tokens at a time:
// den = g'_t (n~ . q_t) + row sum, and the token's factor
// 1 / max(|den|, e^{-m_t}), written into the vector of the stage record that
// the scan reads with the block's output rows (record blk + 1, float slot
// `slot` bytes in, records `rec_bytes` apart).  Each lane holds d_k / 32 consecutive
// channels of q (one 2-, 4- or 8-byte access per row); the four tokens' loads
// are independent.
template <int N> struct Lanes;
template <> struct Lanes<1> { using T = unsigned short; };
template <> struct Lanes<2> { using T = unsigned int; };
template <> struct Lanes<4> { using T = uint2; };

__device__ __forceinline__ void unpack(unsigned short w, float (&x)[1]) {
    x[0] = __uint_as_float((uint32_t)w << 16);
}
__device__ __forceinline__ void unpack(unsigned int w, float (&x)[2]) {
    x[0] = __uint_as_float(w << 16);
    x[1] = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void unpack(uint2 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xffff0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xffff0000u);
}

template <int DK>
__global__ void __launch_bounds__(128)
mlstm_den_kernel(const __nv_bfloat16 *__restrict__ q, const float *__restrict__ aux,
                 const float *__restrict__ nst, uint8_t *__restrict__ recs, size_t rec_bytes,
                 size_t slot, int H, int T, int nblk) {
    constexpr int EK = DK / 32, U = 4;
    using LK = typename Lanes<EK>::T;
    const int blk = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *a = aux + (bh * nblk + blk) * kMlstmAux;
    float nv[EK];
#pragma unroll
    for (int e = 0; e < EK; ++e) nv[e] = nst[(bh * nblk + blk) * DK + EK * lane + e];
    const int t0 = blk * C, n = min(C, T - t0);
    float *fac = reinterpret_cast<float *>(recs + (bh * (nblk + 1) + blk + 1) * rec_bytes + slot);
    const LK *qr = reinterpret_cast<const LK *>(q);
    for (int r0 = warp * U; r0 < n; r0 += 4 * U) {
        LK qw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) qw[u] = qr[(bh * T + t0 + min(r0 + u, n - 1)) * 32 + lane];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u;
            float qf[EK];
            unpack(qw[u], qf);
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < EK; ++e) d += nv[e] * qf[e];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (r < n && lane == 0) {
                const float den = a[kAuxG + r] * d + a[kAuxRs + r];
                fac[r] = 1.f / fmaxf(fabsf(den), __expf(-a[kAuxM + r]));
            }
        }
    }
}

// ---------------------------------------------------------------- fp32 path
// One CTA of 256 threads per (32 value channels, b, h), the blocks in order;
// each CTA keeps its own copy of n~ and m.
constexpr int NT = 256;

template <int DK>
struct MlstmSmem {
    static constexpr int KP = DK + 1, PP = C + 1;
    static constexpr int kK = 0, kQ = kK + C * KP, kS = kQ + C * KP, kV = kS + DVS * KP;
    static constexpr int kP = kV + C * DVS, kVec = kP + C * PP;
    // vectors: At, Bs, g', kd, m_t, den [C each], n~ [DK], scalars
    static constexpr int kAt = kVec, kBs = kAt + C, kG = kBs + C, kKd = kG + C, kM = kKd + C;
    static constexpr int kDen = kM + C, kN = kDen + C, kSc = kN + DK;
    static constexpr int floats = kSc + 8;
    static constexpr int bytes = floats * 4;
};

template <int DK, typename Tin>
__global__ void __launch_bounds__(NT)
chunk_simt_mlstm_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, const float *__restrict__ fgate,
                        const float *__restrict__ igate, const float *__restrict__ C0,
                        const float *__restrict__ n0, const float *__restrict__ m0,
                        Tin *__restrict__ h, float *__restrict__ CT, float *__restrict__ nT,
                        float *__restrict__ mT, int H, int T, int dv) {
    using L = MlstmSmem<DK>;
    constexpr int KP = L::KP, PP = L::PP;
    extern __shared__ float sm[];
    float *Ks = sm + L::kK, *Qs = sm + L::kQ, *Ss = sm + L::kS, *Vs = sm + L::kV, *Ps = sm + L::kP;
    float *At = sm + L::kAt, *Bs = sm + L::kBs, *Gp = sm + L::kG, *Kd = sm + L::kKd;
    float *Mt = sm + L::kM, *Den = sm + L::kDen, *Nv = sm + L::kN, *Sc = sm + L::kSc;
    const int tid = threadIdx.x;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;

    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        Ss[c * KP + j] = C0 ? C0[(bh * dv + c0 + c) * DK + j] : 0.f;
    }
    for (int j = tid; j < DK; j += NT) Nv[j] = n0 ? n0[bh * DK + j] : 0.f;
    if (tid == 0) Sc[0] = m0 ? m0[bh] : -INFINITY;  // m at the block start

    for (int t0 = 0; t0 < T; t0 += C) {
        const int n = min(C, T - t0);
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, j = idx % DK;
            const bool ok = r < n;
            const size_t g = (bh * T + t0 + r) * DK + j;
            Ks[r * KP + j] = ok ? to_f(k[g]) : 0.f;
            Qs[r * KP + j] = ok ? to_f(q[g]) : 0.f;
        }
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            Vs[r * DVS + c] = r < n ? to_f(v[(bh * T + t0 + r) * dv + c0 + c]) : 0.f;
        }
        if (tid == 0) {  // gates of the block, in order (64 steps)
            const float mp = Sc[0];
            float F = 0.f, mx = -INFINITY;
            for (int r = 0; r < C; ++r) {
                const bool ok = r < n;
                F += ok ? logf(fgate[bh * T + t0 + r]) : 0.f;
                const float x = ok ? igate[bh * T + t0 + r] - F : -INFINITY;
                mx = fmaxf(mx, x);
                const float mt = fmaxf(F + mp, F + mx);
                At[r] = F - mt;
                Bs[r] = x;
                Gp[r] = expf(F + mp - mt);
                Mt[r] = mt;
            }
            const float mC = Mt[C - 1];
            for (int r = 0; r < C; ++r) Kd[r] = expf(F - mC + Bs[r]);
            Sc[1] = expf(F + mp - mC);  // g_C
            Sc[2] = mC;
        }
        __syncthreads();

        // ---- scores P_ri = (q_r . k_i) e^{F_r - F_i + igate_i - m_r}, i <= r
        for (int idx = tid; idx < C * C; idx += NT) {
            const int r = idx / C, i = idx % C;
            float p = 0.f;
            if (i <= r) {
                float d = 0.f;
#pragma unroll 8
                for (int j = 0; j < DK; ++j) d += Qs[r * KP + j] * Ks[i * KP + j];
                p = d * expf(At[r] + Bs[i]);
            }
            Ps[r * PP + i] = p;
        }
        __syncthreads();
        // ---- denominators g'_r (n~ . q_r) + sum_i P_ri
        if (tid < C) {
            float d = 0.f, rs = 0.f;
            for (int j = 0; j < DK; ++j) d += Nv[j] * Qs[tid * KP + j];
            for (int i = 0; i <= tid; ++i) rs += Ps[tid * PP + i];
            Den[tid] = Gp[tid] * d + rs;
        }
        __syncthreads();
        // ---- h = (g' Q C~^T + P V) / max(|den|, e^{-m})
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            if (r >= n) continue;
            float qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) qs += Qs[r * KP + j] * Ss[c * KP + j];
            float pv = 0.f;
            for (int i = 0; i <= r; ++i) pv += Ps[r * PP + i] * Vs[i * DVS + c];
            const float num = Gp[r] * qs + pv;
            h[(bh * T + t0 + r) * dv + c0 + c] =
                from_f<Tin>(num / fmaxf(fabsf(Den[r]), expf(-Mt[r])));
        }
        __syncthreads();
        // ---- carry C~ <- g_C C~ + V^T diag(kd) K, n~ <- g_C n~ + K^T kd
        const float gC = Sc[1];
        for (int idx = tid; idx < DVS * DK; idx += NT) {
            const int c = idx / DK, j = idx % DK;
            float acc = 0.f;
#pragma unroll 8
            for (int i = 0; i < C; ++i) acc += Vs[i * DVS + c] * Kd[i] * Ks[i * KP + j];
            Ss[c * KP + j] = gC * Ss[c * KP + j] + acc;
        }
        for (int j = tid; j < DK; j += NT) {
            float acc = 0.f;
            for (int i = 0; i < C; ++i) acc += Kd[i] * Ks[i * KP + j];
            Nv[j] = gC * Nv[j] + acc;
        }
        if (tid == 0) Sc[0] = Sc[2];
    }
    __syncthreads();
    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        CT[(bh * dv + c0 + c) * DK + j] = Ss[c * KP + j];
    }
    if (blockIdx.x == 0) {
        for (int j = tid; j < DK; j += NT) nT[bh * DK + j] = Nv[j];
        if (tid == 0) mT[bh] = Sc[0];
    }
}

// -------------------------------------------------------------------- decode
// One CTA of 128 threads per (n, h), 8 lanes per state row (as the decode step
// of the other modes): C~ rows a C~ + b v_r k, n~ the same with k, and
// h_r = (C~ q)_r / max(|n~ . q|, e^{-m'}).
constexpr int kStepThreads = 128, kLanesPerRow = 8, kRowsPerPass = 16;

__device__ __forceinline__ float sum8(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kStepThreads)
mlstm_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                  const float *__restrict__ fgate, const float *__restrict__ igate,
                  float *__restrict__ S, float *__restrict__ nst, float *__restrict__ mst,
                  Tin *__restrict__ h, int dv) {
    constexpr int NV = DK / (4 * kLanesPerRow);
    const int head = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, rg = lane >> 3;
    const Tin *qh = q + (size_t)head * DK, *kh = k + (size_t)head * DK;
    float *Sh = S + (size_t)head * dv * DK, *nh = nst + (size_t)head * DK;

    const float m = mst[head];
    const float lf = __logf(fgate[head]), ig = igate[head];
    const float mn = fmaxf(lf + m, ig);
    const float a = __expf(lf + m - mn), b = __expf(ig - mn);  // a = 0 from the empty memory
    float4 kr[NV], qr[NV], nr[NV];
    float nq = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int col = 4 * (kLanesPerRow * u + sub);
        kr[u] = load4(kh + col);
        qr[u] = load4(qh + col);
        const float4 o = *reinterpret_cast<const float4 *>(nh + col);
        nr[u] = make_float4(a * o.x + b * kr[u].x, a * o.y + b * kr[u].y, a * o.z + b * kr[u].z,
                            a * o.w + b * kr[u].w);
        nq += nr[u].x * qr[u].x + nr[u].y * qr[u].y + nr[u].z * qr[u].z + nr[u].w * qr[u].w;
    }
    nq = sum8(nq);
    const float inv = 1.f / fmaxf(fabsf(nq), __expf(-mn));
    for (int p = 0; p < dv / kRowsPerPass; ++p) {
        const int r = p * kRowsPerPass + warp * 4 + rg;
        const float vr = b * to_f(v[(size_t)head * dv + r]);
        float sq = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            float *ps = Sh + (size_t)r * DK + 4 * (kLanesPerRow * u + sub);
            float4 s = *reinterpret_cast<const float4 *>(ps);
            s = make_float4(a * s.x + vr * kr[u].x, a * s.y + vr * kr[u].y, a * s.z + vr * kr[u].z,
                            a * s.w + vr * kr[u].w);
            *reinterpret_cast<float4 *>(ps) = s;
            sq += s.x * qr[u].x + s.y * qr[u].y + s.z * qr[u].z + s.w * qr[u].w;
        }
        sq = sum8(sq);
        if (sub == 0) h[(size_t)head * dv + r] = from_f<Tin>(sq * inv);
    }
    __syncthreads();  // every row group read the old n~ and m
    if (warp == 0 && rg == 0) {
#pragma unroll
        for (int u = 0; u < NV; ++u)
            *reinterpret_cast<float4 *>(nh + 4 * (kLanesPerRow * u + sub)) = nr[u];
        if (sub == 0) mst[head] = mn;
    }
}

template <typename Tin>
cudaError_t chunked_typed(const void *q, const void *k, const void *v, const float *fgate,
                          const float *igate, const float *C0, const float *n0, const float *m0,
                          void *h, float *C_T, float *n_T, float *m_T, int B, int H, int T, int dk,
                          int dv, cudaStream_t stream, int slot) {
    auto go = [&](auto kern, int bytes) {
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), bytes, slot);
        if (e != cudaSuccess) return e;
        kern<<<dim3(dv / DVS, H, B), NT, bytes, stream>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
            fgate, igate, C0, n0, m0, static_cast<Tin *>(h), C_T, n_T, m_T, H, T, dv);
        return cudaGetLastError();
    };
    switch (dk) {
    case 32: return go(chunk_simt_mlstm_kernel<32, Tin>, MlstmSmem<32>::bytes);
    case 64: return go(chunk_simt_mlstm_kernel<64, Tin>, MlstmSmem<64>::bytes);
    default: return go(chunk_simt_mlstm_kernel<128, Tin>, MlstmSmem<128>::bytes);
    }
}

}  // namespace

size_t mlstm_workspace_bytes(int B, int H, int T, int dk) { return mlstm_ws(B, H, T, dk).total; }

// Attribute slots 144..147 belong to this file.
cudaError_t launch_mlstm_chunked(const void *q, const void *k, const void *v, const float *fgate,
                                 const float *igate, const float *C0, const float *n0,
                                 const float *m0, void *h, float *C_T, float *n_T, float *m_T,
                                 int B, int H, int T, int dk, int dv, lr_dtype dt, void *ws,
                                 cudaStream_t stream) {
    if (dt == LR_DT_F32)
        return chunked_typed<float>(q, k, v, fgate, igate, C0, n0, m0, h, C_T, n_T, m_T, B, H, T,
                                    dk, dv, stream, 144 + (dk == 32 ? 0 : dk == 64 ? 1 : 2));
    const MlstmWs w = mlstm_ws(B, H, T, dk);
    uint8_t *base = static_cast<uint8_t *>(ws);
    float *m_prev = reinterpret_cast<float *>(base + w.mprev);
    float *aux = reinterpret_cast<float *>(base + w.aux);
    float *nst = reinterpret_cast<float *>(base + w.nst);
    const int nblk = (T + C - 1) / C;
    const int BH = B * H;
    mlstm_stab_kernel<<<BH, kStabThreads, 0, stream>>>(fgate, igate, m0, m_prev, m_T, T, nblk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_mlstm_tc(q, k, v, fgate, igate, m_prev, C0, h, C_T, aux, 0, B, H, T, dk, dv, ws,
                        stream);
    if (e != cudaSuccess) return e;
    switch (dk) {
    case 32: mlstm_nscan_kernel<32><<<BH, 32, 0, stream>>>(aux, n0, nst, n_T, nblk); break;
    case 64: mlstm_nscan_kernel<64><<<BH, 32, 0, stream>>>(aux, n0, nst, n_T, nblk); break;
    default: mlstm_nscan_kernel<128><<<BH, 32, 0, stream>>>(aux, n0, nst, n_T, nblk); break;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 grid(nblk, H, B);
    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(q);
    size_t rb = 0, slot = 0;
    mlstm_factor_slot(dk, &rb, &slot);
    switch (dk) {
    case 32: mlstm_den_kernel<32><<<grid, 128, 0, stream>>>(qb, aux, nst, base, rb, slot, H, T, nblk); break;
    case 64: mlstm_den_kernel<64><<<grid, 128, 0, stream>>>(qb, aux, nst, base, rb, slot, H, T, nblk); break;
    default: mlstm_den_kernel<128><<<grid, 128, 0, stream>>>(qb, aux, nst, base, rb, slot, H, T, nblk); break;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_mlstm_tc(q, k, v, fgate, igate, m_prev, C0, h, C_T, aux, 1, B, H, T, dk, dv, ws,
                           stream);
}

cudaError_t launch_mlstm_step(const void *q, const void *k, const void *v, const float *fgate,
                              const float *igate, float *Cs, float *ns, float *ms, void *h, int N,
                              int H, int dk, int dv, lr_dtype dt, cudaStream_t stream) {
    const int NH = N * H;
    auto go = [&](auto kern, auto tin) {
        using Tin = decltype(tin);
        kern<<<NH, kStepThreads, 0, stream>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
            fgate, igate, Cs, ns, ms, static_cast<Tin *>(h), dv);
        return cudaGetLastError();
    };
    if (dt == LR_DT_F32) {
        switch (dk) {
        case 32: return go(mlstm_step_kernel<32, float>, float{});
        case 64: return go(mlstm_step_kernel<64, float>, float{});
        default: return go(mlstm_step_kernel<128, float>, float{});
        }
    }
    using bf = __nv_bfloat16;
    switch (dk) {
    case 32: return go(mlstm_step_kernel<32, bf>, bf{});
    case 64: return go(mlstm_step_kernel<64, bf>, bf{});
    default: return go(mlstm_step_kernel<128, bf>, bf{});
    }
}

}  // namespace lr
