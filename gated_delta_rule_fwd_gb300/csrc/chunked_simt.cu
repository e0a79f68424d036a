// Chunked forward on CUDA cores, all arithmetic in fp32 (no tensor cores, so
// fp32 inputs keep fp32 accuracy).
//
// The chunkwise form (page "Le architetture lineari: RetNet, RWKV, xLSTM",
// section "RetNet: la retention e le sue tre forme"): blocks of C = 64 tokens
// computed together, the end-of-block state carried to the next block.
// Inside a block, with G_r = sum_{i<=r} ln alpha_i (log-space gate products,
// which depend on the input alone -- page "Scrivere meglio nella memoria: gate
// e delta rule", section "Correggere: la delta rule") and g_r = exp(G_r):
//
//   delta rows, pseudo-values of the WY representation (same section):
//     u_r = beta_r (v_r - g_r S k_r - sum_{i<r} e^{G_r - G_i} (k_i.k_r) u_i)
//     i.e. (I + A) U = diag(beta) (V - diag(g) K S^T),
//          A_ri = beta_r e^{G_r - G_i} k_i.k_r  (i < r);
//   other rows: u_r = v_r;
//   output    O = diag(g) Q S^T + (Q K^T (.) M) U,  M_ri = e^{G_r - G_i}, i <= r;
//   carry     S <- g_C S + U^T diag(e^{G_C - G_i}) K.
//
// Grid: one CTA per (value-channel slice of 32 rows, head, batch); rows of S
// evolve independently given k, alpha and beta, so slices never exchange
// data.  The loop over blocks is sequential inside the CTA.  The triangular
// system is solved by forward substitution, one warp per 4 columns with 8
// lanes splitting each inner sum.  A final block shorter than C is padded
// with k = q = v = 0, alpha = 1, beta = 0, which leaves state and outputs of
// the real tokens unchanged; padded outputs are not stored.
//
// The lr_fuse maps act on what a block stages: the gates as they are read
// (ln alpha formed directly from the pre-activation), and SiLU + L2 of the q
// and k rows in shared memory (fp32, one warp per row).  The output RMSNorm
// needs all d_v channels of a token, which are spread over the CTAs of a
// head; it runs as a separate pass (norm.cu).
#include "lr_internal.cuh"

namespace lr {
namespace {

constexpr int C = 64;     // tokens per block
constexpr int DVS = 32;   // value channels per CTA
constexpr int NT = 256;   // threads per CTA

template <int DK>
struct SimtSmem {
    static constexpr int KP = DK + 1;       // padded key row (bank-conflict-free column walks)
    static constexpr int UP = DVS + 1;      // padded pseudo-value row
    static constexpr int PP = C + 1;        // padded score row
    static constexpr int kK = 0;
    static constexpr int kQ = kK + C * KP;
    static constexpr int kS = kQ + C * KP;
    static constexpr int kV = kS + DVS * KP;
    static constexpr int kU = kV + C * DVS;
    static constexpr int kP = kU + C * UP;
    static constexpr int kA = kP + C * PP;
    static constexpr int kG = kA + C * PP;
    static constexpr int kB = kG + C;
    static constexpr int kW = kB + C;
    static constexpr int floats = kW + C;
    static constexpr int bytes = floats * 4;
};

template <int DK, typename Tin, bool ALPHA, bool DELTA>
__global__ void __launch_bounds__(NT)
chunk_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                  const Tin *__restrict__ v, const float *__restrict__ alpha,
                  const float *__restrict__ beta, const float *__restrict__ S0,
                  Tin *__restrict__ o, float *__restrict__ ST, int H, int T, int dv,
                  const Fuse fz) {
    using L = SimtSmem<DK>;
    constexpr int KP = L::KP, UP = L::UP, PP = L::PP;
    extern __shared__ float sm[];
    float *Ks = sm + L::kK;
    float *Qs = sm + L::kQ;
    float *Ss = sm + L::kS;
    float *Vs = sm + L::kV;
    float *Us = sm + L::kU;
    float *Ps = sm + L::kP;
    float *As = sm + L::kA;
    float *Gs = sm + L::kG;
    float *Bs = sm + L::kB;
    float *Ws = sm + L::kW;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const unsigned fl = fz.flags;
    const bool amap = (fl & kAlphaMaps) != 0;
    const float ac = (ALPHA && (fl & kScaledAlphaMaps)) ? fz.ascale[blockIdx.y] : 0.f;

    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        Ss[c * KP + j] = S0 ? S0[(bh * dv + c0 + c) * DK + j] : 0.f;
    }

    for (int t0 = 0; t0 < T; t0 += C) {
        const int n = min(C, T - t0);
        __syncthreads();  // the previous block is done with every buffer

        // ---- stage the block (fp32 in shared memory)
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
        if (tid < C) {
            const bool ok = tid < n;
            float la = 0.f, b = 0.f;
            if (ALPHA && ok) {
                const float a = alpha[bh * T + t0 + tid];
                la = amap ? log_gate(fl, a, ac) : logf(a);
            }
            if (DELTA && ok) b = write_strength(fl, beta[bh * T + t0 + tid]);
            Gs[tid] = la;
            Bs[tid] = b;
        }
        __syncthreads();

        // ---- SiLU + L2 of the q and k rows (padded rows stay zero)
        if (fl & LR_FUSE_QK_SILU_L2) {
            for (int rr = warp; rr < 2 * C; rr += NT / 32) {
                float *row = rr < C ? Qs + rr * KP : Ks + (rr - C) * KP;
                float x[DK / 32];
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < DK / 32; ++e) {
                    x[e] = silu_f(row[lane + 32 * e]);
                    ss += x[e] * x[e];
                }
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
                const float inv = inv_l2(ss);
#pragma unroll
                for (int e = 0; e < DK / 32; ++e) row[lane + 32 * e] = x[e] * inv;
            }
        }

        // ---- cumulative log decay: inclusive scan of 64 values by warp 0
        if (ALPHA && warp == 0) {
            const float x0 = Gs[2 * lane], x1 = Gs[2 * lane + 1];
            const float pair = x0 + x1;
            float incl = pair;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += y;
            }
            const float excl = incl - pair;
            Gs[2 * lane] = excl + x0;
            Gs[2 * lane + 1] = excl + pair;
        }
        __syncthreads();
        if (tid < C) Ws[tid] = ALPHA ? expf(Gs[C - 1] - Gs[tid]) : 1.f;

        // ---- decay-masked scores P and delta couplings A
        for (int idx = tid; idx < C * C; idx += NT) {
            const int r = idx / C, i = idx % C;
            float p = 0.f, a = 0.f;
            if (i <= r) {
                float dq = 0.f, dk = 0.f;
#pragma unroll 8
                for (int j = 0; j < DK; ++j) {
                    const float kij = Ks[i * KP + j];
                    dq += Qs[r * KP + j] * kij;
                    if (DELTA) dk += Ks[r * KP + j] * kij;
                }
                const float dec = ALPHA ? expf(Gs[r] - Gs[i]) : 1.f;
                p = dq * dec;
                if (DELTA && i < r) a = Bs[r] * dk * dec;
            }
            Ps[r * PP + i] = p;
            if (DELTA) As[r * PP + i] = a;
        }

        // ---- right-hand side of the pseudo-value system (delta rows)
        if (DELTA) {
            for (int idx = tid; idx < C * DVS; idx += NT) {
                const int r = idx / DVS, c = idx % DVS;
                float sk = 0.f;
#pragma unroll 8
                for (int j = 0; j < DK; ++j) sk += Ss[c * KP + j] * Ks[r * KP + j];
                const float g = ALPHA ? expf(Gs[r]) : 1.f;
                Us[r * UP + c] = Bs[r] * (Vs[r * DVS + c] - g * sk);
            }
        } else {
            for (int idx = tid; idx < C * DVS; idx += NT) {
                const int r = idx / DVS, c = idx % DVS;
                Us[r * UP + c] = Vs[r * DVS + c];
            }
        }
        __syncthreads();

        // ---- forward substitution (I + A) U = rhs, in place in Us
        if (DELTA) {
            const int c = warp * 4 + (lane >> 3);
            const int sub = lane & 7;
            for (int r = 1; r < C; ++r) {
                float part = 0.f;
                for (int i = sub; i < r; i += 8) part += As[r * PP + i] * Us[i * UP + c];
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                if (sub == 0) Us[r * UP + c] -= part;
                __syncwarp();
            }
        }
        __syncthreads();

        // ---- output O = diag(g) Q S^T + P U  (S still the block's initial state)
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            if (r >= n) continue;
            float qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) qs += Qs[r * KP + j] * Ss[c * KP + j];
            float pu = 0.f;
            for (int i = 0; i <= r; ++i) pu += Ps[r * PP + i] * Us[i * UP + c];
            const float g = ALPHA ? expf(Gs[r]) : 1.f;
            o[(bh * T + t0 + r) * dv + c0 + c] = from_f<Tin>(g * qs + pu);
        }
        __syncthreads();

        // ---- carry S <- g_C S + U^T diag(e^{G_C - G_i}) K
        const float gC = ALPHA ? expf(Gs[C - 1]) : 1.f;
        for (int idx = tid; idx < DVS * DK; idx += NT) {
            const int c = idx / DK, j = idx % DK;
            float acc = 0.f;
#pragma unroll 8
            for (int i = 0; i < C; ++i) acc += Us[i * UP + c] * Ws[i] * Ks[i * KP + j];
            Ss[c * KP + j] = gC * Ss[c * KP + j] + acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        ST[(bh * dv + c0 + c) * DK + j] = Ss[c * KP + j];
    }
}

// ---------------------------------------------------------- diagonal gate
// The GLA row (page "Scrivere meglio nella memoria: gate e delta rule",
// section "Dimenticare: i gate"): S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T with
// one gate per key channel.  Inside a block, G_r[c] = sum_{i<=r} ln alpha_i[c]
// (per channel), and
//   O   = (Q * e^G) S^T + P V,       P_ri = sum_c q_r[c] k_i[c] e^{G_r[c] - G_i[c]}, i <= r
//   S  <- S Diag(e^{G_last}) + V^T (K * e^{G_last - G}).
// The scores use a second level of 16-token blocks (the summary of the same
// page: GLA needs it for numerical stability): for the key sub-block J,
//   P[:, J] = (Q * e^{G - G_e}) (K_J * e^{G_e - G_J})^T,  G_e = G at the last token of J,
// where the key factor is <= 1 and the query factor is <= 1 for rows after J
// and at most e^80 (clamped) for rows inside J.
template <int DK>
struct DiagSmem {
    static constexpr int KP = DK + 1, PP = C + 1;
    static constexpr int kK = 0;                // K, then K * e^{G_last - G}
    static constexpr int kQ = kK + C * KP;      // Q, then Q * e^G
    static constexpr int kS = kQ + C * KP;      // state slice [DVS][KP]
    static constexpr int kV = kS + DVS * KP;    // V slice [C][DVS]
    static constexpr int kP = kV + C * DVS;     // P [C][PP]
    static constexpr int kG = kP + C * PP;      // G [C][KP]
    static constexpr int kQh = kG + C * KP;     // query factors of one key sub-block
    static constexpr int kKh = kQh + C * KP;    // K * e^{G_e - G}
    static constexpr int floats = kKh + C * KP;
    static constexpr int bytes = floats * 4;
};
constexpr int kSub = 16;

template <int DK, typename Tin>
__global__ void __launch_bounds__(NT)
chunk_simt_diag_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                       const Tin *__restrict__ v, const float *__restrict__ alpha,
                       const float *__restrict__ S0, Tin *__restrict__ o, float *__restrict__ ST,
                       int H, int T, int dv, const Fuse fz) {
    using L = DiagSmem<DK>;
    constexpr int KP = L::KP, PP = L::PP;
    extern __shared__ float sm[];
    float *Ks = sm + L::kK, *Qs = sm + L::kQ, *Ss = sm + L::kS, *Vs = sm + L::kV;
    float *Ps = sm + L::kP, *Gs = sm + L::kG, *Qh = sm + L::kQh, *Kh = sm + L::kKh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const unsigned fl = fz.flags;
    const float ac = (fl & kScaledAlphaMaps) ? fz.ascale[blockIdx.y] : 0.f;

    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        Ss[c * KP + j] = S0 ? S0[(bh * dv + c0 + c) * DK + j] : 0.f;
    }

    for (int t0 = 0; t0 < T; t0 += C) {
        const int n = min(C, T - t0);
        __syncthreads();  // the previous block is done with every buffer

        // ---- stage the block: q, k, v, ln alpha (zero past the end)
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, j = idx % DK;
            const bool ok = r < n;
            const size_t g = (bh * T + t0 + r) * DK + j;
            Ks[r * KP + j] = ok ? to_f(k[g]) : 0.f;
            Qs[r * KP + j] = ok ? to_f(q[g]) : 0.f;
            float la = 0.f;
            if (ok) {
                const float a = alpha[g];
                la = (fl & kAlphaMaps) ? log_gate(fl, a, ac) : logf(a);
            }
            Gs[r * KP + j] = la;
        }
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            Vs[r * DVS + c] = r < n ? to_f(v[(bh * T + t0 + r) * dv + c0 + c]) : 0.f;
        }
        __syncthreads();

        // ---- cumulative log gates per channel; SiLU + L2 of the q and k rows
        if (tid < DK) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) {
                acc += Gs[r * KP + tid];
                Gs[r * KP + tid] = acc;
            }
        } else if (fl & LR_FUSE_QK_SILU_L2) {
            // the warps past the first DK threads normalise the rows meanwhile
            for (int rr = warp - DK / 32; rr < 2 * C; rr += NT / 32 - DK / 32) {
                float *row = rr < C ? Qs + rr * KP : Ks + (rr - C) * KP;
                float x[DK / 32];
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < DK / 32; ++e) {
                    x[e] = silu_f(row[lane + 32 * e]);
                    ss += x[e] * x[e];
                }
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
                const float inv = inv_l2(ss);
#pragma unroll
                for (int e = 0; e < DK / 32; ++e) row[lane + 32 * e] = x[e] * inv;
            }
        }
        __syncthreads();

        // ---- key factors K * e^{G_e - G} (G_e: last token of the key's sub-block)
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int i = idx / DK, j = idx % DK;
            const int e = (i | (kSub - 1));
            Kh[i * KP + j] = Ks[i * KP + j] * __expf(Gs[e * KP + j] - Gs[i * KP + j]);
        }
        // ---- scores, one key sub-block at a time
        for (int J = 0; J < C / kSub; ++J) {
            const int e = J * kSub + kSub - 1, r0 = J * kSub;
            for (int idx = tid; idx < (C - r0) * DK; idx += NT) {
                const int r = r0 + idx / DK, j = idx % DK;
                Qh[r * KP + j] = Qs[r * KP + j] * __expf(fminf(Gs[r * KP + j] - Gs[e * KP + j], 80.f));
            }
            __syncthreads();
            for (int idx = tid; idx < C * kSub; idx += NT) {
                const int r = idx / kSub, i = r0 + idx % kSub;
                float p = 0.f;
                if (i <= r) {
#pragma unroll 8
                    for (int j = 0; j < DK; ++j) p += Qh[r * KP + j] * Kh[i * KP + j];
                }
                Ps[r * PP + i] = p;
            }
            __syncthreads();
        }

        // ---- Q * e^G and K * e^{G_last - G}
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, j = idx % DK;
            const float G = Gs[r * KP + j], Gl = Gs[(C - 1) * KP + j];
            Qs[r * KP + j] *= __expf(G);
            Ks[r * KP + j] *= __expf(Gl - G);
        }
        __syncthreads();

        // ---- output O = (Q * e^G) S^T + P V  (S still the block's initial state)
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, c = idx % DVS;
            if (r >= n) continue;
            float qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) qs += Qs[r * KP + j] * Ss[c * KP + j];
            float pv = 0.f;
            for (int i = 0; i <= r; ++i) pv += Ps[r * PP + i] * Vs[i * DVS + c];
            o[(bh * T + t0 + r) * dv + c0 + c] = from_f<Tin>(qs + pv);
        }
        __syncthreads();

        // ---- carry S <- S Diag(e^{G_last}) + V^T (K * e^{G_last - G})
        for (int idx = tid; idx < DVS * DK; idx += NT) {
            const int c = idx / DK, j = idx % DK;
            float acc = 0.f;
#pragma unroll 8
            for (int i = 0; i < C; ++i) acc += Vs[i * DVS + c] * Ks[i * KP + j];
            Ss[c * KP + j] = __expf(Gs[(C - 1) * KP + j]) * Ss[c * KP + j] + acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < DVS * DK; idx += NT) {
        const int c = idx / DK, j = idx % DK;
        ST[(bh * dv + c0 + c) * DK + j] = Ss[c * KP + j];
    }
}

template <int DK, typename Tin>
cudaError_t launch_diag(const void *q, const void *k, const void *v, const float *alpha,
                        const float *S0, void *o, float *S_T, int B, int H, int T, int dv,
                        const Fuse &fz, cudaStream_t stream, int slot) {
    auto fn = chunk_simt_diag_kernel<DK, Tin>;
    const int bytes = DiagSmem<DK>::bytes;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), bytes, slot);
    if (e != cudaSuccess) return e;
    fn<<<dim3(dv / DVS, H, B), NT, bytes, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, S0, static_cast<Tin *>(o), S_T, H, T, dv, fz);
    return cudaGetLastError();
}

template <int DK, typename Tin, bool ALPHA, bool DELTA>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                         int T, int dv, const Fuse &fz, cudaStream_t stream, int slot) {
    auto fn = chunk_simt_kernel<DK, Tin, ALPHA, DELTA>;
    const int bytes = SimtSmem<DK>::bytes;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), bytes, slot);
    if (e != cudaSuccess) return e;
    dim3 grid(dv / DVS, H, B);
    fn<<<grid, NT, bytes, stream>>>(static_cast<const Tin *>(q), static_cast<const Tin *>(k),
                                    static_cast<const Tin *>(v), alpha, beta, S0,
                                    static_cast<Tin *>(o), S_T, H, T, dv, fz);
    return cudaGetLastError();
}

template <int DK, typename Tin>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                        int T, int dv, lr_mode mode, const Fuse &fz, cudaStream_t stream,
                        int slot) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, Tin, false, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T,
                                                   dv, fz, stream, slot + 0);
    case LR_MODE_DECAY:
        return launch_typed<DK, Tin, true, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T,
                                                  dv, fz, stream, slot + 1);
    case LR_MODE_DELTA:
        return launch_typed<DK, Tin, false, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T,
                                                  dv, fz, stream, slot + 2);
    case LR_MODE_DIAG_DECAY:
        return launch_diag<DK, Tin>(q, k, v, alpha, S0, o, S_T, B, H, T, dv, fz, stream,
                                    slot + 96);
    default:
        return launch_typed<DK, Tin, true, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv,
                                                 fz, stream, slot + 3);
    }
}

template <typename Tin>
cudaError_t launch_dk(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                      int T, int dk, int dv, lr_mode mode, const Fuse &fz, cudaStream_t stream,
                      int slot) {
    switch (dk) {
    case 32:
        return launch_mode<32, Tin>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, fz,
                                    stream, slot + 0);
    case 64:
        return launch_mode<64, Tin>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, fz,
                                    stream, slot + 4);
    default:
        return launch_mode<128, Tin>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode,
                                     fz, stream, slot + 8);
    }
}

}  // namespace

// Attribute slots 0..23 and 96..119 (diagonal gate) belong to this file.
cudaError_t launch_chunked_simt(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *S_T, int B,
                                int H, int T, int dk, int dv, lr_dtype dt, lr_mode mode,
                                const Fuse &fz, cudaStream_t stream) {
    if (dt == LR_DT_F32)
        return launch_dk<float>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, mode, fz,
                                stream, 0);
    return launch_dk<__nv_bfloat16>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, mode, fz,
                                    stream, 12);
}

}  // namespace lr
