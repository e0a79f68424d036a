// Generalised delta rule of RWKV-7 on the tensor cores (page "Le architetture
// lineari: RetNet, RWKV, xLSTM", RWKV section, read in the chapter's
// convention as S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) +
// v_t kw_t^T, o_t = S_t q_t).
//
// Blocks of 32 tokens.  Inside block j, with S_j the state when it starts, L
// the per-channel cumulative log decay (inclusive), b = a * kappa and u_t =
// S_{t-1} kappa_t (first page, delta-rule section: the pseudo-values of the
// WY representation, here with per-channel decays), unrolling the block gives
//   (I + A) U = Kdec S_j^T + Bk V,   A_ts  = (b_s e^{L_{t-1} - L_s}) . kappa_t,
//                                    Bk_ts = (kw_s e^{L_{t-1} - L_s}) . kappa_t  (s < t)
//   O = Qd S_j^T + Qk V - Qb U,      Qk_ts = (kw_s e^{L_t - L_s}) . q_t,
//                                    Qb_ts = (b_s e^{L_t - L_s}) . q_t           (s <= t)
//   S_{j+1} = S_j D_j + V^T Kw' - U^T B'
// with Kdec_t = kappa_t e^{L_{t-1}}, Qd_t = q_t e^{L_t}, Kw'_s = kw_s e^{L_last - L_s},
// B'_s = b_s e^{L_last - L_s} and D_j = Diag(e^{L_last}).  So U = Wg S_j^T + Tb V
// with Wg = (I + A)^{-1} Kdec and Tb = (I + A)^{-1} Bk.
//
// Stacking values on pseudo-values, Ut_j = [V_j; U_j] (64 rows) and Kt_j =
// [Kw'_j; -B'_j] (64 x dk), this is the look-ahead form the tensor-core scan
// evaluates for the delta rule (scan_tc.cuh), with a 64-row U and 32 output rows:
//   Ut_{j+1} = [I; Tb_{j+1}] V_{j+1} + [0; Wg_{j+1} D_j] S_j^T + [0; Wg_{j+1} Kt_j^T] Ut_j
//   O_j      = Qd_j S_j^T + [Qk_j, -Qb_j] Ut_j
//   S_{j+1}  = S_j D_j + Ut_j^T Kt_j
// This file's per-block pass computes everything that does not depend on the
// state, for all blocks in parallel, on the CUDA cores in fp32, and writes the
// scan's record of stage j (the W tile [0; Wg_j D_{j-1}], the T rows
// [I | 0; Tb_j | 0], the Z rows [0; Wg_j Kt_{j-1}^T], D_{j-1} per key channel)
// plus stage j+1's P rows [Qk_j | -Qb_j], and the per-stage q and k operands
// (Qd_j over 32 zero rows; Kt_j).  The previous block's Kt, needed for the Z
// rows, is recomputed from its inputs.
//
// The four score matrices are products over the key channels once the decay
// is split at a reference token r: e^{L_t - L_s} = e^{L_t - L_r} e^{L_r - L_s}.
// r is the last token of the key's 16-token half, so the key factor is at
// most 1; the query factor is too for queries after r and is at most e^80
// (clamped) for queries inside the half, i.e. exact while the decay over any
// 16 consecutive tokens stays above e^-80.
#include "scan_tc.cuh"

namespace lr {
namespace {

constexpr int GC = 32;          // tokens per block (one scan stage)
constexpr int GH = GC / 2;      // tokens per half (reference of the key factors)
constexpr int GNT = 256;        // threads of the per-block pass
constexpr float kMaxUp = 80.f;  // largest exponent of a query factor

// Shared memory of the per-block pass (fp32 rows padded to 16 bytes past a
// multiple of 128 so that 8 consecutive rows read as float4 hit distinct banks).
template <int DK>
struct GdPrep {
    static constexpr int KP = DK + 4;            // row of a [32][DK] operand
    static constexpr int SP = GC + 4;            // row of a 32 x 32 matrix
    static constexpr int ZP = 2 * GC + 4;        // row of the 32 x 64 Z rows
    static constexpr int kQS = 0;                // q_t e^{L_t - L_15}; then Kt_{j-1} rows 0..31
    static constexpr int kKS = kQS + GC * KP;    // kappa_t e^{L_{t-1} - L_15}; then Kt_{j-1} rows 32..63
    static constexpr int kKw = kKS + GC * KP;    // kw_s e^{L_r - L_s}; then the Z rows (over kBv too)
    static constexpr int kBv = kKw + GC * KP;    // b_s e^{L_r - L_s}
    static constexpr int kX = kBv + GC * KP;     // second-half query factors; then Wg
    static constexpr int kA = kX + GC * KP;      // A
    static constexpr int kBk = kA + GC * SP;     // Bk, solved in place into Tb
    static constexpr int kQk = kBk + GC * SP;
    static constexpr int kQb = kQk + GC * SP;
    static constexpr int kD = kQb + GC * SP;     // D_{j-1} per key channel
    static constexpr int floats = kD + DK;
    static constexpr int bytes = floats * 4;
    static_assert(GC * ZP <= 2 * GC * KP, "the Z rows must fit over the kw and b rows");
};

__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ void fma4(float &acc, float4 x, float4 y) {
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
    acc = fmaf(x.z, y.z, acc);
    acc = fmaf(x.w, y.w, acc);
}

// One CTA per (block, head, batch).  q, kw [B*H][T][DK] bf16; w, kappa, a
// [B*H][T][DK] fp32; ws: the records (B*H x (nblk + 1)); qo, ko: the per-stage
// q and k operands, [B*H][nblk * 64][DK] bf16 each.
template <int DK>
__global__ void __launch_bounds__(GNT, 2)
chunk_prep_gd_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ kw,
                     const float *__restrict__ w, const float *__restrict__ kappa,
                     const float *__restrict__ ar, uint8_t *__restrict__ ws, bf16 *__restrict__ qo,
                     bf16 *__restrict__ ko, int H, int T, int nblk) {
    using G = GdPrep<DK>;
    using R = Rec<DK>;
    constexpr int KP = G::KP, SP = G::SP, ZP = G::ZP;
    extern __shared__ float4 gd_smem[];
    float *sm = reinterpret_cast<float *>(gd_smem);
    float *QS = sm + G::kQS, *KS = sm + G::kKS, *KwS = sm + G::kKw, *BvS = sm + G::kBv;
    float *X = sm + G::kX, *Am = sm + G::kA, *Bk = sm + G::kBk, *Qk = sm + G::kQk, *Qb = sm + G::kQb;
    float *Dp = sm + G::kD;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = j * GC, n = min(GC, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + j) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    bf16 *qrow = qo + (bh * nblk + j) * (size_t)(2 * GC) * DK;
    bf16 *krow = ko + (bh * nblk + j) * (size_t)(2 * GC) * DK;
    const bf16 zero = __float2bfloat16_rn(0.f);

    // ---- this block, one thread per key channel: decays, scaled operands,
    //      the stage's q and k rows; Kdec stays in registers for the solve
    float kdec[GC];
    float Dj = 1.f;  // e^{L_last} of this block
    if (tid < DK) {
        const int c = tid;
        const size_t g0 = (bh * T + t0) * DK + c;
        float L[GC];
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < GC; ++t) {
            acc += t < n ? logf(w[g0 + (size_t)t * DK]) : 0.f;
            L[t] = acc;
        }
        const float Lh = L[GH - 1], Ll = L[GC - 1];
        const float fh = __expf(Ll - Lh);               // first half's reference to the block end
        float ks0 = __expf(fminf(-Lh, kMaxUp));         // e^{L_{t-1} - L_15} at t = 0 (L_{-1} = 0)
        float ks1 = 0.f, eprev = 1.f;
#pragma unroll
        for (int t = 0; t < GC; ++t) {
            const bool ok = t < n;
            const size_t g = g0 + (size_t)t * DK;
            const float qf = ok ? __bfloat162float(q[g]) : 0.f;
            const float kf = ok ? __bfloat162float(kw[g]) : 0.f;
            const float kp = ok ? kappa[g] : 0.f;
            const float bf = ok ? ar[g] * kp : 0.f;
            const float Lt = L[t];
            const float fk = __expf((t < GH ? Lh : Ll) - Lt);  // key factor, at most 1
            KwS[t * KP + c] = kf * fk;
            BvS[t * KP + c] = bf * fk;
            const float q0 = __expf(fminf(Lt - Lh, kMaxUp));
            QS[t * KP + c] = qf * q0;
            KS[t * KP + c] = kp * ks0;
            ks0 = q0;
            if (t >= GH) {
                if (t == GH) ks1 = __expf(fminf(Lh - Ll, kMaxUp));
                const float q1 = __expf(fminf(Lt - Ll, kMaxUp));
                X[(t - GH) * KP + c] = qf * q1;  // second-half query rows 0..15
                X[t * KP + c] = kp * ks1;        // second-half removal-key rows 16..31
                ks1 = q1;
            }
            kdec[t] = kp * eprev;
            const float eL = __expf(Lt);
            eprev = eL;
            qrow[t * DK + c] = __float2bfloat16_rn(qf * eL);
            qrow[(GC + t) * DK + c] = zero;
            const float fK = t < GH ? fk * fh : fk;  // e^{L_last - L_t}
            krow[t * DK + c] = __float2bfloat16_rn(kf * fK);
            krow[(GC + t) * DK + c] = __float2bfloat16_rn(-bf * fK);
        }
        Dj = __expf(Ll);
    }
    __syncthreads();

    // ---- the four score matrices: warps 0..3 take queries 0..31 against keys
    //      0..15 (reference 15), warps 4..5 queries 16..31 against keys 16..31
    //      (reference 31); each lane a 2 x 2 tile of all four
    if (warp < 6) {
        const int rt = lane >> 3, ct = lane & 7;
        const bool second = warp >= 4;
        const int tb = second ? GH + 8 * (warp - 4) : 8 * warp, sb = second ? GH : 0;
        const int tr[2] = {tb + rt, tb + rt + 4}, sc[2] = {sb + ct, sb + ct + 8};
        const float *qp[2], *kp[2], *wp[2], *bp[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            qp[i] = second ? X + (tr[i] - GH) * KP : QS + tr[i] * KP;
            kp[i] = second ? X + tr[i] * KP : KS + tr[i] * KP;
            wp[i] = KwS + sc[i] * KP;
            bp[i] = BvS + sc[i] * KP;
        }
        float qk[4] = {0.f, 0.f, 0.f, 0.f}, qb[4] = {0.f, 0.f, 0.f, 0.f};
        float bk[4] = {0.f, 0.f, 0.f, 0.f}, aa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c4 = 0; c4 < DK; c4 += 4) {
            const float4 q0 = lds4(qp[0] + c4), q1 = lds4(qp[1] + c4);
            const float4 k0 = lds4(kp[0] + c4), k1 = lds4(kp[1] + c4);
            const float4 w0 = lds4(wp[0] + c4), w1 = lds4(wp[1] + c4);
            const float4 b0 = lds4(bp[0] + c4), b1 = lds4(bp[1] + c4);
            fma4(qk[0], q0, w0), fma4(qk[1], q0, w1), fma4(qk[2], q1, w0), fma4(qk[3], q1, w1);
            fma4(qb[0], q0, b0), fma4(qb[1], q0, b1), fma4(qb[2], q1, b0), fma4(qb[3], q1, b1);
            fma4(bk[0], k0, w0), fma4(bk[1], k0, w1), fma4(bk[2], k1, w0), fma4(bk[3], k1, w1);
            fma4(aa[0], k0, b0), fma4(aa[1], k0, b1), fma4(aa[2], k1, b0), fma4(aa[3], k1, b1);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int l = 0; l < 2; ++l) {
                const int t = tr[i], s = sc[l], e = 2 * i + l;
                Qk[t * SP + s] = s <= t ? qk[e] : 0.f;
                Qb[t * SP + s] = s <= t ? qb[e] : 0.f;
                Bk[t * SP + s] = s < t ? bk[e] : 0.f;
                Am[t * SP + s] = s < t ? aa[e] : 0.f;
            }
    } else {
        // queries of the first half never see keys of the second
        for (int i = tid - 6 * 32; i < GH * GH; i += 2 * 32) {
            const int t = i / GH, s = GH + i % GH;
            Qk[t * SP + s] = Qb[t * SP + s] = Bk[t * SP + s] = Am[t * SP + s] = 0.f;
        }
    }
    __syncthreads();

    // ---- (I + A) [Wg | Tb] = [Kdec | Bk] by forward substitution, one column
    //      per thread (Kdec columns from registers, Bk columns in place)
    if (tid < DK + GC) {
        const bool tcol = tid >= DK;
        float x[GC];
#pragma unroll
        for (int t = 0; t < GC; ++t) x[t] = tcol ? Bk[t * SP + (tid - DK)] : kdec[t];
#pragma unroll
        for (int t = 1; t < GC; ++t) {
            float acc = x[t];
            // whole float4 groups: A is stored zero on and above the diagonal
#pragma unroll
            for (int s4 = 0; s4 < t; s4 += 4) {
                const float4 a4 = lds4(Am + t * SP + s4);
                acc = fmaf(-a4.x, x[s4], acc);
                acc = fmaf(-a4.y, x[s4 + 1], acc);
                acc = fmaf(-a4.z, x[s4 + 2], acc);
                acc = fmaf(-a4.w, x[s4 + 3], acc);
            }
            x[t] = acc;
        }
        if (tcol) {
#pragma unroll
            for (int t = 0; t < GC; ++t) Bk[t * SP + (tid - DK)] = x[t];
        } else {
#pragma unroll
            for (int t = 0; t < GC; ++t) X[t * KP + tid] = x[t];
        }
    }
    // ---- the previous block's Kt = [Kw'; -B'] and D, recomputed (same threads
    //      as the Kdec columns, disjoint shared memory)
    if (tid < DK) {
        const int c = tid;
        float *Kt = QS;  // [64][KP] over the QS and KS rows
        if (j == 0) {
#pragma unroll 4
            for (int s = 0; s < 2 * GC; ++s) Kt[s * KP + c] = 0.f;
            Dp[c] = 1.f;
        } else {
            const size_t g0 = (bh * T + t0 - GC) * DK + c;  // block j-1 is full
            float Lp[GC];
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < GC; ++s) {
                acc += logf(w[g0 + (size_t)s * DK]);
                Lp[s] = acc;
            }
#pragma unroll
            for (int s = 0; s < GC; ++s) {
                const size_t g = g0 + (size_t)s * DK;
                const float f = __expf(acc - Lp[s]);
                const float kp = kappa[g];
                Kt[s * KP + c] = __bfloat162float(kw[g]) * f;
                Kt[(GC + s) * KP + c] = -ar[g] * kp * f;
            }
            Dp[c] = __expf(acc);
        }
    }
    __syncthreads();

    // ---- Z rows Wg Kt^T (32 x 64), each lane a 2 x 4 tile, staged over the kw and b rows
    {
        const int rt = lane >> 3, ct = lane & 7;
        const int rb = 8 * (warp & 3), cb = 32 * (warp >> 2);
        const float *xp0 = X + (rb + rt) * KP, *xp1 = X + (rb + rt + 4) * KP;
        const float *kt = QS + (cb + ct) * KP;
        float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c4 = 0; c4 < DK; c4 += 4) {
            const float4 x0 = lds4(xp0 + c4), x1 = lds4(xp1 + c4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 k4 = lds4(kt + 8 * i * KP + c4);
                fma4(z[i], x0, k4);
                fma4(z[4 + i], x1, k4);
            }
        }
        float *Z = KwS;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Z[(rb + rt) * ZP + cb + ct + 8 * i] = z[i];
            Z[(rb + rt + 4) * ZP + cb + ct + 8 * i] = z[4 + i];
        }
    }
    __syncthreads();

    // ---- the records, as bf16 tiles in the scan's operand layout
    {
        const float *Z = KwS;
        constexpr int WCH = DK / 8;  // 8-column chunks of a W row
        for (int i = tid; i < 2 * GC * WCH; i += GNT) {  // W = [0; Wg_j D_{j-1}]
            const int r = i / WCH, c8 = (i % WCH) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = r < GC ? 0.f : X[(r - GC) * KP + c8 + e] * Dp[c8 + e];
            *reinterpret_cast<uint4 *>(rec + R::WT + sw128_offset(r, c8, 64)) = pack8(x);
        }
        for (int i = tid; i < 128 * 8; i += GNT) {  // T rows [I | 0; Tb | 0], Z rows [0; Z]
            const int r = i >> 3, c8 = (i & 7) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int col = c8 + e;
                x[e] = r < GC          ? (col == r ? 1.f : 0.f)
                       : r < 2 * GC    ? (col < GC ? Bk[(r - GC) * SP + col] : 0.f)
                       : r < 3 * GC    ? 0.f
                                       : Z[(r - 3 * GC) * ZP + col];
            }
            *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(r, c8, 192)) = pack8(x);
        }
        for (int i = tid; i < 64 * 8; i += GNT) {  // stage j+1's P rows [Qk | -Qb; 0]
            const int r = i >> 3, c8 = (i & 7) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int col = c8 + e;
                x[e] = r >= GC ? 0.f : col < GC ? Qk[r * SP + col] : -Qb[r * SP + col - GC];
            }
            *reinterpret_cast<uint4 *>(rec_next + R::TZP + sw128_offset(128 + r, c8, 192)) = pack8(x);
        }
        float *vec = reinterpret_cast<float *>(rec + R::VEC);
        vec[tid] = tid < DK ? Dp[tid] : 0.f;  // g_C' per key channel (GNT = 256 floats)
        if (j == nblk - 1) {
            // the closing stage reads its gate vector and (unused) T and Z rows
            float *vn = reinterpret_cast<float *>(rec_next + R::VEC);
            vn[tid] = tid < DK ? Dj : 0.f;
            for (int i = tid; i < (R::TZP + 128 * 128) / 16; i += GNT)
                reinterpret_cast<uint4 *>(rec_next)[i] = make_uint4(0, 0, 0, 0);
        }
    }
}

template <int DK>
cudaError_t launch_gd_dk(const void *q, const void *kw, const void *v, const float *w,
                         const float *kappa, const float *a, const float *S0, void *o,
                         float *S_T, int B, int H, int T, int dv, void *ws, cudaStream_t stream,
                         int slot) {
    const int nblk = (T + GC - 1) / GC;
    auto prep = chunk_prep_gd_kernel<DK>;
    auto scan = chunk_scan_kernel<DK, true, true, false, true>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), GdPrep<DK>::bytes, slot);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC, slot + 1);
    if (e != cudaSuccess) return e;
    uint8_t *recs = static_cast<uint8_t *>(ws);
    const size_t rec_bytes = (size_t)B * H * (nblk + 1) * Rec<DK>::BYTES;
    bf16 *qo = reinterpret_cast<bf16 *>(recs + rec_bytes);
    bf16 *ko = qo + (size_t)B * H * nblk * 2 * GC * DK;
    CUtensorMap tmq, tmk, tmv;
    if ((e = make_rows_map(&tmq, qo, DK, nblk * 2 * GC, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmk, ko, DK, nblk * 2 * GC, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmv, v, dv, T, B * H)) != cudaSuccess) return e;
    prep<<<dim3(nblk, H, B), GNT, GdPrep<DK>::bytes, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(kw), w, kappa, a, recs, qo, ko, H,
        T, nblk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    scan<<<dim3(dv / DVS, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
        recs, S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk, qo, ko,
        static_cast<const bf16 *>(v), tmq, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace

size_t gen_delta_tc_workspace_bytes(int B, int H, int T, int dk) {
    const size_t nblk = (size_t)((T + GC - 1) / GC);
    const size_t rec = dk == 32 ? Rec<32>::BYTES : dk == 64 ? Rec<64>::BYTES : Rec<128>::BYTES;
    return (size_t)B * H * ((nblk + 1) * rec + 2 * nblk * 2 * GC * (size_t)dk * 2);
}

// Attribute slots 154..159 belong to this file.
cudaError_t launch_gen_delta_tc(const void *q, const void *kw, const void *v, const float *w,
                                const float *kappa, const float *a, const float *S0, void *o,
                                float *S_T, int B, int H, int T, int dk, int dv, void *ws,
                                cudaStream_t stream) {
    switch (dk) {
    case 32: return launch_gd_dk<32>(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dv, ws, stream, 154);
    case 64: return launch_gd_dk<64>(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dv, ws, stream, 156);
    default:
        return launch_gd_dk<128>(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dv, ws, stream, 158);
    }
}

int read_and_clear_gd_tc_error() {
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_error, sizeof(int)) != cudaSuccess) return -1;
    if (h) cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    return h;
}

}  // namespace lr
