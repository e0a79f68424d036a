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

// Shared memory of the per-block pass: bf16 operand tiles in the 128-byte
// swizzled K-major layout of the tensor cores (1024-byte aligned), then fp32
// matrices for the solve, the barriers and the TMEM slot.
template <int DK>
struct GdPrep {
    static constexpr int KB = (DK + 63) / 64;     // 64-column blocks of a tile row
    static constexpr int SP = GC + 4;             // fp32 row of a 32 x 32 matrix
    static constexpr int AT = 0;                  // [128][DK]: query / removal-key rows, then Wg
    static constexpr int BT = AT + KB * 128 * 128;  // [64][DK]: the key rows [kw; b]
    static constexpr int KT = BT + KB * 64 * 128;   // [64][DK]: the previous block's Kt
    static constexpr int F32 = KT + KB * 64 * 128;  // fp32 A [32][SP], Bk -> Tb [32][SP], D_{j-1} [DK]
    static constexpr int BAR = F32 + (2 * GC * SP + DK) * 4;
    static constexpr int BYTES = BAR + 32;        // two mbarriers and the TMEM slot
    static constexpr int ALLOC = BYTES + 1024;
};

__device__ __forceinline__ void st_tile(uint8_t *tile, int rows, int r, int c, float x) {
    *reinterpret_cast<bf16 *>(tile + sw128_offset(r, c, rows)) = __float2bfloat16_rn(x);
}

// One CTA per (block, head, batch).  q, kw [B*H][T][DK] bf16; w, kappa, a
// [B*H][T][DK] fp32; ws: the records (B*H x (nblk + 1)); qo, ko: the per-stage
// q and k operands, [B*H][nblk * 64][DK] bf16 each.
//
// Threads 0..DK-1 take this block's key channels and threads 128..128+DK-1
// the previous block's (for its Kt).  Then two M = 128 tcgen05 products:
//   S  = [Q e^{L-L_15}; K e^{L_{t-1}-L_15}; Q e^{L-L_31}; K e^{L_{t-1}-L_31}] [kw e^{L_r-L}; b e^{L_r-L}]^T
//        (rows 64..127 only for queries of the second half), TMEM cols 0..63: the
//        four score matrices, keys 0..15 from the first reference and 16..31
//        from the second;
//   Z  = [Wg; *] Kt_{j-1}^T, TMEM cols 64..127 (rows 0..31 used);
// with the solve (I + A)[Wg | Tb] = [Kdec | Bk] on the CUDA cores between them.
template <int DK>
__global__ void __launch_bounds__(GNT, 2)
chunk_prep_gd_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ kw,
                     const float *__restrict__ w, const float *__restrict__ kappa,
                     const float *__restrict__ ar, uint8_t *__restrict__ ws, bf16 *__restrict__ qo,
                     bf16 *__restrict__ ko, int H, int T, int nblk) {
    using G = GdPrep<DK>;
    using R = Rec<DK>;
    constexpr int SP = G::SP;
    extern __shared__ uint8_t gd_raw[];
    uint8_t *sm = align1024(gd_raw);
    uint8_t *At = sm + G::AT, *Bt = sm + G::BT, *Kt = sm + G::KT;
    float *Am = reinterpret_cast<float *>(sm + G::F32);
    float *Bk = Am + GC * SP, *Dp = Am + 2 * GC * SP;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + G::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G::BAR + 16);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = j * GC, n = min(GC, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + j) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    bf16 *qrow = qo + (bh * nblk + j) * (size_t)(2 * GC) * DK;
    bf16 *krow = ko + (bh * nblk + j) * (size_t)(2 * GC) * DK;

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }

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
            acc += t < n ? __logf(w[g0 + (size_t)t * DK]) : 0.f;
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
            st_tile(Bt, 64, t, c, kf * fk);
            st_tile(Bt, 64, GC + t, c, bf * fk);
            const float q0 = __expf(fminf(Lt - Lh, kMaxUp));
            st_tile(At, 128, t, c, qf * q0);
            st_tile(At, 128, GC + t, c, kp * ks0);
            ks0 = q0;
            if (t >= GH) {
                if (t == GH) ks1 = __expf(fminf(Lh - Ll, kMaxUp));
                const float q1 = __expf(fminf(Lt - Ll, kMaxUp));
                st_tile(At, 128, 2 * GC + t, c, qf * q1);
                st_tile(At, 128, 3 * GC + t, c, kp * ks1);
                ks1 = q1;
            } else {
                st_tile(At, 128, 2 * GC + t, c, 0.f);
                st_tile(At, 128, 3 * GC + t, c, 0.f);
            }
            kdec[t] = kp * eprev;
            const float eL = __expf(Lt);
            eprev = eL;
            qrow[t * DK + c] = __float2bfloat16_rn(qf * eL);
            const float fK = t < GH ? fk * fh : fk;  // e^{L_last - L_t}
            krow[t * DK + c] = __float2bfloat16_rn(kf * fK);
            krow[(GC + t) * DK + c] = __float2bfloat16_rn(-bf * fK);
        }
        Dj = __expf(Ll);
    } else if (tid >= 128 && tid < 128 + DK) {
        // ---- the previous block's Kt = [Kw'; -B'] and D (block j-1 is full)
        const int c = tid - 128;
        if (j == 0) {
#pragma unroll 4
            for (int s = 0; s < 2 * GC; ++s) st_tile(Kt, 64, s, c, 0.f);
            Dp[c] = 1.f;
        } else {
            const size_t g0 = (bh * T + t0 - GC) * DK + c;
            float Lp[GC];
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < GC; ++s) {
                acc += __logf(w[g0 + (size_t)s * DK]);
                Lp[s] = acc;
            }
#pragma unroll
            for (int s = 0; s < GC; ++s) {
                const size_t g = g0 + (size_t)s * DK;
                const float f = __expf(acc - Lp[s]);
                st_tile(Kt, 64, s, c, __bfloat162float(kw[g]) * f);
                st_tile(Kt, 64, GC + s, c, -ar[g] * kappa[g] * f);
            }
            Dp[c] = __expf(acc);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- S: the four score matrices, TMEM cols 0..63
    if (tid == 0) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(At), 128, 0, ks), tile_desc(smem_u32(Bt), 64, 0, ks),
                     id, ks > 0);
        mma_commit(&bar[0]);
    }
    bool ok = __syncthreads_and(mbar_wait(&bar[0], 0) ? 1 : 0) != 0;
    tc_fence_after();
    if (ok) {
        // warp w: row quarter w & 3 (queries / removal keys, first / second
        // reference), columns of the kw (w < 4) or b (w >= 4) keys of that
        // reference's half; lane = token t
        const int qr = warp & 3, h = warp >> 2, t = lane;
        const int s0 = qr >= 2 ? GH : 0;
        float x[16];
        tmem_ld16(tmem + ((uint32_t)(32 * qr) << 16) + (uint32_t)(32 * h + s0), x);
        tmem_ld_wait();
        const bool keyrow = qr & 1;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int s = s0 + e;
            if (keyrow ? s >= t : s > t) x[e] = 0.f;
        }
        if (keyrow) {  // Bk (kw keys) or A (b keys), fp32 for the solve
            float *M = h ? Am : Bk;
#pragma unroll
            for (int e = 0; e < 16; ++e) M[t * SP + s0 + e] = x[e];
        } else {       // stage j+1's P row t: [Qk | -Qb]
            if (h) {
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] = -x[e];
            }
#pragma unroll
            for (int i8 = 0; i8 < 2; ++i8)
                *reinterpret_cast<uint4 *>(rec_next + R::TZP +
                                           sw128_offset(128 + t, 32 * h + s0 + 8 * i8, 192)) =
                    pack8(x + 8 * i8);
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- (I + A) [Wg | Tb] = [Kdec | Bk] by forward substitution, one column
    //      per thread; Wg goes to the A tile (rows 0..31) for Z and, times
    //      D_{j-1}, to the record's W rows 32..63.  The other threads write the
    //      record's constant parts.
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
                const float4 a4 = *reinterpret_cast<const float4 *>(Am + t * SP + s4);
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
            const float d = Dp[tid];
#pragma unroll
            for (int t = 0; t < GC; ++t) {
                st_tile(At, 128, t, tid, x[t]);
                *reinterpret_cast<bf16 *>(rec + R::WT + sw128_offset(GC + t, tid, 64)) =
                    __float2bfloat16_rn(x[t] * d);
            }
        }
    } else {
        const int i0 = tid - (DK + GC), ni = GNT - (DK + GC);
        constexpr int WCH = DK / 8;
        const uint4 z4 = make_uint4(0, 0, 0, 0);
        for (int i = i0; i < GC * WCH; i += ni) {  // W rows 0..31 (the value rows of Ut)
            const int r = i / WCH, c8 = (i % WCH) * 8;
            *reinterpret_cast<uint4 *>(rec + R::WT + sw128_offset(r, c8, 64)) = z4;
            reinterpret_cast<uint4 *>(qrow + (GC + r) * DK)[c8 / 8] = z4;  // q rows 32..63
        }
        for (int i = i0; i < 3 * GC * 8; i += ni) {  // T rows 0..31 = [I | 0], rows 64..95 = 0,
            const int r = i >> 3, c8 = (i & 7) * 8;   // stage j+1's P rows 160..191 = 0
            if (r < GC) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = c8 + e == r ? 1.f : 0.f;
                *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(r, c8, 192)) = pack8(x);
            } else if (r < 2 * GC) {
                *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(GC + r, c8, 192)) = z4;
            } else {
                *reinterpret_cast<uint4 *>(rec_next + R::TZP + sw128_offset(96 + r, c8, 192)) = z4;
            }
        }
        if (j == nblk - 1) {
            // the closing stage reads (unused) W, T and Z rows
            for (int i = i0; i < (R::TZP + 128 * 128) / 16; i += ni)
                reinterpret_cast<uint4 *>(rec_next)[i] = z4;
        }
    }
    float *vec = reinterpret_cast<float *>(rec + R::VEC);
    vec[tid] = tid < DK ? Dp[tid] : 0.f;  // g_C' per key channel (GNT = 256 floats)
    if (j == nblk - 1) {
        float *vn = reinterpret_cast<float *>(rec_next + R::VEC);
        vn[tid] = tid < DK ? Dj : 0.f;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- Z = Wg Kt_{j-1}^T, TMEM cols 64..127; meanwhile the T rows [Tb | 0]
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem + 64, tile_desc(smem_u32(At), 128, 0, ks),
                     tile_desc(smem_u32(Kt), 64, 0, ks), id, ks > 0);
        mma_commit(&bar[1]);
    }
    {
        const int r = tid >> 3, c8 = (tid & 7) * 8;  // 32 rows x 8 chunks
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = c8 + e < GC ? Bk[r * SP + c8 + e] : 0.f;
        *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(GC + r, c8, 192)) = pack8(x);
    }
    ok = __syncthreads_and((ok && mbar_wait(&bar[1], 0)) ? 1 : 0) != 0;
    tc_fence_after();
    if (ok && (warp & 3) == 0) {  // warps 0 and 4: Z rows t = lane, columns 32 h ..
        const int h = warp >> 2, t = lane;
        float z[32];
        tmem_ld32(tmem + 64 + 32 * h, z);
        tmem_ld_wait();
#pragma unroll
        for (int i8 = 0; i8 < 4; ++i8)
            *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(3 * GC + t, 32 * h + 8 * i8, 192)) =
                pack8(z + 8 * i8);
    }
    if (!ok && tid == 0) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

template <int DK>
cudaError_t launch_gd_dk(const void *q, const void *kw, const void *v, const float *w,
                         const float *kappa, const float *a, const float *S0, void *o,
                         float *S_T, int B, int H, int T, int dv, void *ws, cudaStream_t stream,
                         int slot) {
    const int nblk = (T + GC - 1) / GC;
    auto prep = chunk_prep_gd_kernel<DK>;
    auto scan = chunk_scan_kernel<DK, true, true, false, true>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), GdPrep<DK>::ALLOC, slot);
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
    prep<<<dim3(nblk, H, B), GNT, GdPrep<DK>::ALLOC, stream>>>(
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
