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
// swizzled K-major layout of the tensor cores (1024-byte aligned), Kdec and
// the partial log-decay sums in fp32, the barrier and the TMEM slot.  After
// the score product the query tile hosts the fp32 matrices of the solve.
template <int DK>
struct GdPrep {
    static constexpr int KB = (DK + 63) / 64;       // 64-column blocks of a tile row
    static constexpr int TPC = GNT / DK;            // threads per key channel
    static constexpr int TPT = GC / TPC;            // tokens per thread
    static constexpr int SP = GC + 4;               // fp32 row of a 32 x 32 matrix
    static constexpr int AT = 0;                    // [128][DK]: query / removal-key rows
    static constexpr int BT = AT + KB * 128 * 128;  // [64][DK]: the key rows [kw; b]
    static constexpr int KD = BT + KB * 64 * 128;   // fp32 [32][DK]: Kdec
    static constexpr int PS = KD + GC * DK * 4;     // fp32 [2][TPC][DK]: partial sums of log w
    static constexpr int BAR = PS + 2 * GNT * 4;
    static constexpr int BYTES = BAR + 24;          // two mbarriers and the TMEM slot
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(2 * GC * SP * 4 <= KB * 128 * 128, "A and Bk must fit over the query tile");
    static_assert(2 * GC * DK * 4 <= KB * 128 * 128, "two blocks of decays must fit over the query tile");
    static_assert(TPT * TPC == GC && TPC * DK == GNT && (GH % TPT) == 0, "token split");
};

// Workspace layout of the bf16 path, per (batch, head): nblk + 1 records,
// then for all heads the per-stage q and k operands ([nblk * 64][DK] bf16
// each) and Wg ([nblk] tiles of 32 rows x DK, 128-byte swizzled like the rows
// 0..31 of a 64-row operand tile).
template <int DK>
struct GdWs {
    static constexpr size_t WG_TILE = (size_t)((DK + 63) / 64) * 32 * 128;
    static size_t rec_bytes(size_t BH, int nblk) { return BH * (nblk + 1) * (size_t)Rec<DK>::BYTES; }
    static size_t qk_elems(size_t BH, int nblk) { return BH * (size_t)nblk * 2 * GC * DK; }
    static size_t bytes(size_t BH, int nblk) {
        return rec_bytes(BH, nblk) + 2 * qk_elems(BH, nblk) * 2 + BH * nblk * WG_TILE;
    }
};

__device__ __forceinline__ void st_tile(uint8_t *tile, int rows, int r, int c, float x) {
    *reinterpret_cast<bf16 *>(tile + sw128_offset(r, c, rows)) = bf16_rn(x);
}

// One CTA per (block, head, batch).  q, kw [B*H][T][DK] bf16; w, kappa, a
// [B*H][T][DK] fp32.  Writes record j (all but its Z rows), stage j+1's P
// rows, the stage's q and k operands and Wg_j.
//
// Thread (part, c) takes key channel c for tokens part*TPT .. part*TPT+TPT-1;
// the log decays are summed per part and combined through shared memory.
// One M = 128, N = 64 tcgen05 product gives the four score matrices for both
// references:
//   [Q e^{L-L_15}; K e^{L_{t-1}-L_15}; Q e^{L-L_31}; K e^{L_{t-1}-L_31}] [kw e^{L_r-L}; b e^{L_r-L}]^T
// (rows 64..127 only for queries of the second half; keys 0..15 from the
// first reference, 16..31 from the second), then the solve
// (I + A)[Wg | Tb] = [Kdec | Bk] runs on the CUDA cores, one column per thread.
template <int DK>
__global__ void __launch_bounds__(GNT, 3)  // 3 CTAs per SM: 80 registers, 67 KB of shared memory
chunk_prep_gd_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ kw,
                     const float *__restrict__ w, const float *__restrict__ kappa,
                     const float *__restrict__ ar, uint8_t *__restrict__ ws, bf16 *__restrict__ qo,
                     bf16 *__restrict__ ko, uint8_t *__restrict__ wgo, int H, int T, int nblk) {
    using G = GdPrep<DK>;
    using R = Rec<DK>;
    constexpr int SP = G::SP, TPC = G::TPC, TPT = G::TPT;
    extern __shared__ uint8_t gd_raw[];
    uint8_t *sm = align1024(gd_raw);
    uint8_t *At = sm + G::AT, *Bt = sm + G::BT;
    float *Kd = reinterpret_cast<float *>(sm + G::KD);
    float *Ps = reinterpret_cast<float *>(sm + G::PS);  // [0]: this block, [1]: the previous one
    float *Am = reinterpret_cast<float *>(sm + G::AT), *Bk = Am + GC * SP;  // after the product
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + G::BAR);  // score product, decays
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G::BAR + 16);
    // decays of the previous block (rows 0..GC-1) and of this one (rows GC..),
    // fp32 [2 GC][DK], in the query tile until the tokens' operands replace them
    const float *Ws = reinterpret_cast<const float *>(sm + G::AT);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid % DK, part = tid / DK, tb = part * TPT;
    const int j = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = j * GC, n = min(GC, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + j) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    bf16 *qrow = qo + (bh * nblk + j) * (size_t)(2 * GC) * DK;
    bf16 *krow = ko + (bh * nblk + j) * (size_t)(2 * GC) * DK;
    uint8_t *wg = wgo + (bh * nblk + j) * GdWs<DK>::WG_TILE;

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        // the decays of this block and the previous one by one bulk copy
        const int prow = j > 0 ? GC : 0;  // previous-block rows copied
        const uint32_t wbytes = (uint32_t)((prow + n) * DK * 4);
        mbar_expect_tx(&bar[1], wbytes);
        bulk_g2s(sm + G::AT + (size_t)(GC - prow) * DK * 4, w + (bh * T + t0 - prow) * DK, wbytes,
                 &bar[1]);
        // the block's rows of q, kw, kappa and a, read after the decays: to L2 now
        const size_t r0 = (bh * T + t0) * DK;
        prefetch_l2(q + r0, (uint32_t)(n * DK * 2));
        prefetch_l2(kw + r0, (uint32_t)(n * DK * 2));
        prefetch_l2(kappa + r0, (uint32_t)(n * DK * 4));
        prefetch_l2(ar + r0, (uint32_t)(n * DK * 4));
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    // the barriers are initialised before any thread waits on them
    __syncthreads();
    const bool wok = mbar_wait(&bar[1], 0);
    // ---- log decays: this block's prefix within the part, the previous
    //      block's total (its D)
    const size_t g0 = (bh * T + t0 + tb) * DK + c;
    float lw[TPT];
    {
        float acc = 0.f, pacc = 0.f;
        const float *wc = Ws + (GC + tb) * DK + c, *wp = Ws + tb * DK + c;
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            acc += (wok && tb + i < n) ? __logf(wc[i * DK]) : 0.f;
            lw[i] = acc;
        }
        if (j > 0 && wok) {
#pragma unroll
            for (int i = 0; i < TPT; ++i) pacc += __logf(wp[i * DK]);
        }
        Ps[part * DK + c] = acc;
        Ps[GNT + part * DK + c] = pacc;
    }
    __syncthreads();
    float off = 0.f, Lh = 0.f, Ll = 0.f, Lp = 0.f;
#pragma unroll
    for (int p = 0; p < TPC; ++p) {
        const float x = Ps[p * DK + c];
        off += p < part ? x : 0.f;
        Lh += p < TPC / 2 ? x : 0.f;
        Ll += x;
        Lp += Ps[GNT + p * DK + c];
    }
    const float Dp = __expf(Lp);  // D_{j-1} (1 for the first block)

    // ---- this thread's tokens: scaled operands, Kdec, the stage's q and k rows
    {
        float Lm = off;  // L_{t-1}
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            const int t = tb + i;
            const bool ok = t < n;
            const size_t g = g0 + (size_t)i * DK;
            const float qf = ok ? __bfloat162float(q[g]) : 0.f;
            const float kf = ok ? __bfloat162float(kw[g]) : 0.f;
            const float kp = ok ? kappa[g] : 0.f;
            const float bf = ok ? ar[g] * kp : 0.f;
            const float Lt = off + lw[i];
            const float fk = __expf((t < GH ? Lh : Ll) - Lt);  // key factor, at most 1
            st_tile(Bt, 64, t, c, kf * fk);
            st_tile(Bt, 64, GC + t, c, bf * fk);
            st_tile(At, 128, t, c, qf * __expf(fminf(Lt - Lh, kMaxUp)));
            st_tile(At, 128, GC + t, c, kp * __expf(fminf(Lm - Lh, kMaxUp)));
            const bool second = t >= GH;
            st_tile(At, 128, 2 * GC + t, c, second ? qf * __expf(fminf(Lt - Ll, kMaxUp)) : 0.f);
            st_tile(At, 128, 3 * GC + t, c, second ? kp * __expf(fminf(Lm - Ll, kMaxUp)) : 0.f);
            Kd[t * DK + c] = kp * __expf(Lm);
            qrow[t * DK + c] = bf16_rn(qf * __expf(Lt));
            const float fK = __expf(Ll - Lt);  // e^{L_last - L_t}
            krow[t * DK + c] = bf16_rn(kf * fK);
            krow[(GC + t) * DK + c] = bf16_rn(-bf * fK);
            Lm = Lt;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- the four score matrices, TMEM cols 0..63
    if (tid == 0) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(At), 128, 0, ks), tile_desc(smem_u32(Bt), 64, 0, ks),
                     id, ks > 0);
        mma_commit(&bar[0]);
    }
    const bool ok = __syncthreads_and(mbar_wait(&bar[0], 0) ? 1 : 0) != 0;
    tc_fence_after();
    if (ok) {
        // warp w: row quarter w & 3 (queries / removal keys, first / second
        // reference), columns of the kw (w < 4) or b (w >= 4) keys of that
        // reference's half; lane = token t
        const int qr = warp & 3, h = warp >> 2, t = lane;
        const int s0 = qr >= 2 ? GH : 0;
        float x[16];
        tmem_ld16(tmem + ((uint32_t)(32 * qr) << 16) + (uint32_t)(32 * h + s0), x);
        tmem_ld_wait(x);
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
    //      per thread: Wg to the workspace (for the Z rows) and, times D_{j-1},
    //      to the record's W rows 32..63.  The other threads write the
    //      record's constant parts.
    if (tid < DK + GC) {
        const bool tcol = tid >= DK;
        float x[GC];
#pragma unroll
        for (int t = 0; t < GC; ++t) x[t] = tcol ? Bk[t * SP + (tid - DK)] : Kd[t * DK + tid];
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
            // D_{j-1} of this column: its own thread's Dp (tid < DK: part 0, c = tid)
#pragma unroll
            for (int t = 0; t < GC; ++t) {
                *reinterpret_cast<bf16 *>(wg + sw128_offset(t, tid, 32)) = bf16_rn(x[t]);
                *reinterpret_cast<bf16 *>(rec + R::WT + sw128_offset(GC + t, tid, 64)) =
                    bf16_rn(x[t] * Dp);
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
        if (j == 0) {  // stage 0 has no Z rows (no previous block)
            for (int i = i0; i < GC * 8; i += ni)
                *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(3 * GC + (i >> 3), (i & 7) * 8, 192)) = z4;
        }
        if (j == nblk - 1) {
            // the closing stage reads (unused) W, T and Z rows
            for (int i = i0; i < (R::TZP + 128 * 128) / 16; i += ni)
                reinterpret_cast<uint4 *>(rec_next)[i] = z4;
        }
    }
    float *vec = reinterpret_cast<float *>(rec + R::VEC);
    if (part == 0) vec[c] = Dp;  // g_C' per key channel
    if (tid >= DK) vec[tid] = 0.f;
    if (j == nblk - 1) {
        float *vn = reinterpret_cast<float *>(rec_next + R::VEC);
        if (part == 0) vn[c] = __expf(Ll);
        if (tid >= DK) vn[tid] = 0.f;
    }
    __syncthreads();
    {   // T rows 32..63 = [Tb | 0]
        const int r = tid >> 3, c8 = (tid & 7) * 8;  // 32 rows x 8 chunks
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = c8 + e < GC ? Bk[r * SP + c8 + e] : 0.f;
        *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(GC + r, c8, 192)) = pack8(x);
    }
    if (!(ok && wok) && tid == 0) atomicExch(&g_tc_error, 1);
    // never leave with the decay copy in flight
    if (!wok && tid == 0) mbar_wait(&bar[1], 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// The Z rows of stage j >= 1: Wg_j Kt_{j-1}^T (32 x 64, K = DK) -> record j's
// T/Z tile rows 96..127.  Wg_j comes from the workspace by bulk copy, Kt_{j-1}
// (the previous stage's k operand) by TMA; one M = 64 tcgen05 product.
template <int DK>
struct GdZ {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int AT = 0;                  // [64][DK]: Wg rows 0..31, zero rows 32..63
    static constexpr int BT = AT + KB * 64 * 128; // [64][DK]: Kt_{j-1}
    static constexpr int BAR = BT + KB * 64 * 128;
    static constexpr int BYTES = BAR + 32;
    static constexpr int ALLOC = BYTES + 1024;
};
constexpr int kZThreads = 128;

template <int DK>
__global__ void __launch_bounds__(kZThreads)
chunk_prep_gd_z_kernel(uint8_t *__restrict__ ws, const uint8_t *__restrict__ wgo, int H, int nblk,
                       const __grid_constant__ CUtensorMap tmk) {
    using G = GdZ<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t gz_raw[];
    uint8_t *sm = align1024(gz_raw);
    uint8_t *At = sm + G::AT, *Bt = sm + G::BT;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + G::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G::BAR + 16);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x + 1;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    uint8_t *rec = ws + (bh * (nblk + 1) + j) * (size_t)R::BYTES;
    const uint8_t *wg = wgo + (bh * nblk + j) * GdWs<DK>::WG_TILE;

    for (int i = tid; i < G::KB * 256; i += kZThreads) {  // rows 32..63 of each A block
        const int kb = i >> 8, o = (i & 255) * 16;
        *reinterpret_cast<uint4 *>(At + kb * 8192 + 4096 + o) = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        mbar_expect_tx(&bar[0], (uint32_t)G::KB * (4096u + 8192u));
#pragma unroll
        for (int kb = 0; kb < G::KB; ++kb) {
            bulk_g2s(At + kb * 8192, wg + kb * 4096, 4096, &bar[0]);
            tma_load_3d(Bt + kb * 8192, &tmk, kb * 64, (j - 1) * 2 * GC, (int)bh, &bar[0]);
        }
    }
    bool ok = mbar_wait(&bar[0], 0);
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t id = idesc_bf16_f32(64, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(At), 64, 0, ks), tile_desc(smem_u32(Bt), 64, 0, ks), id,
                     ks > 0);
        mma_commit(&bar[1]);
    }
    ok = __syncthreads_and((ok && mbar_wait(&bar[1], 0)) ? 1 : 0) != 0;
    tc_fence_after();
    // M = 64: rows 16w .. 16w + 15 in lanes 32w .. 32w + 15; rows 0..31 are warps 0 and 1
    if (ok && warp < 2) {
        const int r = 16 * warp + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float z[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(32 * half), z);
            tmem_ld_wait(z);
            if (lane < 16) {
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8)
                    *reinterpret_cast<uint4 *>(rec + R::TZP +
                                               sw128_offset(3 * GC + r, 32 * half + 8 * i8, 192)) =
                        pack8(z + 8 * i8);
            }
        }
    }
    if (!ok && tid == 0) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

template <int DK>
cudaError_t launch_gd_dk(const void *q, const void *kw, const void *v, const float *w,
                         const float *kappa, const float *a, const float *S0, void *o,
                         float *S_T, int B, int H, int T, int dv, void *ws, cudaStream_t stream,
                         int slot) {
    using W = GdWs<DK>;
    const int nblk = (T + GC - 1) / GC;
    const size_t BH = (size_t)B * H;
    auto prep = chunk_prep_gd_kernel<DK>;
    auto zk = chunk_prep_gd_z_kernel<DK>;
    auto scan = chunk_scan_kernel<DK, true, true, false, true>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), GdPrep<DK>::ALLOC, slot);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC, slot + 1);
    if (e != cudaSuccess) return e;
    uint8_t *recs = static_cast<uint8_t *>(ws);
    bf16 *qo = reinterpret_cast<bf16 *>(recs + W::rec_bytes(BH, nblk));
    bf16 *ko = qo + W::qk_elems(BH, nblk);
    uint8_t *wgo = reinterpret_cast<uint8_t *>(ko + W::qk_elems(BH, nblk));
    CUtensorMap tmq, tmk, tmv;
    if ((e = make_rows_map(&tmq, qo, DK, nblk * 2 * GC, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmk, ko, DK, nblk * 2 * GC, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmv, v, dv, T, B * H)) != cudaSuccess) return e;
    prep<<<dim3(nblk, H, B), GNT, GdPrep<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(kw), w, kappa, a, recs, qo, ko, wgo,
        H, T, nblk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nblk > 1) {
        zk<<<dim3(nblk - 1, H, B), kZThreads, GdZ<DK>::ALLOC, stream>>>(recs, wgo, H, nblk, tmk);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    scan<<<dim3(dv / DVS, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
        recs, S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk, qo, ko,
        static_cast<const bf16 *>(v), tmq, tmk, tmv, nullptr, 0.f, 0);
    return cudaGetLastError();
}

}  // namespace

size_t gen_delta_tc_workspace_bytes(int B, int H, int T, int dk) {
    const int nblk = (T + GC - 1) / GC;
    const size_t BH = (size_t)B * H;
    return dk == 32 ? GdWs<32>::bytes(BH, nblk)
           : dk == 64 ? GdWs<64>::bytes(BH, nblk)
                      : GdWs<128>::bytes(BH, nblk);
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
