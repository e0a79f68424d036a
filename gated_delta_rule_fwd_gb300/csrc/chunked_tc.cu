// Chunked forward on the tensor cores (tcgen05 + TMEM), bf16 operands with
// fp32 accumulation and an fp32 state.
//
// Chunkwise form (page "Le architetture lineari: RetNet, RWKV, xLSTM",
// section "RetNet: la retention e le sue tre forme"): blocks of C = 64
// tokens, only the end-of-block state handed to the next block.  Inside a
// block, with G_r = sum_{i<=r} ln alpha_i (gate products, computable for all
// steps at once -- page "Scrivere meglio nella memoria: gate e delta rule",
// section "Correggere: la delta rule"), g_r = e^{G_r}, kd_i = e^{G_C - G_i}:
//
//   P   = (Q K^T) (.) M,            M_ri = e^{G_r - G_i} for i <= r     (scores)
//   A   = strict_lower(diag(beta) (K K^T) (.) M)                       (delta couplings)
//   T   = (I + A)^-1                (unit lower triangular; the WY / UT step)
//   W   = T diag(beta g) K,         Ut = T diag(beta) V
//   U   = Ut - W S^T                pseudo-values (u_r of the WY representation)
//   O   = diag(g) Q S^T + P U
//   S  <- g_C S + U^T diag(kd) K
// and without the delta term U = V (T unused).  The derivation: the gated
// recurrence unrolled inside a block gives u_r = beta_r (v_r - g_r S k_r -
// sum_{i<r} e^{G_r - G_i} (k_i.k_r) u_i), a unit-lower-triangular system.
//
// Work split.  One CTA of 128 threads per (32 value channels, head, batch);
// rows of S evolve independently, so value-channel slices never exchange
// data.  Every product runs on the tensor cores as an M = 128 tcgen05.mma
// with both operands in shared memory (K-major, 128-byte swizzle) and the
// fp32 accumulator in TMEM.  Two 64-row operands are stacked to fill M:
//   E1  [Q; K] K^T           -> [Q K^T ; K K^T]            (TMEM R1, 64 cols)
//   E3  [T; P] (beta g K)^T  -> [W ; -]                    (R2, dk cols)
//       [T; P] (beta V)^T    -> [Ut ; P beta V]            (R3, 32 cols)
//   S1  [-W; g Q] S^T   +=   -> [U ; P beta V + g Q S^T]   (R3)
//   S3  (kd K)^T U      =    -> Delta S^T                  (R4, 32 cols)
//       [T; P] (U - beta V)^T += -> rows 64..127 = O        (R3)
// The fp32 master copy of the state slice lives in registers (thread j owns
// column j); a bf16 copy in shared memory feeds S1.  T is formed in fp32 on
// the CUDA cores by blocked forward substitution (16 x 16 diagonal blocks).
// Inputs of the next block are prefetched with cp.async while the current
// block computes; a final short block is zero-filled (alpha treated as 1,
// beta as 0), which leaves the real tokens' results unchanged.
#include "lr_internal.cuh"
#include "tc_common.cuh"

namespace lr {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int C = 64;      // tokens per block
constexpr int DVS = 32;    // value channels per CTA
constexpr int NT = 128;    // threads per CTA (one warpgroup)
constexpr int AP = C + 1;  // padded fp32 row of A and T

__device__ int g_tc_error = 0;  // set to 1 when a bounded wait gives up

template <int DK>
struct TcLayout {
    static constexpr int KB = (DK + 63) / 64;           // 64-wide K blocks of a dk-long row
    static constexpr int QK = 0;                         // 2 x [128 rows][DK]   (Q rows, K rows)
    static constexpr int QK_BYTES = 128 * 128 * KB;
    static constexpr int WQ = QK + 2 * QK_BYTES;         // [128][DK]: -W rows, g*Q rows
    static constexpr int TP = WQ + QK_BYTES;             // [128][64]: T rows, P rows
    static constexpr int KBT = TP + 16384;               // [DK][64]:  (beta g K)^T
    static constexpr int KBT_BYTES = (DK < 8 ? 8 : DK) * 128;
    static constexpr int KTT = KBT + ((KBT_BYTES + 1023) / 1024) * 1024;  // [128][64]: (kd K)^T
    static constexpr int VBT = KTT + 16384;              // [32][64]:  (beta V)^T (V^T w/o delta)
    static constexpr int UB = VBT + 4096;                // [32][64]:  U^T
    static constexpr int XB = UB + 4096;                 // [32][64]:  (U - beta V)^T
    static constexpr int SB = XB + 4096;                 // [32][DK]:  bf16 state slice
    static constexpr int VRAW = SB + 32 * 128 * KB;      // 2 x [64][32] bf16 raw V slice
    static constexpr int AB = VRAW + 2 * 4096;           // 2 x {alpha[64], beta[64]} fp32
    static constexpr int AMAT = AB + 2 * 512;            // fp32 [64][65]
    static constexpr int TMAT = AMAT + C * AP * 4;       // fp32 [64][65]
    static constexpr int XTMP = TMAT + C * AP * 4;       // fp32 [16][49]
    static constexpr int VEC = XTMP + 16 * 49 * 4;      // fp32 G, g, kd, bg, b   [5][64]
    static constexpr int BAR = VEC + 5 * 64 * 4;         // mbarrier + TMEM base
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;           // slack for 1024-byte alignment
};

// TMEM columns
constexpr uint32_t kR1 = 0, kR2 = 64, kR3 = 192, kR4 = 224, kTmemCols = 256;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}
__device__ __forceinline__ float bf16_at(const uint8_t *tile, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const bf16 *>(tile + off));
}
__device__ __forceinline__ void st_bf16(uint8_t *tile, uint32_t off, float x) {
    *reinterpret_cast<bf16 *>(tile + off) = __float2bfloat16_rn(x);
}

// Stage block `t0` of (bh, slice) into buffer `buf` with cp.async (zero-filled
// past the end of the sequence).
template <int DK>
__device__ __forceinline__ void prefetch_block(uint8_t *sm, int buf, const bf16 *q, const bf16 *k,
                                               const bf16 *v, const float *alpha,
                                               const float *beta, size_t bh, int T, int t0,
                                               int dv, int c0, int tid) {
    using L = TcLayout<DK>;
    uint8_t *qk = sm + L::QK + buf * L::QK_BYTES;
    constexpr int CPR = DK / 8;  // 16-byte chunks per row
    for (int idx = tid; idx < 2 * C * CPR; idx += NT) {
        const int which = idx / (C * CPR);  // 0: q, 1: k
        const int rem = idx % (C * CPR);
        const int r = rem / CPR, ch = rem % CPR;
        const bool ok = t0 + r < T;
        const bf16 *src = (which ? k : q) + ((bh * T + (ok ? t0 + r : 0)) * DK + ch * 8);
        cp_async16(smem_u32(qk + sw128_offset(which * 64 + r, ch * 8, 128)), src, ok);
    }
    uint8_t *vr = sm + L::VRAW + buf * 4096;
    for (int idx = tid; idx < C * (DVS / 8); idx += NT) {
        const int r = idx / (DVS / 8), ch = idx % (DVS / 8);
        const bool ok = t0 + r < T;
        const bf16 *src = v + ((bh * T + (ok ? t0 + r : 0)) * dv + c0 + ch * 8);
        cp_async16(smem_u32(vr + (r * DVS + ch * 8) * 2), src, ok);
    }
    float *ab = reinterpret_cast<float *>(sm + L::AB + buf * 512);
    if (tid < C) {
        const bool ok = t0 + tid < T;
        const size_t gi = bh * T + (ok ? t0 + tid : 0);
        if (alpha) cp_async4(smem_u32(ab + tid), alpha + gi, ok);
        if (beta) cp_async4(smem_u32(ab + 64 + tid), beta + gi, ok);
    }
    cp_async_commit();
}

template <int DK, bool ALPHA, bool DELTA>
__global__ void __launch_bounds__(NT, 1)
chunk_tc_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                const bf16 *__restrict__ v, const float *__restrict__ alpha,
                const float *__restrict__ beta, const float *__restrict__ S0,
                bf16 *__restrict__ o, float *__restrict__ ST, int H, int T, int dv) {
    using L = TcLayout<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;

    uint8_t *WQ = sm + L::WQ, *TP = sm + L::TP, *KBT = sm + L::KBT, *KTT = sm + L::KTT;
    uint8_t *VBT = sm + L::VBT, *UB = sm + L::UB, *XB = sm + L::XB, *SB = sm + L::SB;
    float *Am = reinterpret_cast<float *>(sm + L::AMAT);
    float *Tm = reinterpret_cast<float *>(sm + L::TMAT);
    float *Xt = reinterpret_cast<float *>(sm + L::XTMP);
    float *Gv = reinterpret_cast<float *>(sm + L::VEC);
    float *gv = Gv + 64, *kdv = Gv + 128, *bgv = Gv + 192, *bv = Gv + 256;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 8);

    // ---- one-time set-up: zero the operand tiles whose padding must read as 0
    for (int i = tid; i < (L::VRAW - L::WQ) / 16; i += NT)
        reinterpret_cast<uint4 *>(sm + L::WQ)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }

    __syncthreads();  // zeroing done before any tile is written

    // fp32 master copy of the state slice: thread j owns S[c0 + c][j], c < 32
    float Sr[DVS];
#pragma unroll
    for (int c = 0; c < DVS; ++c)
        Sr[c] = (S0 && tid < DK) ? S0[(bh * dv + c0 + c) * DK + tid] : 0.f;
    if (tid < DK) {
#pragma unroll
        for (int c = 0; c < DVS; ++c) st_bf16(SB, sw128_offset(c, tid, 32), Sr[c]);
    }

    if (T > 0) prefetch_block<DK>(sm, 0, q, k, v, alpha, beta, bh, T, 0, dv, c0, tid);

    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    uint32_t phase = 0;
    bool ok = true;

    // Every thread waits; the give-up decision is made block-wide so that all
    // threads leave the loop together.
    auto mma_wait = [&]() {
        const bool mine = mbar_wait(bar, phase & 1);
        ++phase;
        ok = __syncthreads_and(mine ? 1 : 0) != 0;
        tc_fence_after();
    };

    const int nblocks = (T + C - 1) / C;
    for (int blk = 0; blk < nblocks && ok; ++blk) {
        const int t0 = blk * C;
        const int n = min(C, T - t0);
        const int buf = blk & 1;
        uint8_t *QK = sm + L::QK + buf * L::QK_BYTES;
        const bf16 *Vraw = reinterpret_cast<const bf16 *>(sm + L::VRAW + buf * 4096);
        const float *ab = reinterpret_cast<const float *>(sm + L::AB + buf * 512);

        cp_async_wait_all();
        __syncthreads();
        if (blk + 1 < nblocks)
            prefetch_block<DK>(sm, buf ^ 1, q, k, v, alpha, beta, bh, T, t0 + C, dv, c0, tid);

        // ---- gate products in log space: G = cumsum(ln alpha) over the block
        if (warp == 0) {
            float x0 = 0.f, x1 = 0.f;
            if (ALPHA) {
                x0 = (2 * lane < n) ? logf(ab[2 * lane]) : 0.f;
                x1 = (2 * lane + 1 < n) ? logf(ab[2 * lane + 1]) : 0.f;
            }
            const float pair = x0 + x1;
            float incl = pair;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += y;
            }
            const float e = incl - pair;
            Gv[2 * lane] = e + x0;
            Gv[2 * lane + 1] = e + pair;
        }
        __syncthreads();
        if (tid < C) {
            const float G = Gv[tid];
            const float b = (DELTA && tid < n) ? ab[64 + tid] : 0.f;
            const float g = ALPHA ? expf(G) : 1.f;
            gv[tid] = g;
            kdv[tid] = ALPHA ? expf(Gv[C - 1] - G) : 1.f;
            bgv[tid] = b * g;
            bv[tid] = b;
        }
        __syncthreads();

        // ---- operand tiles that need no MMA result
        // g * Q -> rows 64..127 of WQ (same swizzle phase as the Q rows of QK)
        for (int idx = tid; idx < C * (DK / 8); idx += NT) {
            const int r = idx / (DK / 8), ch = idx % (DK / 8);
            const uint4 raw = *reinterpret_cast<const uint4 *>(QK + sw128_offset(r, ch * 8, 128));
            const float g = gv[r];
            const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
            uint4 outv;
            outv.x = pack_bf16(g * __bfloat162float(e[0]), g * __bfloat162float(e[1]));
            outv.y = pack_bf16(g * __bfloat162float(e[2]), g * __bfloat162float(e[3]));
            outv.z = pack_bf16(g * __bfloat162float(e[4]), g * __bfloat162float(e[5]));
            outv.w = pack_bf16(g * __bfloat162float(e[6]), g * __bfloat162float(e[7]));
            *reinterpret_cast<uint4 *>(WQ + sw128_offset(64 + r, ch * 8, 128)) = outv;
        }
        // (kd K)^T and, with delta, (beta g K)^T: thread j builds row j
        if (tid < DK) {
            const int j = tid;
#pragma unroll
            for (int i8 = 0; i8 < C / 8; ++i8) {
                float kv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    kv[e] = bf16_at(QK, sw128_offset(64 + i8 * 8 + e, j, 128));
                uint4 a;
                a.x = pack_bf16(kdv[i8 * 8 + 0] * kv[0], kdv[i8 * 8 + 1] * kv[1]);
                a.y = pack_bf16(kdv[i8 * 8 + 2] * kv[2], kdv[i8 * 8 + 3] * kv[3]);
                a.z = pack_bf16(kdv[i8 * 8 + 4] * kv[4], kdv[i8 * 8 + 5] * kv[5]);
                a.w = pack_bf16(kdv[i8 * 8 + 6] * kv[6], kdv[i8 * 8 + 7] * kv[7]);
                *reinterpret_cast<uint4 *>(KTT + sw128_offset(j, i8 * 8, 128)) = a;
                if (DELTA) {
                    uint4 b;
                    b.x = pack_bf16(bgv[i8 * 8 + 0] * kv[0], bgv[i8 * 8 + 1] * kv[1]);
                    b.y = pack_bf16(bgv[i8 * 8 + 2] * kv[2], bgv[i8 * 8 + 3] * kv[3]);
                    b.z = pack_bf16(bgv[i8 * 8 + 4] * kv[4], bgv[i8 * 8 + 5] * kv[5]);
                    b.w = pack_bf16(bgv[i8 * 8 + 6] * kv[6], bgv[i8 * 8 + 7] * kv[7]);
                    *reinterpret_cast<uint4 *>(KBT + sw128_offset(j, i8 * 8, DK < 8 ? 8 : DK)) = b;
                }
            }
        }
        // (beta V)^T with delta, V^T without: row c of a [32][64] tile
        {
            const int c = tid & 31, part = tid >> 5;  // 4 parts of 16 tokens
#pragma unroll
            for (int i8 = 0; i8 < 2; ++i8) {
                const int i0 = part * 16 + i8 * 8;
                float vv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = __bfloat162float(Vraw[(i0 + e) * DVS + c]);
                    vv[e] = DELTA ? bv[i0 + e] * x : x;
                }
                uint4 a;
                a.x = pack_bf16(vv[0], vv[1]);
                a.y = pack_bf16(vv[2], vv[3]);
                a.z = pack_bf16(vv[4], vv[5]);
                a.w = pack_bf16(vv[6], vv[7]);
                *reinterpret_cast<uint4 *>((DELTA ? VBT : XB) + sw128_offset(c, i0, 32)) = a;
                if (!DELTA) *reinterpret_cast<uint4 *>(UB + sw128_offset(c, i0, 32)) = a;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- E1: [Q; K] K^T -> R1
        if (tid == 0) {
            const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_bf16(tmem + kR1, tile_desc(smem_u32(QK), 128, 0, ks),
                         tile_desc(smem_u32(QK), 128, 64, ks), id, ks > 0);
            mma_commit(bar);
        }
        mma_wait();
        if (!ok) break;

        // ---- E2: decay-masked scores P (bf16, rows 64..127 of TP) and couplings A (fp32)
        {
            const int r = 32 * (warp & 1) + lane;  // token of this row
            const bool is_q = warp < 2;
            float a[32];
            const float Gr = Gv[r];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_base + kR1 + 32 * half, a);
                tmem_ld_wait();
                if (is_q) {
#pragma unroll
                    for (int i8 = 0; i8 < 4; ++i8) {
                        float p[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int i = half * 32 + i8 * 8 + e;
                            p[e] = (i <= r) ? a[i8 * 8 + e] * (ALPHA ? expf(Gr - Gv[i]) : 1.f) : 0.f;
                        }
                        uint4 w4;
                        w4.x = pack_bf16(p[0], p[1]);
                        w4.y = pack_bf16(p[2], p[3]);
                        w4.z = pack_bf16(p[4], p[5]);
                        w4.w = pack_bf16(p[6], p[7]);
                        *reinterpret_cast<uint4 *>(TP + sw128_offset(64 + r, half * 32 + i8 * 8, 128)) = w4;
                    }
                } else if (DELTA) {
                    const float br = bv[r];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int i = half * 32 + e;
                        Am[r * AP + i] = (i < r) ? br * a[e] * (ALPHA ? expf(Gr - Gv[i]) : 1.f) : 0.f;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        if (DELTA) {
            // ---- T = (I + A)^-1: diagonal 16x16 blocks by forward substitution
            if (tid < 64) {
                const int b = tid >> 4, c = tid & 15;
                float x[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    float s = (rr == c) ? 1.f : 0.f;
#pragma unroll
                    for (int i = 0; i < rr; ++i) s -= Am[(16 * b + rr) * AP + 16 * b + i] * x[i];
                    x[rr] = s;
                }
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) Tm[(16 * b + rr) * AP + 16 * b + c] = x[rr];
            }
            __syncthreads();
            // off-diagonal blocks, one block row at a time:
            //   X = A[rows b, cols < 16b] T[< 16b, < 16b];  T[rows b, < 16b] = -T_bb X
            for (int b = 1; b < 4; ++b) {
                const int ncol = 16 * b;
                for (int idx = tid; idx < 16 * ncol; idx += NT) {
                    const int rr = idx / ncol, col = idx % ncol;
                    float s = 0.f;
                    for (int i = col; i < ncol; ++i) s += Am[(16 * b + rr) * AP + i] * Tm[i * AP + col];
                    Xt[rr * 49 + col] = s;
                }
                __syncthreads();
                for (int idx = tid; idx < 16 * ncol; idx += NT) {
                    const int rr = idx / ncol, col = idx % ncol;
                    float s = 0.f;
                    for (int i = 0; i <= rr; ++i) s += Tm[(16 * b + rr) * AP + 16 * b + i] * Xt[i * 49 + col];
                    Tm[(16 * b + rr) * AP + col] = -s;
                }
                __syncthreads();
            }
            // T (lower triangle, bf16) -> rows 0..63 of TP
            for (int idx = tid; idx < C * 8; idx += NT) {
                const int r = idx >> 3, i8 = idx & 7;
                float t[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = i8 * 8 + e;
                    t[e] = (i <= r) ? Tm[r * AP + i] : 0.f;
                }
                uint4 w4;
                w4.x = pack_bf16(t[0], t[1]);
                w4.y = pack_bf16(t[2], t[3]);
                w4.z = pack_bf16(t[4], t[5]);
                w4.w = pack_bf16(t[6], t[7]);
                *reinterpret_cast<uint4 *>(TP + sw128_offset(r, i8 * 8, 128)) = w4;
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- E3: [T; P] (beta g K)^T -> R2 (rows 0..63 = W);  [T; P] (beta V)^T -> R3
            if (tid == 0) {
                const uint32_t idw = idesc_bf16_f32(128, DK);
                const uint32_t idu = idesc_bf16_f32(128, DVS);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ad = tile_desc(smem_u32(TP), 128, 0, ks);
                    mma_bf16(tmem + kR2, ad, tile_desc(smem_u32(KBT), DK < 8 ? 8 : DK, 0, ks), idw, ks > 0);
                    mma_bf16(tmem + kR3, ad, tile_desc(smem_u32(VBT), 32, 0, ks), idu, ks > 0);
                }
                mma_commit(bar);
            }
            mma_wait();
            if (!ok) break;

            // ---- E4: -W -> rows 0..63 of WQ
            if (warp < 2) {
                const int r = 32 * warp + lane;
#pragma unroll
                for (int cb = 0; cb < (DK + 31) / 32; ++cb) {
                    float w[32];
                    tmem_ld32(tmem + lane_base + kR2 + 32 * cb, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int i8 = 0; i8 < 4; ++i8) {
                        uint4 w4;
                        w4.x = pack_bf16(-w[i8 * 8 + 0], -w[i8 * 8 + 1]);
                        w4.y = pack_bf16(-w[i8 * 8 + 2], -w[i8 * 8 + 3]);
                        w4.z = pack_bf16(-w[i8 * 8 + 4], -w[i8 * 8 + 5]);
                        w4.w = pack_bf16(-w[i8 * 8 + 6], -w[i8 * 8 + 7]);
                        *reinterpret_cast<uint4 *>(WQ + sw128_offset(r, cb * 32 + i8 * 8, 128)) = w4;
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }

        // ---- S1: [-W; g Q] S^T (+)= R3
        if (tid == 0) {
            const uint32_t id = idesc_bf16_f32(128, DVS);
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_bf16(tmem + kR3, tile_desc(smem_u32(WQ), 128, 0, ks),
                         tile_desc(smem_u32(SB), 32, 0, ks), id, DELTA ? 1u : (ks > 0 ? 1u : 0u));
            mma_commit(bar);
        }
        mma_wait();
        if (!ok) break;

        if (DELTA) {
            // ---- S2: U^T and (U - beta V)^T from rows 0..63 of R3
            if (warp < 2) {
                const int i = 32 * warp + lane;
                float u[32];
                tmem_ld32(tmem + lane_base + kR3, u);
                tmem_ld_wait();
                const float b = bv[i];
#pragma unroll
                for (int c = 0; c < DVS; ++c) {
                    st_bf16(UB, sw128_offset(c, i, 32), u[c]);
                    const float x = __bfloat162float(Vraw[i * DVS + c]);
                    st_bf16(XB, sw128_offset(c, i, 32), u[c] - b * x);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }

        // ---- S3: (kd K)^T U -> R4;  [T; P] (U - beta V)^T += R3
        if (tid == 0) {
            const uint32_t id = idesc_bf16_f32(128, DVS);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                mma_bf16(tmem + kR4, tile_desc(smem_u32(KTT), 128, 0, ks),
                         tile_desc(smem_u32(UB), 32, 0, ks), id, ks > 0);
                mma_bf16(tmem + kR3, tile_desc(smem_u32(TP), 128, 0, ks),
                         tile_desc(smem_u32(XB), 32, 0, ks), id, 1u);
            }
            mma_commit(bar);
        }
        mma_wait();
        if (!ok) break;

        // ---- S4: S <- g_C S + Delta S (registers, bf16 copy to SB); O out
        {
            float d[32];
            tmem_ld32(tmem + lane_base + kR4, d);
            tmem_ld_wait();
            const float gC = gv[C - 1];
            if (tid < DK) {
#pragma unroll
                for (int c = 0; c < DVS; ++c) {
                    Sr[c] = gC * Sr[c] + d[c];
                    st_bf16(SB, sw128_offset(c, tid, 32), Sr[c]);
                }
            }
            if (warp >= 2) {
                const int r = 32 * (warp - 2) + lane;
                float ov[32];
                tmem_ld32(tmem + lane_base + kR3, ov);
                tmem_ld_wait();
                if (r < n) {
                    uint4 *dst = reinterpret_cast<uint4 *>(o + (bh * T + t0 + r) * dv + c0);
#pragma unroll
                    for (int i8 = 0; i8 < 4; ++i8) {
                        uint4 w4;
                        w4.x = pack_bf16(ov[i8 * 8 + 0], ov[i8 * 8 + 1]);
                        w4.y = pack_bf16(ov[i8 * 8 + 2], ov[i8 * 8 + 3]);
                        w4.z = pack_bf16(ov[i8 * 8 + 4], ov[i8 * 8 + 5]);
                        w4.w = pack_bf16(ov[i8 * 8 + 6], ov[i8 * 8 + 7]);
                        dst[i8] = w4;
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (!ok) {
        if (lane == 0) atomicExch(&g_tc_error, 1);
    }
    cp_async_wait_all();
    if (ok && tid < DK) {
#pragma unroll
        for (int c = 0; c < DVS; ++c) ST[(bh * dv + c0 + c) * DK + tid] = Sr[c];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int DK, bool ALPHA, bool DELTA>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                         int T, int dv, cudaStream_t stream, int slot) {
    auto fn = chunk_tc_kernel<DK, ALPHA, DELTA>;
    const int bytes = TcLayout<DK>::ALLOC;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), bytes, slot);
    if (e != cudaSuccess) return e;
    dim3 grid(dv / DVS, H, B);
    fn<<<grid, NT, bytes, stream>>>(static_cast<const bf16 *>(q), static_cast<const bf16 *>(k),
                                    static_cast<const bf16 *>(v), ALPHA ? alpha : nullptr,
                                    DELTA ? beta : nullptr, S0, static_cast<bf16 *>(o), S_T, H,
                                    T, dv);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                        int T, int dv, lr_mode mode, cudaStream_t stream, int slot) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, false, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv,
                                              stream, slot + 0);
    case LR_MODE_DECAY:
        return launch_typed<DK, true, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv,
                                             stream, slot + 1);
    case LR_MODE_DELTA:
        return launch_typed<DK, false, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv,
                                             stream, slot + 2);
    default:
        return launch_typed<DK, true, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv,
                                            stream, slot + 3);
    }
}

}  // namespace

// Attribute slots 32..43 belong to this file.
cudaError_t launch_chunked_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *S_T, int B,
                              int H, int T, int dk, int dv, lr_mode mode, cudaStream_t stream) {
    switch (dk) {
    case 32:
        return launch_mode<32>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, stream, 32);
    case 64:
        return launch_mode<64>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, stream, 36);
    default:
        return launch_mode<128>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, stream, 40);
    }
}

int read_and_clear_tc_error() {
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_error, sizeof(int)) != cudaSuccess) return -1;
    if (h) cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    return h;
}

}  // namespace lr
