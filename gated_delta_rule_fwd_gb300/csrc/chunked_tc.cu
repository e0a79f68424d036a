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
//   P  = (Q K^T) (.) M,          M_ri = e^{G_r - G_i} for i <= r        (scores)
//   A  = strict_lower(diag(beta) (K K^T) (.) M)                        (delta couplings)
//   T  = (I + A)^-1              unit lower triangular (the WY / UT step)
//   W  = T diag(beta g) K,       Ut = T diag(beta) V
//   U  = Ut - W S^T              pseudo-values u_r of the WY representation
//   O  = diag(g) Q S^T + P U
//   S <- g_C S + U^T diag(kd) K
// and without the delta term U = V.  The derivation: the gated recurrence
// unrolled inside a block gives u_r = beta_r (v_r - g_r S k_r -
// sum_{i<r} e^{G_r - G_i} (k_i.k_r) u_i), a unit-lower-triangular system.
//
// Two launches:
//  * prep: one CTA per (block, head, batch), all blocks in parallel.  Computes
//    what does not depend on the state: G, the scores P, the UT inverse T
//    (blocked forward substitution in fp32 on the CUDA cores) and -W, and
//    writes -W, T and P to the workspace as bf16 tiles already in the
//    shared-memory operand layout, plus the per-token gate vectors.
//  * scan: one CTA per (32 value channels, head, batch); rows of S evolve
//    independently given k, alpha and beta, so slices never exchange data.
//    The loop over blocks is sequential; the next block's tiles are fetched
//    and its operand tiles built while the current block's products run.
//
// Every product runs as an M = 128 tcgen05.mma with K-major 128-byte-swizzled
// shared-memory operands and an fp32 accumulator in tensor memory; 64-row
// operands are stacked to fill M:
//   prep  E1  [Q; K] K^T            -> [Q K^T ; K K^T]
//         E3  [T; 0] (beta g K)^T   -> [W ; 0]
//   scan  G1  [T; 0] (beta V)^T     -> [Ut ; 0]           (R3)
//             [-W; g Q] S^T        +=  [U ; g Q S^T]     (R3)
//         G2  (kd K)^T U           ->  Delta S^T          (R4)
//             [0; P] U             +=  rows 64..127 = O   (R3)
// The fp32 master copy of the state slice lives in registers (thread j owns
// column j); a bf16 copy in shared memory feeds the next block.  A final
// short block is zero-filled (alpha treated as 1, beta as 0), which leaves
// the real tokens' results unchanged.
#include "lr_internal.cuh"
#include "tc_common.cuh"

namespace lr {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int C = 64;      // tokens per block
constexpr int DVS = 32;    // value channels per scan CTA
constexpr int NT = 128;    // threads per CTA
constexpr int AP = C + 1;  // padded fp32 row of A and T
constexpr int XP = 49;     // padded fp32 row of the solve scratch

__device__ int g_tc_error = 0;  // set to 1 when a bounded wait gives up

// Workspace record of one (head, block), written by prep and read by scan.
template <int DK>
struct Rec {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int WT = 0;                 // -W: KB blocks of [64 rows][128 B]
    static constexpr int TT = WT + KB * 8192;    // T:  [64][64] bf16 tile
    static constexpr int PT = TT + 8192;         // P:  [64][64] bf16 tile
    static constexpr int VEC = PT + 8192;        // G, g, kd, beta: 4 x 64 fp32
    static constexpr int BYTES = VEC + 1024;
};

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
__device__ __forceinline__ uint4 pack8(const float *x) {
    uint4 r;
    r.x = pack_bf16(x[0], x[1]);
    r.y = pack_bf16(x[2], x[3]);
    r.z = pack_bf16(x[4], x[5]);
    r.w = pack_bf16(x[6], x[7]);
    return r;
}
__device__ __forceinline__ float bf16_at(const uint8_t *tile, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const bf16 *>(tile + off));
}
__device__ __forceinline__ void st_bf16(uint8_t *tile, uint32_t off, float x) {
    *reinterpret_cast<bf16 *>(tile + off) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// ===================================================================== prep

template <int DK>
struct PrepLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int QK = 0;                            // [128 rows][DK]: Q rows, K rows
    static constexpr int TZ = QK + 128 * 128 * KB;          // [128][64]: T rows, zero rows
    static constexpr int KBT = TZ + 16384;                  // [DK][64]: (beta g K)^T
    static constexpr int AM = KBT + ((DK * 128 + 1023) / 1024) * 1024;  // fp32 [64][AP]
    static constexpr int TM = AM + C * AP * 4;              // fp32 [64][AP]
    static constexpr int XT = TM + C * AP * 4;              // fp32 [16][XP]
    static constexpr int VEC = XT + 16 * XP * 4;            // G, ginv, g, kd, bg, b
    static constexpr int BAR = VEC + 6 * 64 * 4;
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};

// One block row of the blocked UT inverse: with the rows of T above it done,
//   X = A[rows b, cols < 16b] T[< 16b, < 16b];   T[rows b, cols < 16b] = -T_bb X.
// 128 threads: thread = (row rr of the block, column group cg), columns cg + 8k.
template <int BR>
__device__ __forceinline__ void ut_block_row(const float *Am, float *Tm, float *Xt, int tid) {
    constexpr int NC = 2 * BR;  // columns per thread (16*BR columns / 8 groups)
    const int rr = tid & 15, cg = tid >> 4;
    const int row = 16 * BR + rr;
    float acc[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) acc[k] = 0.f;
#pragma unroll 4
    for (int i = 0; i < 16 * BR; ++i) {
        const float a = Am[row * AP + i];
#pragma unroll
        for (int k = 0; k < NC; ++k) acc[k] += a * Tm[i * AP + cg + 8 * k];
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) Xt[rr * XP + cg + 8 * k] = acc[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NC; ++k) acc[k] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float t = Tm[row * AP + 16 * BR + i];
#pragma unroll
        for (int k = 0; k < NC; ++k) acc[k] += t * Xt[i * XP + cg + 8 * k];
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) Tm[row * AP + cg + 8 * k] = -acc[k];
    __syncthreads();
}

// T = (I + A)^-1 for a strictly lower A (64 x 64, fp32 in shared memory).
// Tm must hold zeros in the blocks above the block diagonal on entry; on exit
// it holds T's lower triangle with zeros above the diagonal.
__device__ __forceinline__ void ut_inverse(const float *Am, float *Tm, float *Xt, int tid) {
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        const float *Ab = Am + (16 * b) * AP + 16 * b;
        float x[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float s0 = (rr == c) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < rr; ++i) {
                if (i & 1) s1 -= Ab[rr * AP + i] * x[i];
                else s0 -= Ab[rr * AP + i] * x[i];
            }
            x[rr] = s0 + s1;
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Tm[(16 * b + rr) * AP + 16 * b + c] = x[rr];
    }
    __syncthreads();
    ut_block_row<1>(Am, Tm, Xt, tid);
    ut_block_row<2>(Am, Tm, Xt, tid);
    ut_block_row<3>(Am, Tm, Xt, tid);
}

template <int DK, bool ALPHA, bool DELTA>
__global__ void __launch_bounds__(NT)
chunk_prep_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                  const float *__restrict__ alpha, const float *__restrict__ beta,
                  uint8_t *__restrict__ ws, int H, int T, int nblk) {
    using L = PrepLayout<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = blk * C;
    const int n = min(C, T - t0);
    uint8_t *rec = ws + (bh * nblk + blk) * (size_t)R::BYTES;

    uint8_t *QK = sm + L::QK, *TZ = sm + L::TZ, *KBT = sm + L::KBT;
    float *Am = reinterpret_cast<float *>(sm + L::AM);
    float *Tm = reinterpret_cast<float *>(sm + L::TM);
    float *Xt = reinterpret_cast<float *>(sm + L::XT);
    float *Gv = reinterpret_cast<float *>(sm + L::VEC);
    float *giv = Gv + 64, *gv = Gv + 128, *kdv = Gv + 192, *bgv = Gv + 256, *bv = Gv + 320;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 8);

    // ---- stage Q, K (zero-filled past the end) and the gates
    constexpr int CPR = DK / 8;
    for (int idx = tid; idx < 2 * C * CPR; idx += NT) {
        const int which = idx / (C * CPR);
        const int rem = idx % (C * CPR);
        const int r = rem / CPR, ch = rem % CPR;
        const bool ok = r < n;
        const bf16 *src = (which ? k : q) + ((bh * T + (ok ? t0 + r : 0)) * DK + ch * 8);
        cp_async16(smem_u32(QK + sw128_offset(which * 64 + r, ch * 8, 128)), src, ok);
    }
    cp_async_commit();
    if (DELTA) {
        // zero rows 64..127 of [T; 0] and the upper blocks of Tm
        for (int i = tid; i < 8192 / 16; i += NT)
            reinterpret_cast<uint4 *>(TZ + 8192)[i] = make_uint4(0, 0, 0, 0);
        for (int i = tid; i < C * AP; i += NT) Tm[i] = 0.f;
    }
    float la = 0.f, b = 0.f;
    if (tid < C && tid < n) {
        if (ALPHA) la = __logf(alpha[bh * T + t0 + tid]);
        if (DELTA) b = beta[bh * T + t0 + tid];
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    // inclusive scan of ln alpha over the block (warps 0 and 1 hold the 64 values)
    if (warp < 2) {
        float incl = la;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        Gv[tid] = incl;  // warp 1 adds warp 0's total below
    }
    __syncthreads();
    const float Gfull = tid < C ? Gv[tid] + (tid >= 32 ? Gv[31] : 0.f) : 0.f;
    __syncthreads();
    if (tid < C) Gv[tid] = Gfull;
    __syncthreads();
    // exp(G_r - G_i) = g_r * ginv_i when exp(-G_63) is finite in fp32
    const bool factor = !ALPHA || Gv[C - 1] > -80.f;
    if (tid < C) {
        const float G = Gv[tid];
        const float g = ALPHA ? __expf(G) : 1.f;
        gv[tid] = g;
        giv[tid] = ALPHA ? __expf(-G) : 1.f;
        kdv[tid] = ALPHA ? __expf(Gv[C - 1] - G) : 1.f;
        bgv[tid] = b * g;
        bv[tid] = b;
        float *vec = reinterpret_cast<float *>(rec + R::VEC);
        vec[tid] = G;
        vec[64 + tid] = g;
        vec[128 + tid] = ALPHA ? __expf(Gv[C - 1] - G) : 1.f;
        vec[192 + tid] = b;
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- (beta g K)^T for W: thread j builds row j
    if (DELTA && tid < DK) {
        const int j = tid;
#pragma unroll
        for (int i8 = 0; i8 < C / 8; ++i8) {
            float w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                w8[e] = bgv[i8 * 8 + e] * bf16_at(QK, sw128_offset(64 + i8 * 8 + e, j, 128));
            *reinterpret_cast<uint4 *>(KBT + sw128_offset(j, i8 * 8, DK)) = pack8(w8);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = true;

    // ---- E1: [Q; K] K^T -> TMEM cols [0, 64)
    if (tid == 0) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(QK), 128, 0, ks), tile_desc(smem_u32(QK), 128, 64, ks),
                     id, ks > 0);
        mma_commit(bar);
    }
    ok = __syncthreads_and(mbar_wait(bar, 0) ? 1 : 0) != 0;
    tc_fence_after();

    // ---- E2: P rows (bf16 tile to the workspace), A rows (fp32)
    if (ok) {
        const int r = 32 * (warp & 1) + lane;
        const bool is_q = warp < 2;
        const float Gr = Gv[r], gr = gv[r];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float a[32];
            tmem_ld32(tmem + lane_base + 32 * half, a);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = half * 32 + e;
                const float dec = !ALPHA ? 1.f : (factor ? gr * giv[i] : __expf(Gr - Gv[i]));
                a[e] = (i <= r && (is_q || i < r)) ? a[e] * dec : 0.f;
            }
            if (is_q) {
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8)
                    *reinterpret_cast<uint4 *>(rec + R::PT +
                                               sw128_offset(r, half * 32 + i8 * 8, 64)) =
                        pack8(a + i8 * 8);
            } else if (DELTA) {
                const float br = bv[r];
#pragma unroll
                for (int e = 0; e < 32; ++e) Am[r * AP + half * 32 + e] = br * a[e];
            }
        }
    }
    __syncthreads();

    if (DELTA && ok) {
        ut_inverse(Am, Tm, Xt, tid);
        // T (bf16) -> rows 0..63 of [T; 0] and to the workspace
        for (int idx = tid; idx < C * 8; idx += NT) {
            const int r = idx >> 3, i8 = idx & 7;
            float t[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = Tm[r * AP + i8 * 8 + e];
            const uint4 w4 = pack8(t);
            const uint32_t off = sw128_offset(r, i8 * 8, 64);
            *reinterpret_cast<uint4 *>(TZ + off) = w4;
            *reinterpret_cast<uint4 *>(rec + R::TT + off) = w4;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- E3: [T; 0] (beta g K)^T -> TMEM cols [64, 64 + DK)
        if (tid == 0) {
            const uint32_t id = idesc_bf16_f32(128, DK);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                mma_bf16(tmem + 64, tile_desc(smem_u32(TZ), 128, 0, ks),
                         tile_desc(smem_u32(KBT), DK, 0, ks), id, ks > 0);
            mma_commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 1) ? 1 : 0) != 0;
        tc_fence_after();

        // ---- -W rows -> workspace
        if (ok && warp < 2) {
            const int r = 32 * warp + lane;
#pragma unroll
            for (int cb = 0; cb < DK / 32; ++cb) {
                float w[32];
                tmem_ld32(tmem + lane_base + 64 + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = -w[e];
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8)
                    *reinterpret_cast<uint4 *>(rec + R::WT +
                                               sw128_offset(r, cb * 32 + i8 * 8, 64)) =
                        pack8(w + i8 * 8);
            }
        }
    }
    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===================================================================== scan

template <int DK>
struct ScanLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int WQ_BYTES = 128 * 128 * KB;          // [128][DK]: -W rows, g Q rows
    static constexpr int WQ = 0;                              // x2
    static constexpr int TZP = WQ + 2 * WQ_BYTES;             // x2 [192][64]: T, 0, P rows
    static constexpr int KR_BYTES = 64 * 128 * KB;            // raw K block [64][DK]
    static constexpr int KR = TZP + 2 * 24576;                // x2
    static constexpr int KTT = KR + 2 * KR_BYTES;             // x2 [128][64]: (kd K)^T
    static constexpr int VBT = KTT + 2 * 16384;               // x2 [32][64]: (beta V)^T or V^T
    static constexpr int VR = VBT + 2 * 4096;                 // x2 raw V slice [64][32]
    static constexpr int VEC = VR + 2 * 4096;                 // x2 G, g, kd, beta
    static constexpr int UB = VEC + 2 * 1024;                 // [32][64]: U^T
    static constexpr int SB = UB + 4096;                      // [32][DK]: bf16 state slice
    static constexpr int BAR = SB + 32 * 128 * KB;
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};

// TMEM columns of the scan kernel
constexpr uint32_t kR3 = 0, kR4 = 32, kScanCols = 64;

// Fetch block `blk` of (bh, slice) into buffer `buf` (one cp.async group).
template <int DK, bool DELTA>
__device__ __forceinline__ void scan_fetch(uint8_t *sm, int buf, const bf16 *q, const bf16 *k,
                                           const bf16 *v, const uint8_t *rec, size_t bh, int T,
                                           int blk, int dv, int c0, int tid) {
    using L = ScanLayout<DK>;
    using R = Rec<DK>;
    const int t0 = blk * C;
    constexpr int CPR = DK / 8;
    uint8_t *wq = sm + L::WQ + buf * L::WQ_BYTES;
    uint8_t *kr = sm + L::KR + buf * L::KR_BYTES;
    for (int idx = tid; idx < 2 * C * CPR; idx += NT) {
        const int which = idx / (C * CPR);
        const int rem = idx % (C * CPR);
        const int r = rem / CPR, ch = rem % CPR;
        const bool ok = t0 + r < T;
        const bf16 *src = (which ? k : q) + ((bh * T + (ok ? t0 + r : 0)) * DK + ch * 8);
        const uint32_t dst = which ? smem_u32(kr + sw128_offset(r, ch * 8, 64))
                                   : smem_u32(wq + sw128_offset(64 + r, ch * 8, 128));
        cp_async16(dst, src, ok);
    }
    uint8_t *vr = sm + L::VR + buf * 4096;
    for (int idx = tid; idx < C * (DVS / 8); idx += NT) {
        const int r = idx / (DVS / 8), ch = idx % (DVS / 8);
        const bool ok = t0 + r < T;
        cp_async16(smem_u32(vr + (r * DVS + ch * 8) * 2),
                   v + ((bh * T + (ok ? t0 + r : 0)) * dv + c0 + ch * 8), ok);
    }
    if (DELTA) {
        // -W rows -> rows 0..63 of each 64-wide K block of WQ; T -> rows 0..63 of TZP
        for (int idx = tid; idx < R::KB * 512; idx += NT) {
            const int kb = idx >> 9, c16 = idx & 511;
            cp_async16(smem_u32(wq + kb * 16384 + c16 * 16), rec + R::WT + kb * 8192 + c16 * 16, true);
        }
        for (int idx = tid; idx < 512; idx += NT)
            cp_async16(smem_u32(sm + L::TZP + buf * 24576 + idx * 16), rec + R::TT + idx * 16, true);
    }
    for (int idx = tid; idx < 512; idx += NT)
        cp_async16(smem_u32(sm + L::TZP + buf * 24576 + 16384 + idx * 16), rec + R::PT + idx * 16,
                   true);
    for (int idx = tid; idx < 64; idx += NT)
        cp_async16(smem_u32(sm + L::VEC + buf * 1024 + idx * 16), rec + R::VEC + idx * 16, true);
    cp_async_commit();
}

// Operand tiles of block `buf` that need only its fetched inputs:
// g Q in place, (kd K)^T, (beta V)^T (delta) or V^T.
template <int DK, bool DELTA>
__device__ __forceinline__ void scan_tiles(uint8_t *sm, int buf, int tid) {
    using L = ScanLayout<DK>;
    uint8_t *wq = sm + L::WQ + buf * L::WQ_BYTES;
    const uint8_t *kr = sm + L::KR + buf * L::KR_BYTES;
    uint8_t *ktt = sm + L::KTT + buf * 16384;
    uint8_t *vbt = sm + L::VBT + buf * 4096;
    const bf16 *vr = reinterpret_cast<const bf16 *>(sm + L::VR + buf * 4096);
    const float *vec = reinterpret_cast<const float *>(sm + L::VEC + buf * 1024);
    const float *gv = vec + 64, *kdv = vec + 128, *bv = vec + 192;
    for (int idx = tid; idx < C * (DK / 8); idx += NT) {
        const int r = idx / (DK / 8), ch = idx % (DK / 8);
        uint4 *p = reinterpret_cast<uint4 *>(wq + sw128_offset(64 + r, ch * 8, 128));
        const uint4 raw = *p;
        const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
        const float g = gv[r];
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = g * __bfloat162float(e[t]);
        *p = pack8(x);
    }
    if (tid < DK) {
        const int j = tid;
#pragma unroll
        for (int i8 = 0; i8 < C / 8; ++i8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[e] = kdv[i8 * 8 + e] * bf16_at(kr, sw128_offset(i8 * 8 + e, j, 64));
            *reinterpret_cast<uint4 *>(ktt + sw128_offset(j, i8 * 8, 128)) = pack8(x);
        }
    }
    {
        const int c = tid & 31, part = tid >> 5;  // 4 parts of 16 tokens
#pragma unroll
        for (int i8 = 0; i8 < 2; ++i8) {
            const int i0 = part * 16 + i8 * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float vv = __bfloat162float(vr[(i0 + e) * DVS + c]);
                x[e] = DELTA ? bv[i0 + e] * vv : vv;
            }
            *reinterpret_cast<uint4 *>(vbt + sw128_offset(c, i0, 32)) = pack8(x);
        }
    }
}

template <int DK, bool ALPHA, bool DELTA>
__global__ void __launch_bounds__(NT, 1)
chunk_scan_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                  const bf16 *__restrict__ v, const uint8_t *__restrict__ ws,
                  const float *__restrict__ S0, bf16 *__restrict__ o, float *__restrict__ ST,
                  int H, int T, int dv, int nblk) {
    using L = ScanLayout<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const uint8_t *recs = ws + bh * nblk * (size_t)R::BYTES;

    uint8_t *UB = sm + L::UB, *SB = sm + L::SB;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 8);

    // zero everything once: the padding rows of the stacked operands must read 0
    for (int i = tid; i < L::BAR / 16; i += NT)
        reinterpret_cast<uint4 *>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kScanCols);
        tmem_relinquish();
    }
    __syncthreads();

    // fp32 master copy of the state slice: thread j owns S[c0 + c][j], c < 32
    float Sr[DVS];
#pragma unroll
    for (int c = 0; c < DVS; ++c)
        Sr[c] = (S0 && tid < DK) ? S0[(bh * dv + c0 + c) * DK + tid] : 0.f;
    if (tid < DK) {
#pragma unroll
        for (int c = 0; c < DVS; ++c) st_bf16(SB, sw128_offset(c, tid, 32), Sr[c]);
    }

    scan_fetch<DK, DELTA>(sm, 0, q, k, v, recs, bh, T, 0, dv, c0, tid);
    if (nblk > 1)
        scan_fetch<DK, DELTA>(sm, 1, q, k, v, recs + R::BYTES, bh, T, 1, dv, c0, tid);
    if (nblk > 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else cp_async_wait_all();
    __syncthreads();
    scan_tiles<DK, DELTA>(sm, 0, tid);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    uint32_t phase = 0;
    bool ok = true;

    auto mma_wait = [&]() {
        const bool mine = mbar_wait(bar, phase & 1);
        ++phase;
        ok = __syncthreads_and(mine ? 1 : 0) != 0;
        tc_fence_after();
    };

    const uint32_t id32 = idesc_bf16_f32(128, DVS);
    for (int blk = 0; blk < nblk && ok; ++blk) {
        const int buf = blk & 1;
        const int t0 = blk * C;
        const int n = min(C, T - t0);
        const uint32_t wq = smem_u32(sm + L::WQ + buf * L::WQ_BYTES);
        const uint32_t tzp = smem_u32(sm + L::TZP + buf * 24576);
        const uint32_t ktt = smem_u32(sm + L::KTT + buf * 16384);
        const uint32_t vbt = smem_u32(sm + L::VBT + buf * 4096);
        const float *vec = reinterpret_cast<const float *>(sm + L::VEC + buf * 1024);

        // ---- G1: R3 = [T; 0] (beta V)^T + [-W; gQ] S^T   (without delta: [0; gQ] S^T,
        //      and the state update and the P V part of the output go with it)
        if (tid == 0) {
            if (DELTA) {
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(tmem + kR3, tile_desc(tzp, 192, 0, ks), tile_desc(vbt, 32, 0, ks), id32,
                             ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_bf16(tmem + kR3, tile_desc(wq, 128, 0, ks), tile_desc(smem_u32(SB), 32, 0, ks),
                         id32, (DELTA || ks > 0) ? 1u : 0u);
            if (!DELTA) {
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    mma_bf16(tmem + kR4, tile_desc(ktt, 128, 0, ks), tile_desc(vbt, 32, 0, ks), id32,
                             ks > 0);
                    mma_bf16(tmem + kR3, tile_desc(tzp, 192, 64, ks), tile_desc(vbt, 32, 0, ks),
                             id32, 1u);
                }
            }
            mma_commit(bar);
        }
        // meanwhile: the next block's operand tiles
        if (blk + 1 < nblk) {
            cp_async_wait_all();
            __syncthreads();
            scan_tiles<DK, DELTA>(sm, buf ^ 1, tid);
            fence_async_smem();
        }
        mma_wait();
        if (!ok) break;

        if (DELTA) {
            // ---- U^T from rows 0..63 of R3
            if (warp < 2) {
                const int i = 32 * warp + lane;
                float u[32];
                tmem_ld32(tmem + lane_base + kR3, u);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < DVS; ++c) st_bf16(UB, sw128_offset(c, i, 32), u[c]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ---- G2: R4 = (kd K)^T U;  R3 += [0; P] U
            if (tid == 0) {
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    mma_bf16(tmem + kR4, tile_desc(ktt, 128, 0, ks), tile_desc(smem_u32(UB), 32, 0, ks),
                             id32, ks > 0);
                    mma_bf16(tmem + kR3, tile_desc(tzp, 192, 64, ks),
                             tile_desc(smem_u32(UB), 32, 0, ks), id32, 1u);
                }
                mma_commit(bar);
            }
            mma_wait();
            if (!ok) break;
        }

        // ---- state S <- g_C S + Delta S (registers; bf16 copy to SB); O out
        {
            float d[32];
            tmem_ld32(tmem + lane_base + kR4, d);
            tmem_ld_wait();
            const float gC = vec[64 + C - 1];
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
                    for (int i8 = 0; i8 < 4; ++i8) dst[i8] = pack8(ov + i8 * 8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (blk + 2 < nblk)
            scan_fetch<DK, DELTA>(sm, buf, q, k, v, recs + (size_t)(blk + 2) * R::BYTES, bh, T,
                                  blk + 2, dv, c0, tid);
    }

    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    cp_async_wait_all();
    if (ok && tid < DK) {
#pragma unroll
        for (int c = 0; c < DVS; ++c) ST[(bh * dv + c0 + c) * DK + tid] = Sr[c];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kScanCols);
}

// ================================================================== launch

template <int DK, bool ALPHA, bool DELTA>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                         int T, int dv, void *ws, cudaStream_t stream, int slot) {
    const int nblk = (T + C - 1) / C;
    auto prep = chunk_prep_kernel<DK, ALPHA, DELTA>;
    auto scan = chunk_scan_kernel<DK, ALPHA, DELTA>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), PrepLayout<DK>::ALLOC,
                                     slot);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC, slot + 12);
    if (e != cudaSuccess) return e;
    prep<<<dim3(nblk, H, B), NT, PrepLayout<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), ALPHA ? alpha : nullptr,
        DELTA ? beta : nullptr, static_cast<uint8_t *>(ws), H, T, nblk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    scan<<<dim3(dv / DVS, H, B), NT, ScanLayout<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), static_cast<const bf16 *>(v),
        static_cast<const uint8_t *>(ws), S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                        int T, int dv, lr_mode mode, void *ws, cudaStream_t stream, int slot) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, false, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, ws,
                                              stream, slot + 0);
    case LR_MODE_DECAY:
        return launch_typed<DK, true, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, ws,
                                             stream, slot + 1);
    case LR_MODE_DELTA:
        return launch_typed<DK, false, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, ws,
                                             stream, slot + 2);
    default:
        return launch_typed<DK, true, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, ws,
                                            stream, slot + 3);
    }
}

}  // namespace

size_t chunked_tc_workspace_bytes(int B, int H, int T, int dk) {
    const size_t nblk = (size_t)((T + C - 1) / C);
    const size_t rec = dk == 32 ? Rec<32>::BYTES : dk == 64 ? Rec<64>::BYTES : Rec<128>::BYTES;
    return (size_t)B * H * nblk * rec;
}

// Attribute slots 32..55 belong to this file.
cudaError_t launch_chunked_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *S_T, int B,
                              int H, int T, int dk, int dv, lr_mode mode, void *ws,
                              cudaStream_t stream) {
    switch (dk) {
    case 32:
        return launch_mode<32>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, ws, stream, 32);
    case 64:
        return launch_mode<64>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, ws, stream, 36);
    default:
        return launch_mode<128>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, ws, stream,
                                40);
    }
}

int read_and_clear_tc_error() {
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_error, sizeof(int)) != cudaSuccess) return -1;
    if (h) cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    return h;
}

}  // namespace lr
