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
//   scan      [T diag(beta); 0] V  -> [Ut ; 0]
//             [-W; Q] S^T          -> [-W S^T ; Q S^T]    (two K halves)
//             K^T (kd U)           -> Delta S^T           (K read MN-major)
//             [0; P] U             -> rows 64..127 = P U
//   with U = Ut - W S^T and O = diag(g) Q S^T + P U formed in the epilogues.
// The fp32 master copy of the state slice lives in registers (thread j owns
// column j); a bf16 copy in shared memory feeds the next block.  A final
// short block is zero-filled (alpha treated as 1, beta as 0), which leaves
// the real tokens' results unchanged.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

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
    static constexpr int TB = QK + 128 * 128 * KB;          // [64][64] bf16: T diag(beta)
    static constexpr int XT = TB;                           // fp32 [16][XP] solve scratch, inside TB
    static constexpr int AM = TB + 8192;                    // fp32 [64][AP]
    static constexpr int TM = AM + C * AP * 4;              // fp32 [64][AP]
    static constexpr int VEC = TM + C * AP * 4;             // G, ginv, g, beta
    static constexpr int BAR = VEC + 4 * 64 * 4;
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};
static_assert(16 * XP * 4 <= 8192, "solve scratch must fit inside the T tile");

// Element (r, c) of a 64 x 64 fp32 matrix in shared memory, rows padded to 65
// floats so that a warp touching one column of 32 rows hits 32 banks.
__device__ __forceinline__ int sw64(int r, int c) { return r * AP + c; }

// D (16x8, fp32) += A (16x8, tf32) B (8x8, tf32): the warp-level tensor-core
// product, fragments as in the PTX m16n8k8 layout (g = lane/4, t = lane%4):
// a = {A[g][t], A[g+8][t], A[g][t+4], A[g+8][t+4]}, b = {B[t][g], B[t+4][g]},
// d = {D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1]}.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One block row BR of the blocked UT inverse (rows 16BR..16BR+15), with the
// rows above it done:
//   X = A[rows, cols < 16BR] T[< 16BR, < 16BR];   T[rows, cols < 16BR] = -T_bb X
// on the tensor cores (m16n8k8, tf32 in, fp32 accumulate).  Warp w takes the
// 8-column tiles nt = w, w+4, ...; K steps that only meet the zero blocks of T
// above its block diagonal are skipped, so those blocks are never read.
template <int BR>
__device__ __forceinline__ void ut_block_row(const float *Am, float *Tm, float *Xt, int tid) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int r0 = 16 * BR;
    for (int nt = warp; nt < 2 * BR; nt += 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kk = 2 * (nt >> 1); kk < 2 * BR; ++kk) {
            const uint32_t a[4] = {to_tf32(Am[(r0 + g) * AP + 8 * kk + t]),
                                   to_tf32(Am[(r0 + g + 8) * AP + 8 * kk + t]),
                                   to_tf32(Am[(r0 + g) * AP + 8 * kk + t + 4]),
                                   to_tf32(Am[(r0 + g + 8) * AP + 8 * kk + t + 4])};
            mma_tf32(d, a, to_tf32(Tm[(8 * kk + t) * AP + 8 * nt + g]),
                     to_tf32(Tm[(8 * kk + t + 4) * AP + 8 * nt + g]));
        }
        Xt[g * XP + 8 * nt + 2 * t] = d[0];
        Xt[g * XP + 8 * nt + 2 * t + 1] = d[1];
        Xt[(g + 8) * XP + 8 * nt + 2 * t] = d[2];
        Xt[(g + 8) * XP + 8 * nt + 2 * t + 1] = d[3];
    }
    __syncthreads();
    for (int nt = warp; nt < 2 * BR; nt += 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t a[4] = {to_tf32(Tm[(r0 + g) * AP + r0 + 8 * kk + t]),
                                   to_tf32(Tm[(r0 + g + 8) * AP + r0 + 8 * kk + t]),
                                   to_tf32(Tm[(r0 + g) * AP + r0 + 8 * kk + t + 4]),
                                   to_tf32(Tm[(r0 + g + 8) * AP + r0 + 8 * kk + t + 4])};
            mma_tf32(d, a, to_tf32(Xt[(8 * kk + t) * XP + 8 * nt + g]),
                     to_tf32(Xt[(8 * kk + t + 4) * XP + 8 * nt + g]));
        }
        Tm[(r0 + g) * AP + 8 * nt + 2 * t] = -d[0];
        Tm[(r0 + g) * AP + 8 * nt + 2 * t + 1] = -d[1];
        Tm[(r0 + g + 8) * AP + 8 * nt + 2 * t] = -d[2];
        Tm[(r0 + g + 8) * AP + 8 * nt + 2 * t + 1] = -d[3];
    }
    __syncthreads();
}

// T = (I + A)^-1 for a strictly lower A (64 x 64, fp32 in shared memory).  On
// exit Tm holds T's lower triangle (diagonal blocks include their zero upper
// triangles); the blocks above the block diagonal are never written or read.
__device__ __forceinline__ void ut_inverse(const float *Am, float *Tm, float *Xt, int tid) {
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        float x[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float s0 = (rr == c) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < rr; ++i) {
                const float a = Am[sw64(16 * b + rr, 16 * b + i)];
                if (i & 1) s1 -= a * x[i];
                else s0 -= a * x[i];
            }
            x[rr] = s0 + s1;
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Tm[sw64(16 * b + rr, 16 * b + c)] = x[rr];
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
                  uint8_t *__restrict__ ws, int H, int T, int nblk,
                  const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk) {
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

    uint8_t *QK = sm + L::QK, *TB = sm + L::TB;
    float *Am = reinterpret_cast<float *>(sm + L::AM);
    float *Tm = reinterpret_cast<float *>(sm + L::TM);
    float *Xt = reinterpret_cast<float *>(sm + L::XT);
    float *Gv = reinterpret_cast<float *>(sm + L::VEC);
    float *giv = Gv + 64, *gv = Gv + 128, *bv = Gv + 192;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 32);

    // ---- stage Q, K (zero-filled past the end: tiled TMA for dk >= 64, cp.async
    //      otherwise) and the gates
    uint64_t *lbar = bar + 2;
    constexpr bool kTma = DK >= 64;
    if (kTma) {
        if (tid == 0) {
            mbar_init(lbar, 1);
            fence_mbar_init();
            mbar_expect_tx(lbar, 2u * (uint32_t)L::KB * 8192u);
#pragma unroll
            for (int kb = 0; kb < L::KB; ++kb) {
                tma_load_3d(QK + kb * 16384, &tmq, kb * 64, t0, (int)bh, lbar);
                tma_load_3d(QK + kb * 16384 + 8192, &tmk, kb * 64, t0, (int)bh, lbar);
            }
        }
    } else {
        constexpr int CPR = DK / 8;
        for (int idx = tid; idx < 2 * C * CPR; idx += NT) {
            const int which = idx / (C * CPR);
            const int rem = idx % (C * CPR);
            const int r = rem / CPR, ch = rem % CPR;
            const bool okr = r < n;
            const bf16 *src = (which ? k : q) + ((bh * T + (okr ? t0 + r : 0)) * DK + ch * 8);
            cp_async16(smem_u32(QK + sw128_offset(which * 64 + r, ch * 8, 128)), src, okr);
        }
        cp_async_commit();
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
        tmem_alloc(tmem_slot, 128);
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
        bv[tid] = b;
        float *vec = reinterpret_cast<float *>(rec + R::VEC);
        vec[tid] = G;
        vec[64 + tid] = g;
        vec[128 + tid] = ALPHA ? __expf(Gv[C - 1] - G) : 1.f;
        vec[192 + tid] = b;
    }
    bool ok = true;
    if (kTma) ok = mbar_wait(lbar, 0);
    else cp_async_wait_all();
    fence_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    // ---- E1: [Q; K] K^T -> TMEM cols [0, 64)
    if (tid == 0) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(QK), 128, 0, ks), tile_desc(smem_u32(QK), 128, 64, ks),
                     id, ks > 0);
        mma_commit(bar);
    }
    ok = __syncthreads_and((ok && mbar_wait(bar, 0)) ? 1 : 0) != 0;
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
                for (int e = 0; e < 32; ++e) Am[sw64(r, half * 32 + e)] = br * a[e];
            }
        }
    }
    tc_fence_before();  // the score columns are reused by W below
    __syncthreads();

    if (DELTA && ok) {
        ut_inverse(Am, Tm, Xt, tid);
        // T diag(beta) (bf16) -> workspace; T diag(beta g) -> the T tile (over the
        // solve scratch), the A operand of W = T diag(beta g) K
        for (int idx = tid; idx < C * 8; idx += NT) {
            const int r = idx >> 3, i8 = idx & 7;
            float t[8], tg[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = i8 * 8 + e;
                t[e] = i <= r ? Tm[sw64(r, i)] * bv[i] : 0.f;
                tg[e] = t[e] * gv[i];
            }
            const uint32_t off = sw128_offset(r, i8 * 8, 64);
            *reinterpret_cast<uint4 *>(rec + R::TT + off) = pack8(t);
            *reinterpret_cast<uint4 *>(TB + off) = pack8(tg);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- E3: T diag(beta g) K -> W, M = 64 (TMEM cols [0, DK): rows 16w..16w+15
        //      in lanes 32w..32w+15 of warp w); K read MN-major from the K rows
        if (tid == 0) {
            const uint32_t id = idesc_bf16_f32_mn(64, DK, false, true);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                mma_bf16(tmem, tile_desc(smem_u32(TB), 64, 0, ks),
                         desc_mnmajor_sw128(smem_u32(QK) + 8192 + ks * 2048, 16384), id, ks > 0);
            mma_commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 1) ? 1 : 0) != 0;
        tc_fence_after();

        // ---- -W rows -> workspace
        if (ok) {
            const int r = 16 * warp + lane;
#pragma unroll
            for (int cb = 0; cb < DK / 32; ++cb) {
                float w[32];
                tmem_ld32(tmem + lane_base + 32 * cb, w);
                tmem_ld_wait();
                if (lane < 16) {
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
    }
    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ===================================================================== scan

template <int DK>
struct ScanLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int WQ_BYTES = 128 * 128 * KB;          // [128][DK] K-major: -W rows, g Q rows
    static constexpr int WQ = 0;                              // x2
    static constexpr int TZP = WQ + 2 * WQ_BYTES;             // x2 [192][64] K-major: T diag(beta), 0, P
    static constexpr int KR = TZP + 2 * 24576;                // x2 [64 tokens][128] MN-major: kd K
    static constexpr int VR = KR + 2 * 16384;                 // x2 [64 tokens][32] MN-major: V slice
    static constexpr int VK = VR + 2 * 8192;                  // x2 [64 tokens][32] MN-major: kd V (no delta)
    static constexpr int VEC = VK + 2 * 8192;                 // x2 G, g, kd, beta
    static constexpr int UB = VEC + 2 * 1024;                 // [64 tokens][32] MN-major: U (or V)
    static constexpr int UBK = UB + 8192;                     // [64 tokens][32] MN-major: kd U (or kd V)
    static constexpr int SB = UBK + 8192;                     // [DK][32] MN-major: bf16 state slice^T
    static constexpr int BAR = SB + 128 * 128;
    static constexpr int BYTES = BAR + 256;
    static constexpr int ALLOC = BYTES + 1024;
};

// TMEM columns of the scan kernel (fp32 accumulators, 32 columns each)
constexpr uint32_t kS1a = 0, kS1b = 32, kDSa = 64, kDSb = 96, kUt = 128, kPU = 160;
constexpr uint32_t kScanCols = 256;

// Fetch block `blk` of (bh, slice) into buffer `buf`: workspace tiles by bulk
// copy and, for dk >= 64, the q and k rows by tiled TMA (128-byte swizzle,
// zero fill past the end of the sequence), all completing on full[buf]; v
// rows (and q, k rows for dk = 32) by cp.async (one group).
template <int DK, bool DELTA>
__device__ __forceinline__ void scan_fetch(uint8_t *sm, int buf, const bf16 *q, const bf16 *k,
                                           const bf16 *v, const void *tmq, const void *tmk,
                                           const uint8_t *rec, uint64_t *full, size_t bh, int T,
                                           int blk, int dv, int c0, int tid) {
    using L = ScanLayout<DK>;
    using R = Rec<DK>;
    constexpr bool kTma = DK >= 64;
    const int t0 = blk * C;
    uint8_t *wq = sm + L::WQ + buf * L::WQ_BYTES;
    uint8_t *tzp = sm + L::TZP + buf * 24576;
    uint8_t *kr = sm + L::KR + buf * 16384;
    if (tid == 0) {
        const uint32_t bytes = (DELTA ? (uint32_t)R::KB * 8192u + 8192u : 0u) + 8192u + 1024u +
                               (kTma ? 2u * (uint32_t)R::KB * 8192u : 0u);
        mbar_expect_tx(full, bytes);
        if (DELTA) {
#pragma unroll
            for (int kb = 0; kb < R::KB; ++kb)
                bulk_g2s(wq + kb * 16384, rec + R::WT + kb * 8192, 8192, full);
            bulk_g2s(tzp, rec + R::TT, 8192, full);
        }
        bulk_g2s(tzp + 16384, rec + R::PT, 8192, full);
        bulk_g2s(sm + L::VEC + buf * 1024, rec + R::VEC, 1024, full);
        if (kTma) {
#pragma unroll
            for (int kb = 0; kb < R::KB; ++kb) {
                tma_load_3d(wq + kb * 16384 + 8192, tmq, kb * 64, t0, (int)bh, full);
                tma_load_3d(kr + kb * 8192, tmk, kb * 64, t0, (int)bh, full);
            }
        }
    }
    if (!kTma) {
        constexpr int CPR = DK / 8;
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
    }
    uint8_t *vr = sm + L::VR + buf * 8192;
    for (int idx = tid; idx < C * (DVS / 8); idx += NT) {
        const int r = idx / (DVS / 8), ch = idx % (DVS / 8);
        const bool ok = t0 + r < T;
        cp_async16(smem_u32(vr + sw128_offset(r, ch * 8, 64)),
                   v + ((bh * T + (ok ? t0 + r : 0)) * dv + c0 + ch * 8), ok);
    }
    cp_async_commit();
}

// L2 prefetch of everything block `blk` will fetch (one thread).
template <int DK>
__device__ __forceinline__ void scan_prefetch_l2(const bf16 *q, const bf16 *k, const bf16 *v,
                                                 const uint8_t *rec, size_t bh, int T, int blk,
                                                 int dv) {
    const int t0 = blk * C;
    const int n = min(C, T - t0);
    prefetch_l2(rec, Rec<DK>::BYTES);
    prefetch_l2(q + (bh * T + t0) * DK, (uint32_t)n * DK * 2);
    prefetch_l2(k + (bh * T + t0) * DK, (uint32_t)n * DK * 2);
    prefetch_l2(v + (bh * T + t0) * dv, (uint32_t)n * dv * 2);
}

// g Q rows and kd K rows of buffer `buf`, scaled in place.
template <int DK>
__device__ __forceinline__ void scan_scale(uint8_t *sm, int buf, int tid) {
    using L = ScanLayout<DK>;
    uint8_t *wq = sm + L::WQ + buf * L::WQ_BYTES;
    uint8_t *kr = sm + L::KR + buf * 16384;
    const float *vec = reinterpret_cast<const float *>(sm + L::VEC + buf * 1024);
    constexpr int CPR = DK / 8;
    for (int idx = tid; idx < 2 * C * CPR; idx += NT) {
        const int which = idx / (C * CPR);
        const int rem = idx % (C * CPR);
        const int r = rem / CPR, ch = rem % CPR;
        uint4 *p = reinterpret_cast<uint4 *>(which ? kr + sw128_offset(r, ch * 8, 64)
                                                   : wq + sw128_offset(64 + r, ch * 8, 128));
        const float f = vec[(which ? 128 : 64) + r];
        const uint4 raw = *p;
        const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = f * __bfloat162float(e[t]);
        *p = pack8(x);
    }
}

// Scan kernel roles (256 threads):
//   warp 0, lane 0  issues the products on the state chain: S1 = [-W; Q] S^T
//                   and Delta S (and, without delta, Delta S from K^T (kd V))
//   warp 1, lane 0  issues the products off the chain: P U (P V) and the next
//                   block's Ut = T diag(beta) V
//   warps 2, 3      producers: fetch a block into a free buffer (TMA / bulk /
//                   cp.async) and wait for it to land
//   warps 4..7      epilogue (TMEM lanes 0..127): U rows, the state update and
//                   its bf16 copy, the output rows
// Hand-offs are mbarriers; every wait is bounded.  TMEM accumulators are kept
// per block parity so that the output of block b can still be read while
// block b+1 runs.  Every barrier is waited on by all of its consumers before
// it can complete again (so a parity wait is never ambiguous).
constexpr int kScanThreads = 256;
constexpr int kProducers = 64;

// Arrive once per warp on `bar`: every lane has finished its part (and its own
// fences) before lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

struct ScanBars {
    uint64_t ready[2];  // buffer filled                                   (2 producer warps)
    uint64_t full[2];   // loads landed                                    (1 + tx bytes)
    uint64_t empty[2];  // both issuers done with the buffer + epilogue read its gates (2 + 4 warps)
    uint64_t tfree[2];  // output rows of the block with this parity read  (2 warps)
    uint64_t g1;        // S1 products done                                (commit)
    uint64_t ut;        // Ut products done                                (commit)
    uint64_t u;         // U rows written                                  (2 warps)
    uint64_t ds;        // Delta S products done                           (commit)
    uint64_t pu[2];     // P U products of the block with this parity done (commit)
    uint64_t s;         // bf16 state copy written                         (4 warps)
    uint32_t tmem;
};

template <int DK, bool ALPHA, bool DELTA>
__global__ void __launch_bounds__(kScanThreads, 1)
chunk_scan_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                  const bf16 *__restrict__ v, const uint8_t *__restrict__ ws,
                  const float *__restrict__ S0, bf16 *__restrict__ o, float *__restrict__ ST,
                  int H, int T, int dv, int nblk, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk) {
    using L = ScanLayout<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.x * DVS;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const uint8_t *recs = ws + bh * nblk * (size_t)R::BYTES;
    uint8_t *UB = sm + L::UB, *SB = sm + L::SB;
    ScanBars *bars = reinterpret_cast<ScanBars *>(sm + L::BAR);

    // zero everything once: padding rows and columns of the operands must read 0
    for (int i = tid; i < L::BAR / 16; i += kScanThreads)
        reinterpret_cast<uint4 *>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->ready[b], kProducers / 32);
            mbar_init(&bars->full[b], 1);
            mbar_init(&bars->empty[b], 2 + 4);
            mbar_init(&bars->tfree[b], 2);
        }
        mbar_init(&bars->g1, 1);
        mbar_init(&bars->ut, 1);
        mbar_init(&bars->u, 2);
        mbar_init(&bars->ds, 1);
        mbar_init(&bars->pu[0], 1);
        mbar_init(&bars->pu[1], 1);
        mbar_init(&bars->s, 4);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem;
    bool ok = true;

    const uint32_t id_kn = idesc_bf16_f32_mn(128, DVS, false, true);
    const uint32_t id_nn = idesc_bf16_f32_mn(128, DVS, true, true);
    auto wq_desc = [&](int buf) { return tile_desc(smem_u32(sm + L::WQ + buf * L::WQ_BYTES), 128, 0, 0); };
    auto tz_desc = [&](int buf) { return tile_desc(smem_u32(sm + L::TZP + buf * 24576), 192, 0, 0); };
    auto zp_desc = [&](int buf) { return tile_desc(smem_u32(sm + L::TZP + buf * 24576), 192, 64, 0); };
    auto kr_desc = [&](int buf) { return tile_desc_mn(smem_u32(sm + L::KR + buf * 16384), 64, 0); };
    auto vr_desc = [&](int buf) { return tile_desc_mn(smem_u32(sm + L::VR + buf * 8192), 64, 0); };
    auto vk_desc = [&](int buf) { return tile_desc_mn(smem_u32(sm + L::VK + buf * 8192), 64, 0); };

    if (warp == 0) {
        // ================================================ chain products
        if (lane == 0) {
            const uint64_t d_sb = tile_desc_mn(smem_u32(SB), DK, 0);
            const uint64_t d_ubk = tile_desc_mn(smem_u32(sm + L::UBK), 64, 0);
            constexpr int KS = DK / 16, KH = (KS + 1) / 2;
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int buf = blk & 1;
                const uint32_t base = (blk & 1) * 192;
                const uint64_t d_wq = wq_desc(buf), d_kr = kr_desc(buf), d_vk = vk_desc(buf);
                ok = mbar_wait(&bars->ready[buf], (blk >> 1) & 1);
                // accumulators of this parity free: outputs of block blk-2 read
                if (blk >= 2) ok = ok && mbar_wait(&bars->tfree[blk & 1], ((blk >> 1) - 1) & 1);
                ok = ok && mbar_wait(&bars->s, blk & 1);
                if (!ok) break;
                tc_fence_after();
                // S1 = [-W; Q] S^T in two K halves
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                    mma_bf16(tmem + base + (ks < KH ? 0 : 32), kdesc_step(d_wq, 128, ks),
                             mndesc_step(d_sb, ks), id_kn, (ks == 0 || ks == KH) ? 0u : 1u);
                if (DELTA) {
                    mma_commit(&bars->g1);
                    ok = mbar_wait(&bars->u, blk & 1);
                    if (!ok) break;
                    tc_fence_after();
                }
                // Delta S^T = K^T (kd U), or K^T (kd V) without delta; the commit also
                // covers S1, which reads the bf16 state copy the epilogue rewrites
                // once Delta S is done
                const uint64_t d_b = DELTA ? d_ubk : d_vk;
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(tmem + base + (ks < 2 ? 128 : 160), mndesc_step(d_kr, ks),
                             mndesc_step(d_b, ks), id_nn, (ks & 1) ? 1u : 0u);
                mma_commit(&bars->ds);
                mma_commit(&bars->empty[buf]);
            }
        }
    } else if (warp == 1) {
        // ============================================ off-chain products
        if (lane == 0) {
            const uint64_t d_ub = tile_desc_mn(smem_u32(UB), 64, 0);
            auto issue_ut = [&](int blk) {  // Ut = T diag(beta) V  (delta only)
                const int buf = blk & 1;
                const uint64_t d_tz = tz_desc(buf), d_vr = vr_desc(buf);
                const uint32_t col = (blk & 1) * 192 + 64;
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(tmem + col, kdesc_step(d_tz, 192, ks), mndesc_step(d_vr, ks), id_kn,
                             ks > 0);
                mma_commit(&bars->ut);
            };
            if (DELTA && nblk > 0) {
                ok = mbar_wait(&bars->ready[0], 0);
                if (ok) {
                    tc_fence_after();
                    issue_ut(0);
                }
            }
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int buf = blk & 1;
                const uint32_t base = (blk & 1) * 192;
                const uint64_t d_zp = zp_desc(buf);
                if (DELTA) {
                    ok = mbar_wait(&bars->u, blk & 1);
                } else {
                    ok = mbar_wait(&bars->ready[buf], (blk >> 1) & 1);
                    if (blk >= 2) ok = ok && mbar_wait(&bars->tfree[blk & 1], ((blk >> 1) - 1) & 1);
                }
                if (!ok) break;
                tc_fence_after();
                const uint64_t d_x = DELTA ? d_ub : vr_desc(buf);  // U, or V without delta
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_bf16(tmem + base + 96, kdesc_step(d_zp, 192, ks), mndesc_step(d_x, ks),
                             id_kn, ks > 0);
                mma_commit(&bars->pu[blk & 1]);
                mma_commit(&bars->empty[buf]);
                if (DELTA && blk + 1 < nblk) {
                    ok = mbar_wait(&bars->ready[buf ^ 1], ((blk + 1) >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_ut(blk + 1);
                }
            }
        }
    } else if (warp < 4) {
        // ========================================================== producers
        const int pt = tid - 64;
        for (int blk = 0; blk < nblk && ok; ++blk) {
            const int buf = blk & 1;
            if (blk >= 2) ok = mbar_wait(&bars->empty[buf], ((blk >> 1) - 1) & 1);
            ok = __all_sync(0xffffffffu, ok);  // warp-uniform, for the warp-level arrives
            if (!ok) break;
            const int t0 = blk * C;
            const uint8_t *rec = recs + (size_t)blk * R::BYTES;
            uint8_t *wq = sm + L::WQ + buf * L::WQ_BYTES;
            uint8_t *tzp = sm + L::TZP + buf * 24576;
            uint8_t *kr = sm + L::KR + buf * 16384;
            uint8_t *vr = sm + L::VR + buf * 8192;
            constexpr bool kTma = DK >= 64;
            if (pt == 0) {
                if (blk + 2 < nblk) scan_prefetch_l2<DK>(q, k, v, rec + 2 * R::BYTES, bh, T, blk + 2, dv);
                const uint32_t bytes = (DELTA ? (uint32_t)R::KB * 8192u + 8192u : 0u) + 8192u +
                                       1024u + (kTma ? 2u * (uint32_t)R::KB * 8192u : 0u);
                mbar_expect_tx(&bars->full[buf], bytes);
                if (DELTA) {
#pragma unroll
                    for (int kb = 0; kb < R::KB; ++kb)
                        bulk_g2s(wq + kb * 16384, rec + R::WT + kb * 8192, 8192, &bars->full[buf]);
                    bulk_g2s(tzp, rec + R::TT, 8192, &bars->full[buf]);
                }
                bulk_g2s(tzp + 16384, rec + R::PT, 8192, &bars->full[buf]);
                bulk_g2s(sm + L::VEC + buf * 1024, rec + R::VEC, 1024, &bars->full[buf]);
                if (kTma) {
#pragma unroll
                    for (int kb = 0; kb < R::KB; ++kb) {
                        tma_load_3d(wq + kb * 16384 + 8192, &tmq, kb * 64, t0, (int)bh,
                                    &bars->full[buf]);
                        tma_load_3d(kr + kb * 8192, &tmk, kb * 64, t0, (int)bh, &bars->full[buf]);
                    }
                }
            }
            if (!kTma) {
                constexpr int CPR = DK / 8;
                for (int idx = pt; idx < 2 * C * CPR; idx += kProducers) {
                    const int which = idx / (C * CPR);
                    const int rem = idx % (C * CPR);
                    const int r = rem / CPR, ch = rem % CPR;
                    const bool okr = t0 + r < T;
                    const bf16 *src = (which ? k : q) + ((bh * T + (okr ? t0 + r : 0)) * DK + ch * 8);
                    const uint32_t dst = which ? smem_u32(kr + sw128_offset(r, ch * 8, 64))
                                               : smem_u32(wq + sw128_offset(64 + r, ch * 8, 128));
                    cp_async16(dst, src, okr);
                }
            }
            for (int idx = pt; idx < C * (DVS / 8); idx += kProducers) {
                const int r = idx / (DVS / 8), ch = idx % (DVS / 8);
                const bool okr = t0 + r < T;
                cp_async16(smem_u32(vr + sw128_offset(r, ch * 8, 64)),
                           v + ((bh * T + (okr ? t0 + r : 0)) * dv + c0 + ch * 8), okr);
            }
            cp_async_commit();
            cp_async_wait_all();
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[buf], (blk >> 1) & 1));
            if (!ok) break;
            if (!DELTA) {
                // kd V (B operand of Delta S = K^T diag(kd) V); g and kd are folded
                // into the epilogues everywhere else
                const float *vec = reinterpret_cast<const float *>(sm + L::VEC + buf * 1024);
                uint8_t *vk = sm + L::VK + buf * 8192;
                for (int idx = pt; idx < C * (DVS / 8); idx += kProducers) {
                    const int r = idx / (DVS / 8), ch = idx % (DVS / 8);
                    const uint32_t off = sw128_offset(r, ch * 8, 64);
                    const uint4 raw = *reinterpret_cast<const uint4 *>(vr + off);
                    const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
                    const float f = vec[128 + r];
                    float x[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) x[t] = f * __bfloat162float(e[t]);
                    *reinterpret_cast<uint4 *>(vk + off) = pack8(x);
                }
            }
            fence_async_smem();
            warp_arrive(&bars->ready[buf]);
        }
    } else {
        // =========================================================== epilogue
        const int j = tid - 128;  // TMEM lane; key channel of the state column
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        float Sr[DVS];
#pragma unroll
        for (int c = 0; c < DVS; ++c) Sr[c] = (S0 && j < DK) ? S0[(bh * dv + c0 + c) * DK + j] : 0.f;
        if (j < DK) {
#pragma unroll
            for (int c8 = 0; c8 < DVS / 8; ++c8)
                *reinterpret_cast<uint4 *>(SB + sw128_offset(j, c8 * 8, DK)) = pack8(Sr + c8 * 8);
        }
        fence_async_smem();
        warp_arrive(&bars->s);
        for (int blk = 0; blk < nblk && ok; ++blk) {
            const int buf = blk & 1, p = blk & 1;
            const uint32_t base = p * 192;
            const int t0 = blk * C;
            const int n = min(C, T - t0);
            // gates of this block, read before the buffer is released: g_C for
            // the state, g_r of this thread's output row, kd_i of its U row
            const float *vec = reinterpret_cast<const float *>(sm + L::VEC + buf * 1024);
            float gC, gr = 0.f, kdi = 0.f;
            if (DELTA) {
                ok = mbar_wait(&bars->g1, blk & 1);
                if (warp < 6) ok = ok && mbar_wait(&bars->ut, blk & 1);  // only the U rows need Ut
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                gC = vec[64 + C - 1];
                if (warp >= 6) gr = vec[64 + j - 64];
                else kdi = vec[128 + j];
                warp_arrive(&bars->empty[buf]);
                if (warp < 6) {  // U rows = tokens 0..63
                    float u[32], x[32];
                    tmem_ld32(tmem + lane_base + base + 64, u);
                    tmem_ld32(tmem + lane_base + base + 0, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) u[c] += x[c];
                    tmem_ld32(tmem + lane_base + base + 32, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) u[c] += x[c];
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        *reinterpret_cast<uint4 *>(UB + sw128_offset(j, c8 * 8, 64)) =
                            pack8(u + c8 * 8);
#pragma unroll
                    for (int c = 0; c < 32; ++c) u[c] *= kdi;
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        *reinterpret_cast<uint4 *>(sm + L::UBK + sw128_offset(j, c8 * 8, 64)) =
                            pack8(u + c8 * 8);
                    fence_async_smem();
                    tc_fence_before();
                    warp_arrive(&bars->u);
                }
            }
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->ds, blk & 1));
            if (!ok) break;
            tc_fence_after();
            if (!DELTA) {
                gC = vec[64 + C - 1];
                if (warp >= 6) gr = vec[64 + j - 64];
                warp_arrive(&bars->empty[buf]);
            }
            {
                float d[32], e[32];
                tmem_ld32(tmem + lane_base + base + 128, d);
                tmem_ld32(tmem + lane_base + base + 160, e);
                tmem_ld_wait();
                if (j < DK) {
#pragma unroll
                    for (int c = 0; c < DVS; ++c) Sr[c] = gC * Sr[c] + d[c] + e[c];
#pragma unroll
                    for (int c8 = 0; c8 < DVS / 8; ++c8)
                        *reinterpret_cast<uint4 *>(SB + sw128_offset(j, c8 * 8, DK)) =
                            pack8(Sr + c8 * 8);
                }
                fence_async_smem();
                tc_fence_before();
                warp_arrive(&bars->s);
            }
            if (warp >= 6) {  // output rows = tokens 0..63
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->pu[p], (blk >> 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const int r = j - 64;
                float d[32], e[32];
                tmem_ld32(tmem + lane_base + base + 0, d);
                tmem_ld32(tmem + lane_base + base + 32, e);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) d[c] = gr * (d[c] + e[c]);  // g_r Q S^T
                tmem_ld32(tmem + lane_base + base + 96, e);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) d[c] += e[c];              // + P U
                tc_fence_before();
                warp_arrive(&bars->tfree[p]);
                if (r < n) {
                    uint4 *dst = reinterpret_cast<uint4 *>(o + (bh * T + t0 + r) * dv + c0);
#pragma unroll
                    for (int i8 = 0; i8 < 4; ++i8) dst[i8] = pack8(d + i8 * 8);
                }
            }
        }
        if (ok && j < DK) {
#pragma unroll
            for (int c = 0; c < DVS; ++c) ST[(bh * dv + c0 + c) * DK + j] = Sr[c];
        }
    }

    if (!ok) atomicExch(&g_tc_error, 1);
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================== launch

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [B*H][T][d] bf16 tensor, boxes of 64 rows x 64 columns, 128-byte swizzle,
// zero fill outside.
cudaError_t make_rows_map(CUtensorMap *m, const void *base, int d, int T, int BH) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)T};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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
    CUtensorMap tmq, tmk;
    memset(&tmq, 0, sizeof(tmq));
    memset(&tmk, 0, sizeof(tmk));
    if (DK >= 64) {
        e = make_rows_map(&tmq, q, DK, T, B * H);
        if (e != cudaSuccess) return e;
        e = make_rows_map(&tmk, k, DK, T, B * H);
        if (e != cudaSuccess) return e;
    }
    prep<<<dim3(nblk, H, B), NT, PrepLayout<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), ALPHA ? alpha : nullptr,
        DELTA ? beta : nullptr, static_cast<uint8_t *>(ws), H, T, nblk, tmq, tmk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    scan<<<dim3(dv / DVS, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), static_cast<const bf16 *>(v),
        static_cast<const uint8_t *>(ws), S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk, tmq,
        tmk);
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
