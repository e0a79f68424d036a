// Chunked forward on the tensor cores (tcgen05 + TMEM), bf16 operands with
// fp32 accumulation and an fp32 state.
//
// Chunkwise form (page "Le architetture lineari: RetNet, RWKV, xLSTM",
// section "RetNet: la retention e le sue tre forme"): blocks of C = 64
// tokens, only the end-of-block state handed to the next block.  Inside block
// j, with G_r = sum_{i<=r} ln alpha_i (gate products, computable for all
// steps at once -- page "Scrivere meglio nella memoria: gate e delta rule",
// section "Correggere: la delta rule"), g_r = e^{G_r}, kd_i = e^{G_C - G_i},
// g_C = e^{G_C} and S_j the state when the block starts:
//
//   P_j = (Q K^T) (.) M,        M_ri = e^{G_r - G_i} for i <= r        (scores)
//   A_j = strict_lower(diag(beta) (K K^T) (.) M)                       (delta couplings)
//   T_j = (I + A_j)^-1          unit lower triangular (the WY / UT step)
//   W_j = T_j diag(beta g) K,   Ut_j = T_j diag(beta) V
//   U_j = Ut_j - W_j S_j^T      pseudo-values u_r of the WY representation
//   O_j = diag(g) Q S_j^T + P_j U_j
//   S_{j+1} = g_C S_j + U_j^T diag(kd) K
// and without the delta term U = V.  The derivation: the gated recurrence
// unrolled inside a block gives u_r = beta_r (v_r - g_r S k_r -
// sum_{i<r} e^{G_r - G_i} (k_i.k_r) u_i), a unit-lower-triangular system.
//
// Look-ahead form used by the scan.  Substituting the state update into the
// next block's U gives
//   U_{j+1} = Ut_{j+1} - g_C W_{j+1} S_j^T - Z_j U_j,
//   Z_j = W_{j+1} K_j^T diag(kd_j)          (64 x 64, independent of the state)
// so one accumulator D_{j+1} (M = 128 rows) collects
//   rows  0..63:  [T diag(beta)]_{j+1} V_{j+1} + (-g_C W_{j+1}) S_j^T + (-Z_j) U_j  = U_{j+1}
//   rows 64..127:                                   Q_j S_j^T  +  P_j U_j         (O_j before g)
// from three products whose A operands stack a row block of block j+1 on a
// row block of block j.  The loop-carried chain is then U_j -> one K = 64
// product -> U_{j+1}; the state update S_{j+1} = g_C S_j + K_j^T (kd U_j)
// runs beside it and is needed one block later.
//
// Two launches:
//  * prep: one CTA per (block, head, batch), all blocks in parallel.  Computes
//    what does not depend on the state: the gates, the scores P, the UT
//    inverse T (fp32, in place; 16 x 16 diagonal blocks on the CUDA cores,
//    then 32 x 32 and 64 x 64 block inversion on warp-level tf32 MMAs), W and
//    Z, and writes the workspace record of "stage" j: W_j, T_j diag(beta),
//    -Z_{j-1}, P_{j-1} and the gate vectors, as bf16 tiles already in the
//    shared-memory operand layout (primes: the previous block).  Stage j's P
//    row block is written by the CTA of block j-1; there is one more stage
//    than blocks.
//  * scan: one CTA per (32 value channels, head, batch); rows of S evolve
//    independently given k, alpha and beta, so slices never exchange data.
//    It walks the stages in order with warp-specialised roles (below).
//
// Every product runs as an M = 128 tcgen05.mma with 128-byte-swizzled
// shared-memory operands and an fp32 accumulator in tensor memory:
//   prep  E1  [Q; K] K^T              -> [Q K^T ; K K^T]
//         E3  T diag(beta g) K        -> W           (M = 64, K read MN-major)
//         E4  W K'^T                  -> Z'          (M = 64)
//   scan  a   [T diag(beta); *] V     -> Ut rows
//         b   [W; Q'] S'^T            -> U (times -g_C') and O' parts
//         c   [-Z'; P'] U'            -> U and O' parts
//         ds  K'^T (kd' U')           -> Delta S'^T  (K read MN-major)
// A final short block is zero-filled (alpha treated as 1, beta as 0), which
// leaves the real tokens' results unchanged.
//
// The lr_fuse maps live in prep (page "Scrivere meglio nella memoria: gate e
// delta rule"), in a separate instantiation so the plain path is untouched.
// The gates are mapped as they are read.  SiLU + L2 of q and k: each thread
// takes one row of the staged [Q; K] tile through SiLU in place (fp32, one
// rounding to bf16) and keeps the row's inverse L2 norm in fp32; the norms
// are never applied to the tiles but folded into the per-row and per-column
// factors every product is already scaled by:
//   P_ri  *= 1/|q_r| 1/|k_i|        A_ri *= 1/|k_r| 1/|k_i|      (E2)
//   W = T diag(beta g / |k|) K~                                     (E3)
//   -Z' diag(kd' / |k'|)                                           (E4)
//   record vectors g' / |q'| (output rows) and kd / |k| (the kd U rows)
// so that every result equals the one with normalised q and k.  The CTA
// writes its SiLU'd q and k rows to the workspace by TMA stores and the scan
// reads them there unchanged; the previous block's k rows, staged again for
// E4, go through the same SiLU, so they match the stored copy bit for bit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_internal.cuh"
#include "scan_tc.cuh"

namespace lr {
namespace {

constexpr int NT = 128;    // threads per prep CTA
constexpr int AP = C + 4;  // fp32 row of A and T: 16-byte rows, 8-row groups on distinct banks
constexpr int XS = 40;     // fp32 row of the solve scratch

// ===================================================================== prep

// Shared memory of a prep CTA, with the regions reused as the block goes:
//   QK  [128 rows][DK] K-major: Q rows 0..63 and K rows 64..127 (E1); then
//       the Q rows host the T diag(beta g) tile and the solve scratch, and
//       after E3 the K rows are refilled with the previous block's K rows (E4)
//   AT  fp32 [64][AP]: A, inverted in place into T; then bf16 W [64][DK]
// 51 KB at d_k = 128: four CTAs per SM.
template <int DK>
struct PrepLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int QK = 0;
    static constexpr int TB = QK;                           // [64][64] bf16, in the Q rows of block 0
    static constexpr int XT = TB;                           // fp32 [32][XS] solve scratch, inside TB
    static constexpr int AT = QK + 128 * 128 * KB;
    static constexpr int VEC = AT + C * AP * 4;             // G (later kd'), ginv, g, beta,
                                                            // 1/|q|, 1/|k|, 1/|k'| (maps)
    static constexpr int BAR = VEC + 7 * 64 * 4;            // 3 barriers, TMEM slot
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};
static_assert(32 * XS * 4 <= 8192, "solve scratch must fit inside the T tile");
static_assert(128 * 64 * 2 <= C * AP * 4, "the W tile must fit over the A matrix");
static_assert(PrepLayout<128>::AT % 1024 == 0, "the W tile must be 1024-byte aligned");

// Thread 0 waits on `bar` (when `ok`) while the rest of the CTA is parked
// at the barrier, which issues nothing; returns the CTA-wide outcome.
// Reads of what the barrier guarded are ordered after it by the CTA
// barrier (callers add tcgen05.fence::after_thread_sync before TMEM reads).
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, bool ok) {
    bool w = ok;
    if (threadIdx.x == 0 && ok) w = mbar_wait(bar, parity);
    tc_fence_before();
    return __syncthreads_and(w ? 1 : 0) != 0;
}

// Element (r, c) of a 64 x 64 fp32 matrix in shared memory, rows padded to
// AP floats.
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
// A fragment of the rows r0..r0+15, columns c0..c0+7 (c0 % 4 == 0) of a fp32
// matrix with row stride AP, rounded to tf32.  ldmatrix.x4 on 32-bit data:
// each 8 x 8 b16 matrix is 8 rows x 4 floats, and thread (g, t) receives
// element (g, t) of each of the four 8 x 4 quarters.
__device__ __forceinline__ void lda_tf32(uint32_t (&a)[4], const float *m, int r0, int c0,
                                         int lane) {
    const int q = lane >> 3, rr = lane & 7;
    const float *p = m + (r0 + rr + 8 * (q & 1)) * AP + c0 + 4 * (q >> 1);
    uint32_t v[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(smem_u32(p)));
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = to_tf32(__uint_as_float(v[i]));
}

// T = (I + A)^-1 for a strictly lower A (64 x 64, fp32 in shared memory),
// computed in place by block inversion: with A = [A11 0; A21 A22],
//   T = [T11 0; -T22 A21 T11  T22],
// applied to the 16 x 16 diagonal blocks (CUDA cores, fp32), then to the two
// 32 x 32 diagonal blocks, then to the whole (tf32 warp-level MMAs with fp32
// accumulation).  On exit AT holds T's lower triangle; the blocks above the
// block diagonal keep A's zeros.  Xt is a 32 x XS fp32 scratch.
__device__ __forceinline__ void ut_inverse(float *AT, float *Xt, int tid) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    // ---- 16 x 16 diagonal blocks: thread (b, c) solves column c of block b
    float x[16];
    const int b = tid >> 4, c = tid & 15;
    if (tid < 64) {
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float s0 = (rr == c) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < rr; ++i) {
                const float a = AT[sw64(16 * b + rr, 16 * b + i)];
                if (i & 1) s1 -= a * x[i];
                else s0 -= a * x[i];
            }
            x[rr] = s0 + s1;
        }
    }
    __syncthreads();  // every diagonal block of A read before T replaces it
    if (tid < 64) {
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) AT[sw64(16 * b + rr, 16 * b + c)] = x[rr];
    }
    __syncthreads();
    // ---- 32 x 32 diagonal blocks: T[R, C] = -T[R, R] A[R, C] T[C, C] for the
    //      16-row blocks (R, C) = (1, 0) and (3, 2); warp w: pair w/2, column tile w%2
    {
        const int pr = warp >> 1, nt = warp & 1;
        const int R = 32 * pr + 16, Cc = 32 * pr;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kk = nt; kk < 2; ++kk) {  // rows of T[C, C] above 8 nt are zero in this tile
            uint32_t a[4];
            lda_tf32(a, AT, R, Cc + 8 * kk, lane);
            mma_tf32(d, a, to_tf32(AT[sw64(Cc + 8 * kk + t, Cc + 8 * nt + g)]),
                     to_tf32(AT[sw64(Cc + 8 * kk + t + 4, Cc + 8 * nt + g)]));
        }
        float *xw = Xt + (16 * pr) * XS + 8 * nt;  // this warp's 16 x 8 tile of X
        xw[g * XS + 2 * t] = d[0];
        xw[g * XS + 2 * t + 1] = d[1];
        xw[(g + 8) * XS + 2 * t] = d[2];
        xw[(g + 8) * XS + 2 * t + 1] = d[3];
        __syncwarp();
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t a[4];
            lda_tf32(a, AT, R, R + 8 * kk, lane);
            mma_tf32(e, a, to_tf32(xw[(8 * kk + t) * XS + g]),
                     to_tf32(xw[(8 * kk + t + 4) * XS + g]));
        }
        __syncthreads();  // both column tiles have read A[R, C]
        AT[sw64(R + g, Cc + 8 * nt + 2 * t)] = -e[0];
        AT[sw64(R + g, Cc + 8 * nt + 2 * t + 1)] = -e[1];
        AT[sw64(R + g + 8, Cc + 8 * nt + 2 * t)] = -e[2];
        AT[sw64(R + g + 8, Cc + 8 * nt + 2 * t + 1)] = -e[3];
    }
    __syncthreads();
    // ---- whole matrix: X = A21 T11 (32 x 32) to the scratch; warp w takes the
    //      tiles (w%2, w/2) and (1 - w%2, 3 - w/2), five k steps in all
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int mt = h ? 1 - (warp & 1) : (warp & 1);
        const int nt = h ? 3 - (warp >> 1) : (warp >> 1);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kk = nt; kk < 4; ++kk) {  // rows of T11 above 8 nt are zero in this tile
            uint32_t a[4];
            lda_tf32(a, AT, 32 + 16 * mt, 8 * kk, lane);
            mma_tf32(d, a, to_tf32(AT[sw64(8 * kk + t, 8 * nt + g)]),
                     to_tf32(AT[sw64(8 * kk + t + 4, 8 * nt + g)]));
        }
        float *xw = Xt + (16 * mt) * XS + 8 * nt;
        xw[g * XS + 2 * t] = d[0];
        xw[g * XS + 2 * t + 1] = d[1];
        xw[(g + 8) * XS + 2 * t] = d[2];
        xw[(g + 8) * XS + 2 * t + 1] = d[3];
    }
    __syncthreads();  // X complete, A21 no longer read
    //      T21 = -T22 X: warp w takes column tile w, both row tiles
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int nt = warp;
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kk = 0; kk < 2 * mt + 2; ++kk) {  // T22 row tile mt is zero right of 16 (mt + 1)
            uint32_t a[4];
            lda_tf32(a, AT, 32 + 16 * mt, 32 + 8 * kk, lane);
            mma_tf32(e, a, to_tf32(Xt[(8 * kk + t) * XS + 8 * nt + g]),
                     to_tf32(Xt[(8 * kk + t + 4) * XS + 8 * nt + g]));
        }
        AT[sw64(32 + 16 * mt + g, 8 * nt + 2 * t)] = -e[0];
        AT[sw64(32 + 16 * mt + g, 8 * nt + 2 * t + 1)] = -e[1];
        AT[sw64(32 + 16 * mt + g + 8, 8 * nt + 2 * t)] = -e[2];
        AT[sw64(32 + 16 * mt + g + 8, 8 * nt + 2 * t + 1)] = -e[3];
    }
    __syncthreads();
}

// SiLU(x) = x sigmoid(x) = h + h tanh(h), h = x / 2, with the hardware tanh
// approximation (one special-function operation per element).  Its error,
// about 2^-11 relative to tanh, makes an absolute error of about 2^-12 |x| in
// SiLU: below a bf16 rounding of the result for x > -1, larger relative to
// the small values SiLU takes far below 0 (about 1.4 % at x = -4), which
// carry little weight after the L2 normalisation.
__device__ __forceinline__ float silu_fast(float x) {
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// SiLU of columns [c0, c0 + ncol) (multiples of 8) of row `row` of a bf16
// K-major 128-byte-swizzled tile of `rows` rows (sw128_offset layout), in
// place (fp32, rounded once to bf16); returns the sum of squares of the fp32
// values.  Zero entries stay zero.
template <int NCOL>
__device__ __forceinline__ float silu_cols(uint8_t *tile, int row, int rows, int c0) {
    uint8_t *base = tile + row * 128;
    float ss = 0.f;
#pragma unroll 4
    for (int c = 0; c < NCOL / 8; ++c) {
        const int k = c0 + 8 * c, kb = k >> 6, ch = (k & 63) >> 3;
        {
            uint4 *p = reinterpret_cast<uint4 *>(base + kb * rows * 128 + ((ch ^ (row & 7)) << 4));
            const uint4 raw = *p;
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            float x[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = silu_fast(__uint_as_float(w[i] << 16));
                x[2 * i + 1] = silu_fast(__uint_as_float(w[i] & 0xffff0000u));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
            *p = pack8(x);
        }
    }
    return ss;
}

// Prep of block j = blockIdx.x.  Writes to record j: W_j, T_j diag(beta),
// -Z_{j-1} and the gate vectors; to record j+1: P_j (and, for the last block,
// record j+1's gate vectors).  MAPS 1: the gate maps of `fz`; MAPS 2: also
// SiLU + L2 of q and k, with the block's SiLU'd q and k rows written through
// tmqn and tmkn.  With maps every block also writes record j+1's
// previous-block vectors (they carry the norms).
template <int DK, bool ALPHA, bool DELTA, int MAPS>
__global__ void __launch_bounds__(NT)
chunk_prep_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                  const float *__restrict__ alpha, const float *__restrict__ beta,
                  uint8_t *__restrict__ ws, int H, int T, int nblk,
                  const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const Fuse fz, const __grid_constant__ CUtensorMap tmqn,
                  const __grid_constant__ CUtensorMap tmkn) {
    using L = PrepLayout<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = blk * C;
    const int n = min(C, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + blk) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    float *vec = reinterpret_cast<float *>(rec + R::VEC);
    float *vec_next = reinterpret_cast<float *>(rec_next + R::VEC);

    uint8_t *QK = sm + L::QK, *TB = sm + L::TB, *WB = sm + L::AT;
    float *Am = reinterpret_cast<float *>(sm + L::AT);  // A, then T in place
    float *Xt = reinterpret_cast<float *>(sm + L::XT);
    float *Gv = reinterpret_cast<float *>(sm + L::VEC);
    float *giv = Gv + 64, *gv = Gv + 128, *bv = Gv + 192;
    float *kdv = Gv;  // kd of the previous block, once G is no longer needed
    float *inq = Gv + 256, *ink = Gv + 320, *inkp = Gv + 384;  // inverse norms (maps)
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);  // MMA, q/k tiles, previous k tile
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 32);
    const bool zprev = DELTA && blk > 0;  // Z_{j-1} exists
    // gate inputs first, so their global-load latency overlaps the staging:
    // threads 0-63 this block's tokens, 64-127 the previous block's
    const int tok = tid & 63;
    const unsigned fl = MAPS ? fz.flags : 0u;
    constexpr bool qk = MAPS == 2;
    float araw = 1.f, b = 0.f;
    if (tid < C) {
        if (tok < n) {
            if (ALPHA) araw = alpha[bh * T + t0 + tok];
            if (DELTA) b = beta[bh * T + t0 + tok];
            if (MAPS && DELTA) b = write_strength(fl, b);
        }
    } else if (ALPHA && blk > 0) {
        araw = alpha[bh * T + t0 - C + tok];
    }

    // ---- stage Q, K by tiled TMA (zero-filled past the end of the sequence
    //      and, for d_k = 32, in the outer half of the 64-column box)
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[1], 2u * (uint32_t)L::KB * 8192u);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
            tma_load_3d(QK + kb * 16384, &tmq, kb * 64, t0, (int)bh, &bar[1]);
            tma_load_3d(QK + kb * 16384 + 8192, &tmk, kb * 64, t0, (int)bh, &bar[1]);
        }
    }
    // ---- gates: warps 0-1 hold this block's tokens, warps 2-3 the previous
    //      block's (all ones for block 0)
    float la = ALPHA ? __logf(araw) : 0.f;
    if (MAPS) {
        const bool has_a = ALPHA && (tid < C ? tok < n : blk > 0);
        la = has_a ? log_gate(fl, araw, (fl & kScaledAlphaMaps) ? fz.ascale[blockIdx.y] : 0.f)
                   : 0.f;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    float incl = la;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    Am[tid] = incl;  // scratch (A is written only after E1)
    __syncthreads();
    const int pb = tid & 64;
    const float G = incl + ((tid & 32) ? Am[pb + 31] : 0.f);
    const float Glast = Am[pb + 31] + Am[pb + 63];
    // exp(G_r - G_i) = g_r * ginv_i when exp(-G_63) is finite in fp32
    const bool factor = !ALPHA || Am[31] + Am[63] > -80.f;
    float kdp = 1.f, my_g = 1.f, my_kd = 1.f;
    if (tid < C) {
        const float g = ALPHA ? __expf(G) : 1.f;
        const float kd = ALPHA ? __expf(Glast - G) : 1.f;
        Gv[tok] = G;
        gv[tok] = g;
        giv[tok] = ALPHA ? __expf(-G) : 1.f;
        bv[tok] = b;
        my_g = g;
        my_kd = kd;
        if (!MAPS) {
            vec[kVkd + tok] = kd;
            if (blk == nblk - 1) {  // the stage after the last block reads this block as its previous one
                vec_next[kVgPrev + tok] = g;
                vec_next[kVkdPrev + tok] = kd;
                if (tok == C - 1) vec_next[kVgCPrev] = ALPHA ? __expf(Glast) : 1.f;
            }
        }
    } else {
        const float g = ALPHA ? __expf(G) : 1.f;
        kdp = ALPHA ? __expf(Glast - G) : 1.f;
        // with the maps record j's previous-block vectors come from the CTA of
        // block j-1 (they carry its norms); stage 0 has no previous block
        if (!MAPS || blk == 0) {
            vec[kVgPrev + tok] = g;
            vec[kVkdPrev + tok] = kdp;
            if (tok == C - 1) {
                const float gc = ALPHA ? __expf(Glast) : 1.f;
                vec[kVgCPrev] = gc;
            }
        }
    }
    bool ok = mbar_wait(&bar[1], 0);
    if (qk && ok) {  // thread t: row t of [Q; K]
        const float in = inv_l2(silu_cols<DK>(QK, tid, 128, 0));
        if (tid < C) inq[tid] = in;
        else ink[tok] = in;
        fence_async_smem();
    }
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    if (MAPS && tid < C) {  // the vectors that carry this block's norms
        const float sq = qk ? inq[tok] : 1.f, sk = qk ? ink[tok] : 1.f;
        vec[kVkd + tok] = my_kd * sk;
        vec_next[kVgPrev + tok] = my_g * sq;
        vec_next[kVkdPrev + tok] = my_kd * sk;
        if (tok == C - 1) vec_next[kVgCPrev] = ALPHA ? __expf(Glast) : 1.f;
    }
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    // ---- E1: [Q; K] K^T -> TMEM cols [0, 64)
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(QK), 128, 0, ks), tile_desc(smem_u32(QK), 128, 64, ks),
                     id, ks > 0);
        mma_commit(&bar[0]);
        if (qk) {  // the SiLU'd rows -> workspace (rows past T are not written)
#pragma unroll
            for (int kb = 0; kb < L::KB; ++kb) {
                tma_store_3d(&tmqn, QK + kb * 16384, kb * 64, t0, (int)bh);
                tma_store_3d(&tmkn, QK + kb * 16384 + 8192, kb * 64, t0, (int)bh);
            }
            bulk_commit();
        }
    }
    ok = __syncthreads_and((ok && mbar_wait(&bar[0], 0)) ? 1 : 0) != 0;
    tc_fence_after();

    // ---- E2: P rows (bf16 tile to the next stage's record), A rows (fp32)
    if (ok) {
        const int r = 32 * (warp & 1) + lane;
        const bool is_q = warp < 2;
        const float Gr = Gv[r], gr = gv[r];
        const float rs = qk ? (is_q ? inq[r] : ink[r]) : 1.f;  // 1/|q_r| or 1/|k_r|
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float a[32];
            tmem_ld32(tmem + lane_base + 32 * half, a);
            tmem_ld_wait(a);
            float gi[32];  // 1 / g of the key tokens of this half
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 v4 = reinterpret_cast<const float4 *>(giv + half * 32)[e4];
                gi[4 * e4] = v4.x;
                gi[4 * e4 + 1] = v4.y;
                gi[4 * e4 + 2] = v4.z;
                gi[4 * e4 + 3] = v4.w;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = half * 32 + e;
                const float dec = !ALPHA ? 1.f : (factor ? gr * gi[e] : __expf(Gr - Gv[i]));
                a[e] = (i <= r && (is_q || i < r)) ? a[e] * dec : 0.f;
            }
            if (qk) {  // the norms: 1/|q_r| (or 1/|k_r|) times 1/|k_i|
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 v4 = reinterpret_cast<const float4 *>(ink + half * 32)[e4];
                    a[4 * e4] *= rs * v4.x;
                    a[4 * e4 + 1] *= rs * v4.y;
                    a[4 * e4 + 2] *= rs * v4.z;
                    a[4 * e4 + 3] *= rs * v4.w;
                }
            }
            if (is_q) {
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8)
                    *reinterpret_cast<uint4 *>(rec_next + R::TZP +
                                               sw128_offset(128 + r, half * 32 + i8 * 8, 192)) =
                        pack8(a + i8 * 8);
            } else if (DELTA) {
                const float br = bv[r];
                float4 *row = reinterpret_cast<float4 *>(Am + sw64(r, half * 32));
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4)
                    row[e4] = make_float4(br * a[4 * e4], br * a[4 * e4 + 1], br * a[4 * e4 + 2],
                                          br * a[4 * e4 + 3]);
            }
        }
    }
    if (qk && tid == 0) bulk_wait_read();  // the stores have read the [Q; K] tile (reused below)
    tc_fence_before();  // the score columns are reused by W below
    __syncthreads();

    if (DELTA && ok) {
        if (tid >= C) kdv[tok] = kdp;  // G is dead; read after the syncs below
        ut_inverse(Am, Xt, tid);
        // T diag(beta) (bf16) -> record; T diag(beta g) -> the T tile (over the
        // solve scratch), the A operand of W = T diag(beta g) K
        for (int idx = tid; idx < C * 8; idx += NT) {
            const int r = idx >> 3, i8 = idx & 7;
            float t[8], tg[8], tv[8], bb[8], gg[8];
            *reinterpret_cast<float4 *>(tv) =
                *reinterpret_cast<const float4 *>(Am + sw64(r, i8 * 8));
            *reinterpret_cast<float4 *>(tv + 4) =
                *reinterpret_cast<const float4 *>(Am + sw64(r, i8 * 8 + 4));
            *reinterpret_cast<float4 *>(bb) = reinterpret_cast<const float4 *>(bv)[2 * i8];
            *reinterpret_cast<float4 *>(bb + 4) = reinterpret_cast<const float4 *>(bv)[2 * i8 + 1];
            *reinterpret_cast<float4 *>(gg) = reinterpret_cast<const float4 *>(gv)[2 * i8];
            *reinterpret_cast<float4 *>(gg + 4) = reinterpret_cast<const float4 *>(gv)[2 * i8 + 1];
            if (qk) {  // W = T diag(beta g / |k|) K~
                const float4 k0 = reinterpret_cast<const float4 *>(ink)[2 * i8];
                const float4 k1 = reinterpret_cast<const float4 *>(ink)[2 * i8 + 1];
                gg[0] *= k0.x, gg[1] *= k0.y, gg[2] *= k0.z, gg[3] *= k0.w;
                gg[4] *= k1.x, gg[5] *= k1.y, gg[6] *= k1.z, gg[7] *= k1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = i8 * 8 + e;
                t[e] = i <= r ? tv[e] * bb[e] : 0.f;
                tg[e] = t[e] * gg[e];
            }
            *reinterpret_cast<uint4 *>(rec + R::TZP + sw128_offset(r, i8 * 8, 192)) = pack8(t);
            *reinterpret_cast<uint4 *>(TB + sw128_offset(r, i8 * 8, 64)) = pack8(tg);
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
            mma_commit(&bar[0]);
        }
        ok = __syncthreads_and(mbar_wait(&bar[0], 1) ? 1 : 0) != 0;
        tc_fence_after();

        // ---- the K rows are free: fetch the previous block's K rows there (for Z)
        if (zprev && ok && tid == 0) {
            mbar_expect_tx(&bar[2], (uint32_t)L::KB * 8192u);
#pragma unroll
            for (int kb = 0; kb < L::KB; ++kb)
                tma_load_3d(QK + kb * 16384 + 8192, &tmk, kb * 64, t0 - C, (int)bh, &bar[2]);
        }

        // ---- W rows (bf16) -> the W tile over T: the A operand of Z and, by one
        //      bulk copy, the record's W tile (same layout)
        if (ok) {
            const int r = 16 * warp + lane;
#pragma unroll
            for (int cb = 0; cb < DK / 32; ++cb) {
                float w[32];
                tmem_ld32(tmem + lane_base + 32 * cb, w);
                tmem_ld_wait(w);
                if (lane < 16) {
#pragma unroll
                    for (int i8 = 0; i8 < 4; ++i8)
                        *reinterpret_cast<uint4 *>(WB + sw128_offset(r, cb * 32 + i8 * 8, 64)) =
                            pack8(w + i8 * 8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        tc_fence_after();
        if (tid == 0 && ok) {
            bulk_s2g(rec + R::WT, WB, (uint32_t)R::KB * 8192u);
            bulk_commit();
        }

        // ---- E4: Z' = W K'^T (M = 64, N = 64 previous tokens, K = DK) -> TMEM
        //      cols [0, 64); record rows 64..127 of the TZP tile get -Z' diag(kd')
        if (zprev) {
            ok = mbar_wait(&bar[2], 0) && ok;
            if (qk && __all_sync(0xffffffffu, ok)) {  // two threads (adjacent lanes) per row, half the columns each
                float ss = silu_cols<DK / 2>(QK, C + (tid >> 1), 128, (tid & 1) * (DK / 2));
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (!(tid & 1)) inkp[tid >> 1] = inv_l2(ss);
                fence_async_smem();
            }
            ok = __syncthreads_and(ok ? 1 : 0) != 0;
            if (tid == 0 && ok) {
                const uint32_t id = idesc_bf16_f32(64, 64);
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_bf16(tmem, tile_desc(smem_u32(WB), 64, 0, ks),
                             tile_desc(smem_u32(QK), 128, 64, ks), id, ks > 0);
                mma_commit(&bar[0]);
            }
            ok = __syncthreads_and((ok && mbar_wait(&bar[0], 0)) ? 1 : 0) != 0;
            tc_fence_after();
            if (ok) {
                const int r = 16 * warp + lane;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float z[32];
                    tmem_ld32(tmem + lane_base + 32 * half, z);
                    tmem_ld_wait(z);
                    if (lane < 16) {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {  // -Z' diag(kd') (/ |k'|)
                            float4 v4 = reinterpret_cast<const float4 *>(kdv + half * 32)[e4];
                            if (qk) {
                                const float4 n4 = reinterpret_cast<const float4 *>(inkp + half * 32)[e4];
                                v4.x *= n4.x, v4.y *= n4.y, v4.z *= n4.z, v4.w *= n4.w;
                            }
                            z[4 * e4] *= -v4.x;
                            z[4 * e4 + 1] *= -v4.y;
                            z[4 * e4 + 2] *= -v4.z;
                            z[4 * e4 + 3] *= -v4.w;
                        }
#pragma unroll
                        for (int i8 = 0; i8 < 4; ++i8)
                            *reinterpret_cast<uint4 *>(
                                rec + R::TZP + sw128_offset(64 + r, half * 32 + i8 * 8, 192)) =
                                pack8(z + i8 * 8);
                    }
                }
            }
        }
    }
    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    if (tid == 0) bulk_wait_all();  // the W tile copy has read shared memory and landed
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ============================================================ diagonal gate
// The GLA row (page "Scrivere meglio nella memoria: gate e delta rule",
// section "Dimenticare: i gate"): S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T, one
// gate per key channel.  With G_r[c] the cumulative log gate of the block,
//   O = (Q * e^G) S^T + P V,   P_ri = sum_c q_r[c] k_i[c] e^{G_r[c] - G_i[c]} (i <= r),
//   S <- S Diag(e^{G_last}) + V^T (K * e^{G_last - G}).
// So the scan is the one without delta, reading Q * e^G and K * e^{G_last - G}
// (prepared here, to the workspace) in place of q and k, with unit g and kd and
// a per-key-channel g_C for the state.  The scores use the second level of
// blocks GLA needs for stability (summary of the same page): for key sub-block
// J (16 tokens, last token e), P[:, J] = (Q * e^{G - G_e}) (K_J * e^{G_e - G_J})^T,
// four tcgen05 products of M = 64, N = 16, one per J, into one 64-column
// accumulator.  The key factors are <= 1; the query factors are <= 1 after J
// and at most e^80 (clamped) inside J.  All factors are products of the gates
// (prefix products along the tokens).  Two threads per key channel, one per
// half of the block (32 tokens): each keeps its half's gates in registers,
// and the products that cross the halves are formed from the gate products
// of the four 16-token sub-blocks, exchanged through shared memory.
constexpr int NTD = 256;  // threads per CTA of the diagonal-gate pass

template <int DK>
struct DiagPrepLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int TILE = KB * 8192;          // [64 rows][DK] bf16, K-major, 128-byte swizzle
    static constexpr int QT = 0;                     // q, then q * e^G (to the workspace)
    static constexpr int KT = QT + TILE;             // k, then k * e^{G_last - G} (to the workspace)
    static constexpr int QH = KT + TILE;             // query factors of one key sub-block
    static constexpr int KH = QH + TILE;             // k * e^{G_e - G}
    static constexpr int NRM = KH + TILE;            // fp32 1/|q| [64], 1/|k| [64] (SiLU + L2)
    static constexpr int PRD = NRM + 512;            // fp32 gate product per sub-block [4][128]
    static constexpr int BAR = PRD + 2048;           // 2 barriers, TMEM slot
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(C * DK * 4 <= 2 * TILE, "the block's gates must fit over the QH and KH tiles");
    static_assert(KH == QH + TILE, "QH and KH must be contiguous");
};

template <int DK, bool QKN>
__global__ void __launch_bounds__(NTD, 3)
chunk_prep_diag_kernel(const float *__restrict__ alpha, uint8_t *__restrict__ ws, int H, int T,
                       int nblk, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk, const Fuse fz,
                       const __grid_constant__ CUtensorMap tmqn,
                       const __grid_constant__ CUtensorMap tmkn) {
    using L = DiagPrepLayout<DK>;
    using R = Rec<DK>;
    constexpr int NS = C / 16;  // key sub-blocks
    constexpr int CH = C / 2;   // tokens per thread
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = blk * C;
    const int n = min(C, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + blk) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    uint8_t *QT = sm + L::QT, *KT = sm + L::KT, *QH = sm + L::QH, *KH = sm + L::KH;
    float *inq = reinterpret_cast<float *>(sm + L::NRM), *ink = inq + 64;
    float *prd = reinterpret_cast<float *>(sm + L::PRD);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);  // q/k tiles, products
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 16);
    const unsigned fl = fz.flags;
    const int c = tid & 127;  // key channel of this thread (threads with c >= DK have none)
    const int hf = tid >> 7;  // half of the block: tokens CH hf .. CH hf + CH - 1
    const int r0 = hf * CH;

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        const uint32_t abytes = (uint32_t)n * DK * 4u;
        mbar_expect_tx(&bar[0], 2u * (uint32_t)L::KB * 8192u + abytes);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
            tma_load_3d(QT + kb * 8192, &tmq, kb * 64, t0, (int)bh, &bar[0]);
            tma_load_3d(KT + kb * 8192, &tmk, kb * 64, t0, (int)bh, &bar[0]);
        }
        // the block's gates ([n][DK] fp32, contiguous) by one bulk copy into
        // the QH and KH tiles, which are not written before the keys pass
        bulk_g2s(QH, alpha + (bh * T + t0) * DK, abytes, &bar[0]);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    // the barriers are initialised before any thread waits on them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = cta_wait(&bar[0], 0, true);
    // this channel's gates of this half (1 past the end of the sequence), and
    // the product over each of its two sub-blocks
    float a[CH];
    if (c < DK) {
        const float ac = (fl & kScaledAlphaMaps) ? fz.ascale[blockIdx.y] : 0.f;
        const float *sa = reinterpret_cast<const float *>(QH) + r0 * DK + c;
#pragma unroll
        for (int rl = 0; rl < CH; ++rl) {
            float x = 1.f;
            if (ok && r0 + rl < n) {
                x = sa[rl * DK];
                if (fl & kAlphaMaps) x = gate(fl, x, ac);
            }
            a[rl] = x;
        }
        float p0 = 1.f, p1 = 1.f;
#pragma unroll
        for (int rl = 0; rl < 16; ++rl) {
            p0 *= a[rl];
            p1 *= a[16 + rl];
        }
        prd[(2 * hf) * 128 + c] = p0;
        prd[(2 * hf + 1) * 128 + c] = p1;
    }
    if (QKN && ok && tid < 2 * C) {  // SiLU of the q and k rows in place; their inverse norms
        const float in = inv_l2(silu_cols<DK>(tid < C ? QT : KT, tid & 63, 64, 0));
        if (tid < C) inq[tid] = in;
        else ink[tid - C] = in;
    }
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Element (r0 + il, c) of a [64][DK] tile (sw128_offset layout).  Every
    // row a thread touches is r0 + il with il < CH, and r0 is a multiple of 8,
    // so the swizzle term depends on il alone: the offsets are a per-thread
    // base, a constant XOR and an immediate.
    const uint32_t cofs = (uint32_t)((c >> 6) * 64 * 128 + (c & 7) * 2 + r0 * 128);
    const uint32_t cx = (uint32_t)((c & 63) >> 3) << 4;
    auto eo = [&](int il) { return cofs + (uint32_t)il * 128u + (cx ^ ((uint32_t)(il & 7) << 4)); };
    auto ld = [&](const uint8_t *t, int il) {
        return __bfloat162float(*reinterpret_cast<const bf16 *>(t + eo(il)));
    };
    auto st = [&](uint8_t *t, int il, float x) {
        *reinterpret_cast<bf16 *>(t + eo(il)) = bf16_rn(x);
    };
    const float *inqh = inq + r0, *inkh = ink + r0;
    auto qrow = [&](int il) {
        float qv = ld(QT, il);
        if (QKN) qv *= inqh[il];
        return qv;
    };
    // gate products of the first half and of its second sub-block
    const float plo = c < DK ? prd[c] * prd[128 + c] : 1.f;
    const float psb1 = c < DK ? prd[128 + c] : 1.f;

    // One reference point for the whole block (token 31) when every channel's
    // decay over the block stays above e^-60: each score factor
    // e^{G_r - G_i} = e^{G_r - G_31} e^{G_31 - G_i} then splits into a query
    // factor and a key factor within [e^-60, e^60], and one product (N = 64
    // keys) gives all of P.  Otherwise the 16-token key sub-blocks below.
    const bool single =
        __syncthreads_and((!ok || c >= DK || hf == 1 ||
                           prd[c] * prd[128 + c] * prd[256 + c] * prd[384 + c] > 8.75e-27f)
                              ? 1 : 0) != 0;
    float gC = 1.f;
    if (single) {
        if (ok && c < DK) {
            if (hf == 1) {
                // tokens 32 + il: query factor = the gates 32..32+il, key factor its inverse
                float pfx = 1.f;
#pragma unroll
                for (int il = 0; il < CH; ++il) {
                    pfx *= a[il];
                    float kv = ld(KT, il);
                    if (QKN) kv *= inkh[il];
                    st(KH, il, kv * fminf(__fdividef(1.f, pfx), 5.5e34f));
                    st(QH, il, qrow(il) * pfx);
                }
            }
            // K * e^{G_last - G} (descending), and for the first half the key
            // factor = the gates il+1..31, the query factor its inverse
            float sfx = 1.f;
            gC = hf == 0 ? prd[2 * 128 + c] * prd[3 * 128 + c] : 1.f;
#pragma unroll
            for (int rl = CH - 1; rl >= 0; --rl) {
                float kv = ld(KT, rl);
                if (QKN) kv *= inkh[rl];
                if (hf == 0) {
                    st(KH, rl, kv * sfx);
                    st(QH, rl, qrow(rl) * fminf(__fdividef(1.f, sfx), 5.5e34f));
                }
                st(KT, rl, kv * gC);
                sfx *= a[rl];
                gC *= a[rl];
            }
            // q * e^G in place over the raw rows (after the query factors read them)
            float g = hf == 0 ? 1.f : plo;
#pragma unroll
            for (int il = 0; il < CH; ++il) {
                g *= a[il];
                st(QT, il, qrow(il) * g);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16_f32(64, 64);
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_bf16(tmem, tile_desc(smem_u32(QH), 64, 0, ks), tile_desc(smem_u32(KH), 64, 0, ks),
                         id, ks > 0);
            mma_commit(&bar[1]);
        }
        ok = cta_wait(&bar[1], 0, ok);
        tc_fence_after();
    } else {
        // ---- keys: K * e^{G_e - G} (sub-block suffix products) and K * e^{G_last - G};
        // the first half starts from the product of the second half's gates, so
        // its gC ends as the product over the whole block
        if (ok && c < DK) {
            if (hf == 0) gC = prd[2 * 128 + c] * prd[3 * 128 + c];
            float s_sub = 1.f;
    #pragma unroll
            for (int rl = CH - 1; rl >= 0; --rl) {
                if ((rl & 15) == 15) s_sub = 1.f;
                float kv = ld(KT, rl);
                if (QKN) kv *= inkh[rl];
                st(KH, rl, kv * s_sub);
                st(KT, rl, kv * gC);
                s_sub *= a[rl];
                gC *= a[rl];
            }
        }
        // ---- scores, one key sub-block per product (unrolled: a[] stays in
        // registers).  Rows of sub-block J get e^{G_r - G_e} (inside J: the
        // inverse of the gates r < j <= e; after J: the gates e < j <= r); each
        // half writes its own rows.  q * e^G replaces the raw q rows of a half
        // once that half's last sub-block has been formed: the first half at
        // J = 2, the second at J = 3.
    #pragma unroll
        for (int J = 0; J < NS; ++J) {
            if (!ok) break;
            if (c < DK) {
                if (hf == (J >> 1)) {  // rows inside J
                    float s = 1.f;
    #pragma unroll
                    for (int rl = 15; rl >= 0; --rl) {
                        const int il = 16 * (J & 1) + rl;
                        st(QH, il, qrow(il) * fminf(__fdividef(1.f, s), 5.5e34f));
                        s *= a[il];
                    }
                }
                if (hf == 0 && J == 0) {  // rows 16..31 after J = 0
                    float p = 1.f;
    #pragma unroll
                    for (int il = 16; il < CH; ++il) {
                        p *= a[il];
                        st(QH, il, qrow(il) * p);
                    }
                }
                if (hf == 1 && J < 2) {  // rows 32..63 after J = 0 or 1
                    float p = J == 0 ? psb1 : 1.f;
    #pragma unroll
                    for (int il = 0; il < CH; ++il) {
                        p *= a[il];
                        st(QH, il, qrow(il) * p);
                    }
                }
                if (hf == 1 && J == 2) {  // rows 48..63 after J = 2
                    float p = 1.f;
    #pragma unroll
                    for (int il = 16; il < CH; ++il) {
                        p *= a[il];
                        st(QH, il, qrow(il) * p);
                    }
                }
                if (J >= 2 && hf == J - 2) {  // q * e^G in place over this half's raw rows
                    float g = hf == 0 ? 1.f : plo;
    #pragma unroll
                    for (int il = 0; il < CH; ++il) {
                        g *= a[il];
                        st(QT, il, qrow(il) * g);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
                const uint32_t id = idesc_bf16_f32(64, 16);
    #pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_bf16(tmem + 16 * J, tile_desc(smem_u32(QH), 64, 0, ks),
                             tile_desc(smem_u32(KH), 64, 16 * J, ks), id, ks > 0);
                mma_commit(&bar[1]);
            }
            ok = cta_wait(&bar[1], J & 1, true);  // QH may be rewritten after the product
            tc_fence_after();
        }
    }
    // ---- the transformed q and k rows -> workspace (rows past T are not written)
    if (tid == 0 && ok) {
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
            tma_store_3d(&tmqn, QT + kb * 8192, kb * 64, t0, (int)bh);
            tma_store_3d(&tmkn, KT + kb * 8192, kb * 64, t0, (int)bh);
        }
        bulk_commit();
    }
    // ---- P rows (M = 64: rows 16w..16w+15 in lanes 32w..32w+15) -> record j+1;
    // warp w takes lane quarter w & 3 and column half w >> 2
    if (ok) {
        const int wq = warp & 3, half = warp >> 2;
        const int r = 16 * wq + lane;
        float x[32];
        tmem_ld32(tmem + ((uint32_t)(32 * wq) << 16) + 32 * half, x);
        tmem_ld_wait(x);
        if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (half * 32 + e > r) x[e] = 0.f;
#pragma unroll
            for (int i8 = 0; i8 < 4; ++i8)
                *reinterpret_cast<uint4 *>(rec_next + R::TZP +
                                           sw128_offset(128 + r, half * 32 + i8 * 8, 192)) =
                    pack8(x + i8 * 8);
        }
    }
    // ---- gate vectors: unit g' and kd' (folded above), per-channel g_C
    float *vn = reinterpret_cast<float *>(rec_next + R::VEC);
    if (tid < 2 * C) vn[tid] = 1.f;
    if (hf == 0 && c < DK) vn[128 + c] = gC;
    if (blk == 0) {  // stage 0 has no previous block
        float *v0 = reinterpret_cast<float *>(rec + R::VEC);
        if (tid < 2 * C) v0[tid] = 1.f;
        if (hf == 0 && c < DK) v0[128 + c] = 1.f;
    }
    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ==================================================================== mLSTM
// The mLSTM memory (page "Le architetture lineari: RetNet, RWKV, xLSTM", xLSTM
// section) in its stabilised form: with F_t the cumulative log forget gate of
// block j, m_prev the stabiliser at the block start (given) and
// m_t = max(F_t + m_prev, max_{s<=t} (F_t - F_s + igate_s)),
//   numerator  g'_t (Q C~^T)_t + sum_s P_ts v_s,   g'_t = e^{F_t + m_prev - m_t},
//              P_ts = (q_t . k_s) e^{F_t - F_s + igate_s - m_t}   (s <= t)
//   normaliser g'_t (n~ . q_t) + sum_s P_ts
//   carry      C~ <- g_C C~ + V^T diag(kd) K,  n~ <- g_C n~ + K^T kd,
//              g_C = e^{F_C + m_prev - m_C},  kd_s = e^{F_C - F_s + igate_s - m_C}.
// Every exponent is <= 0.  The numerator is the scan without delta with these
// factors in the records (g' for the output rows, kd for Delta C, g_C for the
// state); this pass also writes, per block, the row sums of P, m_t and
// Delta n = K^T kd for the normaliser pass.  A final short block is padded
// with log f = 0 and igate = -inf, which changes nothing.
// floats per block of the aux record: row sums [64] at 0, m_t [64] at 64, g'_t [64] at 128,
// g_C at 192, Delta n [<= 128] at 256 (the same constants are in mlstm.cu)
constexpr int kMlstmAux = 384, kAuxRs = 0, kAuxM = 64, kAuxG = 128, kAuxGC = 192, kAuxDn = 256;

// Shared memory of the mLSTM per-block pass: the [Q; K] tile, 384 floats of
// scratch vectors, the barriers (35 KB at d_k = 128: six CTAs per SM; with
// the 51 KB layout of the delta pass it ran four, and the call took 3 % longer).
template <int DK>
struct MlstmPrepLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int QK = 0;
    static constexpr int SV = QK + 128 * 128 * KB;
    static constexpr int BAR = SV + 2048;
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};

template <int DK>
__global__ void __launch_bounds__(NT)
chunk_prep_mlstm_kernel(const float *__restrict__ fgate, const float *__restrict__ igate,
                        const float *__restrict__ m_prev_all, uint8_t *__restrict__ ws,
                        float *__restrict__ aux_all, int H, int T, int nblk,
                        const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmk) {
    using L = MlstmPrepLayout<DK>;
    using R = Rec<DK>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const int t0 = blk * C;
    const int n = min(C, T - t0);
    uint8_t *rec = ws + (bh * (nblk + 1) + blk) * (size_t)R::BYTES;
    uint8_t *rec_next = rec + R::BYTES;
    float *vn = reinterpret_cast<float *>(rec_next + R::VEC);
    float *aux = aux_all + (bh * nblk + blk) * kMlstmAux;
    uint8_t *QK = sm + L::QK;
    float *Sv = reinterpret_cast<float *>(sm + L::SV);  // scratch vectors
    float *At = Sv, *Bs = Sv + 64, *kdv = Sv + 128, *red = Sv + 192;  // F_t - m_t, igate_s - F_s, kd_s
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 32);
    const float m_prev = m_prev_all[bh * nblk + blk];

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[1], 2u * (uint32_t)L::KB * 8192u);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
            tma_load_3d(QK + kb * 16384, &tmq, kb * 64, t0, (int)bh, &bar[1]);
            tma_load_3d(QK + kb * 16384 + 8192, &tmk, kb * 64, t0, (int)bh, &bar[1]);
        }
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    // ---- gates (warps 0-1, token = tid): F_t by a scan of log f, the prefix
    //      max of igate_s - F_s, then m_t and the factors
    float F = 0.f, X = -INFINITY;
    if (tid < C) {
        const float lf = tid < n ? __logf(fgate[bh * T + t0 + tid]) : 0.f;
        const float ig = tid < n ? igate[bh * T + t0 + tid] : -INFINITY;
        F = lf;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, F, d);
            if (lane >= d) F += y;
        }
        X = ig - F;  // with the warp-local F; corrected below for warp 1
        if (warp == 0) red[lane] = F;  // warp 0's inclusive sums
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < C) {
        if (warp == 1) {
            F += red[31];
            X -= red[31];
        }
        float mx = X;  // inclusive prefix max within the warp
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, mx, d);
            if (lane >= d) mx = fmaxf(mx, y);
        }
        if (warp == 0 && lane == 31) red[32] = mx;
        Bs[tid] = X;
        red[64 + tid] = F;
        red[128 + tid] = mx;  // before warp 1 combines with warp 0's maximum
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const float FC = red[64 + 63];
    float mC;
    {
        const float mx63 = fmaxf(red[128 + 63], red[32]);
        mC = fmaxf(FC + m_prev, FC + mx63);
    }
    if (tid < C) {
        const float mx = warp == 1 ? fmaxf(red[128 + tid], red[32]) : red[128 + tid];
        const float mt = fmaxf(F + m_prev, F + mx);
        At[tid] = F - mt;
        const float gp = __expf(F + m_prev - mt);  // 0 when the memory is empty
        vn[kVgPrev + tid] = gp;
        const float kd = __expf(FC - mC + Bs[tid]);
        kdv[tid] = kd;
        vn[kVkdPrev + tid] = kd;
        aux[kAuxM + tid] = mt;
        aux[kAuxG + tid] = gp;
        if (tid == 0) {
            const float gc = __expf(FC + m_prev - mC);
            vn[kVgCPrev] = gc;
            aux[kAuxGC] = gc;
        }
    }
    if (blk == 0) {  // stage 0 has no previous block
        float *v0 = reinterpret_cast<float *>(rec + R::VEC);
        if (tid < 2 * C) v0[tid] = 1.f;
        if (tid == 0) v0[kVgCPrev] = 1.f;
    }
    bool ok = mbar_wait(&bar[1], 0);
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    // ---- Delta n = K^T kd (thread = key channel)
    if (ok && tid < DK) {
        float acc = 0.f;
#pragma unroll 8
        for (int s2 = 0; s2 < C; ++s2)
            acc += kdv[s2] * __bfloat162float(*reinterpret_cast<const bf16 *>(
                                 QK + sw128_offset(64 + s2, tid, 128)));
        aux[kAuxDn + tid] = acc;
    }
    // ---- E1: [Q; K] K^T -> TMEM cols [0, 64) (only the Q rows are used)
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem, tile_desc(smem_u32(QK), 128, 0, ks), tile_desc(smem_u32(QK), 128, 64, ks),
                     id, ks > 0);
        mma_commit(&bar[0]);
    }
    ok = __syncthreads_and((ok && mbar_wait(&bar[0], 0)) ? 1 : 0) != 0;
    tc_fence_after();
    // ---- P rows (bf16, to the next stage's record) and their fp32 sums
    if (ok && warp < 2) {
        const int r = 32 * warp + lane;
        const float ar = At[r];
        float rs = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float a[32];
            tmem_ld32(tmem + lane_base + 32 * half, a);
            tmem_ld_wait(a);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = half * 32 + e;
                a[e] = i <= r ? a[e] * __expf(ar + Bs[i]) : 0.f;
                rs += a[e];
            }
#pragma unroll
            for (int i8 = 0; i8 < 4; ++i8)
                *reinterpret_cast<uint4 *>(rec_next + R::TZP +
                                           sw128_offset(128 + r, half * 32 + i8 * 8, 192)) =
                    pack8(a + i8 * 8);
        }
        aux[kAuxRs + r] = rs;
    }
    if (!ok && lane == 0) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ================================================================== launch


// Value channels per scan CTA.  Each (batch, head) takes dv / NV scan CTAs of
// one SM each.  The scan's stage time is set by the issue and hand-off latency
// of its products, which N = 64 costs barely more than N = 32, so 64-channel
// CTAs pay off when 32-channel ones would need more waves over the SMs than
// 64-channel ones (many heads); otherwise 32 keeps more SMs busy and each
// SM's epilogues short.
int scan_width(int B, int H, int dv) {
    if (dv < 64) return 32;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 32;
    const long long n32 = (long long)B * H * (dv / 32), n64 = n32 / 2;
    return (n64 + sms - 1) / sms < (n32 + sms - 1) / sms ? 64 : 32;
}

// Attribute slot of a 64-channel scan instantiation (the 32-channel ones use
// the slots their launchers pass): 160 + 4 log2(DK / 32) + mode for the lr
// modes, 172 + log2(DK / 32) for the diagonal gate, 175 + log2(DK / 32) for
// mLSTM.  The scans with the folded output norm take 180 + 2 (4 log2(DK / 32) +
// mode) + (NV == 64).
constexpr int wide_slot_base(int dk) { return dk == 32 ? 0 : dk == 64 ? 1 : 2; }

// One record per stage: a head of nblk blocks has nblk + 1 stages.  With
// SiLU + L2 of q and k, the normalised q and k ([B, H, T, dk] bf16 each)
// follow the records.
size_t records_bytes(int B, int H, int T, int dk) {
    const size_t nblk = (size_t)((T + C - 1) / C);
    const size_t rec = dk == 32 ? Rec<32>::BYTES : dk == 64 ? Rec<64>::BYTES : Rec<128>::BYTES;
    return (size_t)B * H * (nblk + 1) * rec;
}

// The diagonal gate: the GLA prep, then the scan without delta reading the
// transformed q and k from the workspace.
template <int DK>
cudaError_t launch_diag(const void *q, const void *k, const void *v, const float *alpha,
                        const float *S0, void *o, float *S_T, int B, int H, int T, int dv,
                        const Fuse &fz, void *ws, cudaStream_t stream, int slot) {
    const int nblk = (T + C - 1) / C;
    const bool qk = (fz.flags & LR_FUSE_QK_SILU_L2) != 0;
    auto prep = qk ? chunk_prep_diag_kernel<DK, true> : chunk_prep_diag_kernel<DK, false>;
    const int nv = scan_width(B, H, dv);
    auto scan = nv == 64 ? chunk_scan_kernel<DK, true, false, true, false, 64>
                         : chunk_scan_kernel<DK, true, false, true>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep),
                                     DiagPrepLayout<DK>::ALLOC, slot + (qk ? 1 : 0));
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC,
                         nv == 64 ? 172 + wide_slot_base(DK) : slot + 2);
    if (e != cudaSuccess) return e;
    CUtensorMap tmq, tmk, tmv, tmqn, tmkn;
    bf16 *qn = reinterpret_cast<bf16 *>(static_cast<uint8_t *>(ws) + records_bytes(B, H, T, DK));
    bf16 *kn = qn + (size_t)B * H * T * DK;
    if ((e = make_rows_map(&tmq, q, DK, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmk, k, DK, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmv, v, dv, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmqn, qn, DK, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmkn, kn, DK, T, B * H)) != cudaSuccess) return e;
    prep<<<dim3(nblk, H, B), NTD, DiagPrepLayout<DK>::ALLOC, stream>>>(
        alpha, static_cast<uint8_t *>(ws), H, T, nblk, tmq, tmk, fz, tmqn, tmkn);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    scan<<<dim3(dv / nv, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
        static_cast<const uint8_t *>(ws), S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk, qn, kn,
        static_cast<const bf16 *>(v), tmqn, tmkn, tmv, nullptr, 0.f, 0);
    return cudaGetLastError();
}

// mLSTM: the per-block pass, then the scan without delta (the numerator).
template <int DK>
cudaError_t launch_mlstm_dk(const void *q, const void *k, const void *v, const float *fgate,
                            const float *igate, const float *m_prev, const float *C0, void *h,
                            float *C_T, float *aux, int phase, int B, int H, int T, int dv,
                            void *ws, cudaStream_t stream, int slot) {
    const int nblk = (T + C - 1) / C;
    auto prep = chunk_prep_mlstm_kernel<DK>;
    const int nv = scan_width(B, H, dv);
    auto scan = nv == 64 ? chunk_scan_kernel<DK, true, false, false, false, 64>
                         : chunk_scan_kernel<DK, true, false>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), MlstmPrepLayout<DK>::ALLOC,
                                     slot);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC,
                         nv == 64 ? 175 + wide_slot_base(DK) : slot + 1);
    if (e != cudaSuccess) return e;
    CUtensorMap tmq, tmk, tmv;
    if ((e = make_rows_map(&tmq, q, DK, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmk, k, DK, T, B * H)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tmv, v, dv, T, B * H)) != cudaSuccess) return e;
    if (phase == 0) {
        prep<<<dim3(nblk, H, B), NT, MlstmPrepLayout<DK>::ALLOC, stream>>>(
            fgate, igate, m_prev, static_cast<uint8_t *>(ws), aux, H, T, nblk, tmq, tmk);
        return cudaGetLastError();
    }
    scan<<<dim3(dv / nv, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
        static_cast<const uint8_t *>(ws), C0, static_cast<bf16 *>(h), C_T, H, T, dv, nblk,
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), static_cast<const bf16 *>(v),
        tmq, tmk, tmv, nullptr, 0.f, 1);
    return cudaGetLastError();
}

template <int DK, bool ALPHA, bool DELTA>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                         int T, int dv, const Fuse &fz, void *ws, cudaStream_t stream, int slot) {
    const int nblk = (T + C - 1) / C;
    // the maps that prep applies (the output RMSNorm runs after the scan)
    const int maps = (fz.flags & LR_FUSE_QK_SILU_L2) ? 2 : (fz.flags & ~LR_FUSE_O_RMSNORM) ? 1 : 0;
    auto prep = maps == 2 ? chunk_prep_kernel<DK, ALPHA, DELTA, 2>
                : maps == 1 ? chunk_prep_kernel<DK, ALPHA, DELTA, 1>
                            : chunk_prep_kernel<DK, ALPHA, DELTA, 0>;
    const int nv = scan_width(B, H, dv);
    // the output norm is applied by the scan (a cluster of the head's dv / nv CTAs)
    const bool norm =
        (fz.flags & LR_FUSE_O_RMSNORM) != 0 && chunked_tc_applies_norm(LR_MODE_DECAY, B, H, dv);
    auto scan = norm ? (nv == 64 ? chunk_scan_kernel<DK, ALPHA, DELTA, false, false, 64, true>
                                 : chunk_scan_kernel<DK, ALPHA, DELTA, false, false, 32, true>)
                     : (nv == 64 ? chunk_scan_kernel<DK, ALPHA, DELTA, false, false, 64>
                                 : chunk_scan_kernel<DK, ALPHA, DELTA>);
    constexpr int mode_ix = (ALPHA ? 1 : 0) + (DELTA ? 2 : 0);  // LINEAR, DECAY, DELTA, GATED_DELTA
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep), PrepLayout<DK>::ALLOC,
                                     slot + 24 * maps);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(scan), ScanLayout<DK>::ALLOC,
                         norm ? 180 + 2 * (4 * wide_slot_base(DK) + mode_ix) + (nv == 64 ? 1 : 0)
                         : nv == 64 ? 160 + 4 * wide_slot_base(DK) + mode_ix : slot + 12);
    if (e != cudaSuccess) return e;
    // q, k and v as [B*H][T][d] with 64 x 64 boxes (for d = 32 the box is
    // wider than a row; its outer half reads zeros)
    CUtensorMap tmq, tmk, tmv;
    e = make_rows_map(&tmq, q, DK, T, B * H);
    if (e != cudaSuccess) return e;
    e = make_rows_map(&tmk, k, DK, T, B * H);
    if (e != cudaSuccess) return e;
    e = make_rows_map(&tmv, v, dv, T, B * H);
    if (e != cudaSuccess) return e;
    // SiLU'd q and k in the workspace (the scan reads them instead)
    const bool qk = maps == 2;
    const bf16 *qs = static_cast<const bf16 *>(q), *ks = static_cast<const bf16 *>(k);
    CUtensorMap tmqn = tmq, tmkn = tmk;
    if (qk) {
        bf16 *qn = reinterpret_cast<bf16 *>(static_cast<uint8_t *>(ws) + records_bytes(B, H, T, DK));
        bf16 *kn = qn + (size_t)B * H * T * DK;
        e = make_rows_map(&tmqn, qn, DK, T, B * H);
        if (e != cudaSuccess) return e;
        e = make_rows_map(&tmkn, kn, DK, T, B * H);
        if (e != cudaSuccess) return e;
        qs = qn;
        ks = kn;
    }
    prep<<<dim3(nblk, H, B), NT, PrepLayout<DK>::ALLOC, stream>>>(
        static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), ALPHA ? alpha : nullptr,
        DELTA ? beta : nullptr, static_cast<uint8_t *>(ws), H, T, nblk, tmq, tmk, fz, tmqn, tmkn);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!norm) {
        scan<<<dim3(dv / nv, H, B), kScanThreads, ScanLayout<DK>::ALLOC, stream>>>(
            static_cast<const uint8_t *>(ws), S0, static_cast<bf16 *>(o), S_T, H, T, dv, nblk, qs,
            ks, static_cast<const bf16 *>(v), qk ? tmqn : tmq, qk ? tmkn : tmk, tmv, nullptr, 0.f, 0);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dv / nv, H, B);
    cfg.blockDim = dim3(kScanThreads);
    cfg.dynamicSmemBytes = ScanLayout<DK>::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(dv / nv);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scan, static_cast<const uint8_t *>(ws), S0,
                              static_cast<bf16 *>(o), S_T, H, T, dv, nblk, qs, ks,
                              static_cast<const bf16 *>(v), qk ? tmqn : tmq, qk ? tmkn : tmk, tmv,
                              fz.norm_w, fz.norm_eps, 0);
}

template <int DK>
cudaError_t launch_mode(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                        int T, int dv, lr_mode mode, const Fuse &fz, void *ws,
                        cudaStream_t stream, int slot) {
    switch (mode) {
    case LR_MODE_LINEAR:
        return launch_typed<DK, false, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, fz,
                                              ws, stream, slot + 0);
    case LR_MODE_DECAY:
        return launch_typed<DK, true, false>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, fz,
                                             ws, stream, slot + 1);
    case LR_MODE_DELTA:
        return launch_typed<DK, false, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, fz,
                                             ws, stream, slot + 2);
    case LR_MODE_DIAG_DECAY:
        return launch_diag<DK>(q, k, v, alpha, S0, o, S_T, B, H, T, dv, fz, ws, stream,
                               120 + (slot - 32));
    default:
        return launch_typed<DK, true, true>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, fz,
                                            ws, stream, slot + 3);
    }
}

}  // namespace

size_t chunked_tc_workspace_bytes(int B, int H, int T, int dk, lr_mode mode, unsigned flags) {
    const bool qk = (flags & LR_FUSE_QK_SILU_L2) || mode == LR_MODE_DIAG_DECAY;
    return records_bytes(B, H, T, dk) + (qk ? 2 * (size_t)B * H * T * dk * 2 : 0);
}

// Attribute slots 32..91 and 120..131 (diagonal gate) belong to this file.
cudaError_t launch_chunked_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *S_T, int B,
                              int H, int T, int dk, int dv, lr_mode mode, const Fuse &fz,
                              void *ws, cudaStream_t stream) {
    switch (dk) {
    case 32:
        return launch_mode<32>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, fz, ws, stream,
                               32);
    case 64:
        return launch_mode<64>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, fz, ws, stream,
                               36);
    default:
        return launch_mode<128>(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dv, mode, fz, ws,
                                stream, 40);
    }
}

size_t records_bytes_tc(int B, int H, int T, int dk) { return records_bytes(B, H, T, dk); }

// The scan folds the output norm when a head's value channels span at most
// two CTAs.  With four (d_v = 128 on 32-channel CTAs) the exchange cost as
// much as the separate pass saved, or more, depending on the device: 0.495
// against 0.499 ms on one GB300 and 0.507 against 0.500 ms on another for the
// gated-delta prefill B=2 H=16 T=16384; with two it saved 3 to 8 %.
bool chunked_tc_applies_norm(lr_mode mode, int B, int H, int dv) {
    return mode != LR_MODE_DIAG_DECAY && dv / scan_width(B, H, dv) <= 2;
}

// Attribute slots 136..141 belong to the mLSTM launch.
cudaError_t launch_mlstm_tc(const void *q, const void *k, const void *v, const float *fgate,
                            const float *igate, const float *m_prev, const float *C0, void *h,
                            float *C_T, float *aux, int phase, int B, int H, int T, int dk,
                            int dv, void *ws, cudaStream_t stream) {
    switch (dk) {
    case 32:
        return launch_mlstm_dk<32>(q, k, v, fgate, igate, m_prev, C0, h, C_T, aux, phase, B, H, T,
                                   dv, ws, stream, 136);
    case 64:
        return launch_mlstm_dk<64>(q, k, v, fgate, igate, m_prev, C0, h, C_T, aux, phase, B, H, T,
                                   dv, ws, stream, 138);
    default:
        return launch_mlstm_dk<128>(q, k, v, fgate, igate, m_prev, C0, h, C_T, aux, phase, B, H, T,
                                    dv, ws, stream, 140);
    }
}

// Where the per-token factor of block j's output rows goes: the record of
// stage j + 1, at this byte offset within it (vector slot kVrs), records of
// this many bytes, nblk + 1 per (batch, head) from the start of the workspace.
void mlstm_factor_slot(int dk, size_t *rec_bytes, size_t *offset) {
    const int rb = dk == 32 ? Rec<32>::BYTES : dk == 64 ? Rec<64>::BYTES : Rec<128>::BYTES;
    const int vo = dk == 32 ? Rec<32>::VEC : dk == 64 ? Rec<64>::VEC : Rec<128>::VEC;
    *rec_bytes = (size_t)rb;
    *offset = (size_t)vo + (size_t)kVrs * 4;
}

cudaError_t set_scan_fault_tc(unsigned on) {
    return cudaMemcpyToSymbol(g_scan_fault, &on, sizeof(on));
}

int read_and_clear_tc_error() {
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_error, sizeof(int)) != cudaSuccess) return -1;
    if (h) cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    return h;
}

}  // namespace lr
