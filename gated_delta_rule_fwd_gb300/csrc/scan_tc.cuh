// Sequential pass of the chunked forward on the tensor cores (tcgen05 +
// TMEM, TMA, mbarriers), the workspace record it reads, and the tensor maps
// of its operands.  Included by the translation units whose per-block passes
// write records for it: chunked_tc.cu (the lr modes, the diagonal gate, the
// mLSTM numerator) and gen_delta_tc.cu (the RWKV-7 generalised delta rule).
// The block algebra and the look-ahead form the scan evaluates are described
// at the top of chunked_tc.cu.  Every definition sits in an anonymous
// namespace, so each including file has its own copy, error word included.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_internal.cuh"
#include "tc_common.cuh"

namespace lr {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int C = 64;      // tokens per block
constexpr int DVS = 32;    // value channels per scan CTA (the default width; 64 when that
                           // halves the waves of CTAs, see scan_width)

__device__ int g_tc_error = 0;  // set to 1 when a bounded wait gives up
// Failure-detection test hook, set from the host (0 = off): a scan launched
// while it is set polls each barrier at most kFaultSpinLimit times and its
// late-group load thread skips the loads of stage 1, so the waits for that
// stage run out and the kernel takes its exit path.
__device__ unsigned g_scan_fault = 0;

// Workspace record of stage j of one head (stages 0..nblk), written by the
// prep CTAs of blocks j and j-1 and read by the scan.
template <int DK>
struct Rec {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int WT = 0;                // W_j: KB blocks of [64 rows][128 B]
    static constexpr int TZP = WT + KB * 8192;  // [192 rows][64] bf16: T_j diag(beta), -Z_{j-1}, P_{j-1}
    static constexpr int VEC = TZP + 24576;     // fp32: g' [64], kd' [64], kd [64], g_C'
    static constexpr int BYTES = VEC + 1024;
};
// offsets (in floats) inside the gate vector of a record
constexpr int kVgPrev = 0, kVkdPrev = 64, kVkd = 128, kVgCPrev = 192;
constexpr int kVrs = 128;  // without delta (kd unused): a factor per output row (mLSTM)
constexpr int kVgCDiag = 128;  // diagonal gate: g_C' per key channel (128 floats)
constexpr int kVgCGen = 0;     // generalised delta rule: g_C' per key channel (128 floats)

// a in the low half, b in the high half, both rounded to nearest even by one
// paired conversion (two single conversions run at a fraction of its rate)
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8(const float *x) {
    uint4 r;
    r.x = pack_bf16(x[0], x[1]);
    r.y = pack_bf16(x[2], x[3]);
    r.z = pack_bf16(x[4], x[5]);
    r.w = pack_bf16(x[6], x[7]);
    return r;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// ===================================================================== scan

template <int DK>
struct ScanLayout {
    static constexpr int KB = (DK + 63) / 64;
    static constexpr int AW_BYTES = 128 * 128 * KB;  // [128][DK] K-major: W rows, Q' rows
    static constexpr int AW = 0;                      // x2
    static constexpr int TZP = AW + 2 * AW_BYTES;     // x2 [192][64] K-major: T diag(beta), -Z', P'
    static constexpr int KR = TZP + 2 * 24576;        // x2 [64 tokens][128] MN-major: K'
    static constexpr int VR = KR + 2 * 16384;         // x2 [64 tokens][64] MN-major: v box (this CTA: 32 channels)
    static constexpr int VEC = VR + 2 * 8192;         // x2 gate vectors of the stage
    static constexpr int UB = VEC + 2 * 1024;         // [64 tokens][64] MN-major: U
    static constexpr int UBK = UB + 8192;             // x2 [64 tokens][64] MN-major: kd U (kd' V')
    static constexpr int SB_BYTES = 128 * DK;         // [DK][64] MN-major: bf16 S^T slice (32 used)
    static constexpr int SB = UBK + 2 * 8192;         // x2
    // output norm folded into the scan: per slot (parity of the output block),
    // per (cluster rank, warp half) and per token row, a partial sum of squares
    static constexpr int PS = SB + 2 * SB_BYTES;      // fp32 [2][8][64]
    static constexpr int BAR = PS + 2 * 8 * 64 * 4;
    static constexpr int BYTES = BAR + 256;
    static constexpr int ALLOC = BYTES + 1024;
};

// TMEM columns of the scan kernel with NV value channels per CTA: per stage
// parity p, at p * 4 NV, four fp32 accumulators of NV columns (M = 128 lanes):
// a at 0, b at NV, c at 2 NV, ds at 3 NV; 8 NV columns in all.
template <int NV>
struct ScanCols {
    static constexpr uint32_t Da = 0, Db = NV, Dc = 2 * NV, DS = 3 * NV, PAR = 4 * NV, ALL = 8 * NV;
};

// L2 prefetch of what stage `st` will fetch (one thread).
template <int DK, bool DELTA, bool GEN>
__device__ __forceinline__ void scan_prefetch_l2(const bf16 *q, const bf16 *k, const bf16 *v,
                                                 const uint8_t *rec, size_t bh, int T, int st,
                                                 int nblk, int dv) {
    constexpr int TS = GEN ? C / 2 : C;  // tokens per stage
    const int Tq = GEN ? nblk * C : T;   // rows of the q and k operands
    prefetch_l2(rec, Rec<DK>::BYTES);
    const int pb = st - 1;
    if (pb >= 0 && pb < nblk) {
        const int t0 = pb * C, n = min(C, Tq - t0);
        prefetch_l2(q + (bh * Tq + t0) * DK, (uint32_t)n * DK * 2);
        prefetch_l2(k + (bh * Tq + t0) * DK, (uint32_t)n * DK * 2);
    }
    const int vb = DELTA ? st : st - 1;
    if (vb >= 0 && vb < nblk) {
        const int t0 = vb * TS, n = min(TS, T - t0);
        prefetch_l2(v + (bh * T + t0) * dv, (uint32_t)n * dv * 2);
    }
}

// Scan kernel roles (384 threads), stage j = 0..nblk (parity p = j & 1):
//   warp 0, lane 0   issues b_j = [W_j; Q_{j-1}] S_{j-1}^T (the U rows take -g_C') and
//                    c_j = [-Z_{j-1}; P_{j-1}] U_{j-1}   (P_{j-1} V_{j-1} without delta)
//   warp 1, lane 0   issues a_j = [T_j diag(beta); *] V_j and
//                    ds = K_{j-1}^T (kd U_{j-1})          (K^T (kd V) without delta)
//   warp 2, lane 0   loads the early group of stage j into buffer p: what b_j
//                    reads (W_j, Q_{j-1})
//   warp 3, lane 0   loads the late group: what a_j, c_j, ds and the epilogues
//                    read (T_j diag(beta), -Z_{j-1}, P_{j-1}, K_{j-1}, the gates,
//                    V_j; V_{j-1} without delta)
//   warps 4, 5, 8, 9 U rows (TMEM lanes 0..63): U_j = Da + Db + Dc -> bf16 U,
//                    kd U; without delta they form kd' V' for ds instead
//   warps 6, 7, 10, 11  output rows (lanes 64..127): O_{j-1} = g' Db + Dc
//   warps 12..19     state (lanes 0..127 = key channels): S_j = g_C' S_{j-1} + ds,
//                    fp32 in registers, bf16 copy for b_{j+1}
// Each epilogue role is split over two warps per TMEM lane quarter, one per
// half of the 32 value channels, to keep the per-warp instruction chains short.
// All loads are TMA or bulk copies completing on the group's `full` barrier,
// which the consumers wait on directly.  The early group is released as soon
// as b_j is done, so the next fill of that part of the buffer starts about
// half a stage earlier than the late one; it is kept small (32 KB at
// d_k = 128) because b_j sits on the state chain.
// The state before the first block plays S_{-1} (with g_C = 1 and U_{-1} = 0).
// GEN (the generalised delta rule): a stage covers 32 tokens; the 64 U rows
// are [V_j; U_j] (values stacked on pseudo-values), the output rows 32; q and
// k are per-stage operands of 64 rows that the per-block pass wrote (the
// decayed queries and the stacked removal and write keys); the record's W
// tile, Z and P rows already carry every factor (g' = kd = 1, -g_C' = 1 on W)
// and g_C' is per key channel; v is read from token 32 j with the usual
// 64-row box, the second half meeting zero columns of T.
// Hand-offs are mbarriers, every wait bounded.  Each barrier is waited on by
// all of its consumers before it can complete again: barriers that complete
// once per stage and could run ahead are kept per parity, and every consumer
// arrives on a group's `empty` barrier only after its waits of that stage.
constexpr int kScanThreads = 640;

// Arrive once per warp on `bar`: every lane has finished its part (and its own
// fences) before lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

struct ScanBars {
    uint64_t fullE[2];   // early group landed                           (1 + tx bytes)
    uint64_t emptyE[2];  // early group read                             (1 commit)
    uint64_t fullL[2];   // late group landed                            (1 + tx bytes)
    uint64_t emptyL[2];  // late group read                              (2 commits + 16 warps)
    uint64_t vkr[2];     // kd' V' written (no delta)                    (4 warps)
    uint64_t dA[2];      // b and c products of the stage done           (commit)
    uint64_t dB[2];      // a product of the stage done                  (commit)
    uint64_t dsf[2];     // ds product of the stage done                 (commit)
    uint64_t tfree[2];   // output rows of the stage read                (4 warps)
    uint64_t uk[2];      // kd U rows of this parity written             (4 warps)
    uint64_t s[2];       // bf16 state copy of this parity written       (8 warps)
    uint64_t u;          // U rows written                               (4 warps)
    uint64_t fin[2];     // every product an issuer issued has completed (commit)
    uint64_t psfull[2];  // folded norm: every CTA's partial sums of slot s in   (1 + 512 bytes per CTA)
    uint32_t tmem;
};
static_assert(sizeof(ScanBars) <= 256, "the barriers must fit their shared-memory slot");
constexpr uint32_t kEmptyLCount = 2 + 4 + 4 + 8;  // both issuers' commits, U, output and state warps
constexpr uint32_t kPsBytes = 4 * 32 * 4;         // partial sums one CTA sends a CTA per block

// NORM: the output RMSNorm folded into the output rows (o_t / sqrt(mean over the
// d_v channels of o_t^2 + eps) * weight).  The dv / NV CTAs of a head run as one
// cluster.  Per output block each output warp sends its 32 rows' partial sums
// of squares to every CTA of the cluster with st.async (16 bytes per 4 rows),
// into slot blk & 1 of the receiver, counted as transaction bytes on the
// receiver's psfull[blk & 1]; the rows are then normalised with the total and
// stored.  Two slots suffice: a CTA sends block m only after it has read block
// m - 1, so once every CTA's sums of block m - 1 are in, every CTA is done with
// block m - 2.  Each receiver arms a slot's next use (expect_tx) after its wait;
// bytes that arrive first leave the transaction count negative until then.
// Cluster barriers at the start (barriers initialised and armed) and at the
// exit (no CTA leaves while another may still send to it) bracket the
// exchange; a CTA whose wait gave up still meets the others there, and every
// store it was sent was issued before its sender reached that barrier.
template <int DK, bool ALPHA, bool DELTA, bool DIAG = false, bool GEN = false, int NV = DVS,
          bool NORM = false>
__global__ void __launch_bounds__(kScanThreads, 1)
chunk_scan_kernel(const uint8_t *__restrict__ ws, const float *__restrict__ S0,
                  bf16 *__restrict__ o, float *__restrict__ ST, int H, int T, int dv, int nblk,
                  const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                  const bf16 *__restrict__ v, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const float *__restrict__ norm_w, float norm_eps, int row_scale) {
    using L = ScanLayout<DK>;
    using R = Rec<DK>;
    static_assert(!GEN || (DELTA && !DIAG), "the generalised delta rule runs the delta protocol");
    static_assert(NV == 32 || (NV == 64 && !GEN), "32 or 64 value channels per CTA");
    static_assert(!NORM || (!GEN && !DIAG), "the folded norm serves the lr modes");
    using TC = ScanCols<NV>;
    constexpr uint32_t kDa = TC::Da, kDb = TC::Db, kDc = TC::Dc, kDS = TC::DS, kParCols = TC::PAR;
    constexpr uint32_t kScanCols = TC::ALL;
    constexpr int TS = GEN ? C / 2 : C;  // tokens per stage
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = align1024(sm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.x * NV;
    const int vx = c0 & ~63;                           // TMA box column of the v slice
    const uint32_t voff = (uint32_t)(c0 & 63) * 2u;    // byte offset of the slice in a box row
    const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
    const uint8_t *recs = ws + bh * (nblk + 1) * (size_t)R::BYTES;
    ScanBars *bars = reinterpret_cast<ScanBars *>(sm + L::BAR);
    auto vec_of = [&](int p) { return reinterpret_cast<const float *>(sm + L::VEC + p * 1024); };

    // zero everything once: padding rows and columns of the operands must read 0
    for (int i = tid; i < L::BAR / 16; i += kScanThreads)
        reinterpret_cast<uint4 *>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->fullE[b], 1);
            mbar_init(&bars->emptyE[b], 1);
            mbar_init(&bars->fullL[b], 1);
            mbar_init(&bars->emptyL[b], kEmptyLCount);
            mbar_init(&bars->vkr[b], 4);
            mbar_init(&bars->dA[b], 1);
            mbar_init(&bars->dB[b], 1);
            mbar_init(&bars->dsf[b], 1);
            mbar_init(&bars->tfree[b], 4);
            mbar_init(&bars->uk[b], 4);
            mbar_init(&bars->s[b], 8);
            mbar_init(&bars->fin[b], 1);
        }
        mbar_init(&bars->u, 4);
        if (NORM) {
            for (int b = 0; b < 2; ++b) mbar_init(&bars->psfull[b], 1);
        }
        fence_mbar_init();
        if (NORM)  // each slot's first use: blocks 0 and 1
            for (int b = 0; b < 2; ++b) mbar_expect_tx(&bars->psfull[b], kPsBytes * gridDim.x);
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem, kScanCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the peers' barriers are initialised before any CTA arrives on them
    if (NORM) cluster_sync_all();
    const uint32_t tmem = bars->tmem;
    bool ok = true;
    const bool fault = g_scan_fault != 0;
    const uint32_t limit = fault ? kFaultSpinLimit : kSpinLimit;
    auto wait = [limit](uint64_t *bar, uint32_t parity) { return mbar_wait(bar, parity, limit); };

    const uint32_t id_kn = idesc_bf16_f32_mn(128, NV, false, true);
    const uint32_t id_nn = idesc_bf16_f32_mn(128, NV, true, true);
    auto aw_desc = [&](int p) { return tile_desc(smem_u32(sm + L::AW + p * L::AW_BYTES), 128, 0, 0); };
    auto tz_desc = [&](int p) { return tile_desc(smem_u32(sm + L::TZP + p * 24576), 192, 0, 0); };
    auto zp_desc = [&](int p) { return tile_desc(smem_u32(sm + L::TZP + p * 24576), 192, 64, 0); };
    auto kr_desc = [&](int p) { return tile_desc_mn(smem_u32(sm + L::KR + p * 16384), 64, 0); };
    // the v box holds 64 channels; this CTA's 32 start `voff` bytes into each row
    auto vr_desc = [&](int p) { return tile_desc_mn(smem_u32(sm + L::VR + p * 8192) + voff, 64, 0); };
    auto ubk_desc = [&](int i) { return tile_desc_mn(smem_u32(sm + L::UBK + i * 8192), 64, 0); };
    auto sb_desc = [&](int i) { return tile_desc_mn(smem_u32(sm + L::SB + i * L::SB_BYTES), DK, 0); };

    if (warp == 0) {
        // ======================================= b and c products (issuer A)
        if (lane == 0) {
            const uint64_t d_ub = tile_desc_mn(smem_u32(sm + L::UB), 64, 0);
            for (int j = 0; j <= nblk && ok; ++j) {
                const int p = j & 1;
                const uint32_t ph = (j >> 1) & 1, base = p * kParCols;
                ok = wait(&bars->fullE[p], ph);
                // output rows of stage j-2 (same accumulators) read
                if (ok && j >= 2) ok = wait(&bars->tfree[p], ph ^ 1);
                // S_{j-1} in state copy p
                if (ok) ok = wait(&bars->s[p], ph);
                if (!ok) break;
                tc_fence_after();
                const uint64_t d_aw = aw_desc(p), d_sb = sb_desc(p);
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_bf16(tmem + base + kDb, kdesc_step(d_aw, 128, ks), mndesc_step(d_sb, ks),
                             id_kn, ks > 0);
                mma_commit(&bars->emptyE[p]);
                if (j >= 1) {
                    ok = wait(&bars->fullL[p], ph);
                    if (ok && DELTA) ok = wait(&bars->u, (j - 1) & 1);  // U_{j-1}
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t d_zp = zp_desc(p), d_x = DELTA ? d_ub : vr_desc(p);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(tmem + base + kDc, kdesc_step(d_zp, 192, ks), mndesc_step(d_x, ks),
                                 id_kn, ks > 0);
                }
                mma_commit(&bars->dA[p]);
                mma_commit(&bars->emptyL[p]);
            }
            mma_commit(&bars->fin[0]);
            if (!wait(&bars->fin[0], 0)) ok = false;
        }
    } else if (warp == 1) {
        // ====================================== a and ds products (issuer B)
        if (lane == 0) {
            for (int j = 0; j <= nblk && ok; ++j) {
                const int p = j & 1;
                const uint32_t ph = (j >> 1) & 1, base = p * kParCols;
                ok = wait(&bars->fullL[p], ph);
                if (!ok) break;
                tc_fence_after();
                if (DELTA && j < nblk) {
                    const uint64_t d_tz = tz_desc(p), d_vr = vr_desc(p);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(tmem + base + kDa, kdesc_step(d_tz, 192, ks), mndesc_step(d_vr, ks),
                                 id_kn, ks > 0);
                }
                mma_commit(&bars->dB[p]);
                if (j >= 1) {
                    if (ok) ok = DELTA ? wait(&bars->uk[(j - 1) & 1], ((j - 1) >> 1) & 1)  // kd U_{j-1}
                                       : wait(&bars->vkr[p], ph);                          // kd' V'
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t d_kr = kr_desc(p), d_y = ubk_desc(DELTA ? (j - 1) & 1 : p);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16(tmem + base + kDS, mndesc_step(d_kr, ks), mndesc_step(d_y, ks),
                                 id_nn, ks > 0);
                }
                mma_commit(&bars->dsf[p]);
                mma_commit(&bars->emptyL[p]);
            }
            mma_commit(&bars->fin[1]);
            if (!wait(&bars->fin[1], 0)) ok = false;
        }
    } else if (warp == 2) {
        // ============================================ early-group loads
        if (lane == 0) {
            int issued = -1;
            for (int j = 0; j <= nblk && ok; ++j) {
                const int p = j & 1;
                if (j >= 2) ok = wait(&bars->emptyE[p], ((j >> 1) - 1) & 1);
                if (!ok) break;
                const uint8_t *rec = recs + (size_t)j * R::BYTES;
                uint8_t *aw = sm + L::AW + p * L::AW_BYTES;
                if (j + 2 <= nblk && blockIdx.x == 0)  // one CTA of the head suffices
                    scan_prefetch_l2<DK, DELTA, GEN>(q, k, v, rec + 2 * (size_t)R::BYTES, bh, T, j + 2,
                                                nblk, dv);
                const bool cur = DELTA && j < nblk, prev = j >= 1;
                const uint32_t bytes = (cur ? (uint32_t)R::KB * 8192u : 0u) +
                                       (prev ? (uint32_t)R::KB * 8192u : 0u);
                mbar_expect_tx(&bars->fullE[p], bytes);
                if (cur) {
#pragma unroll
                    for (int kb = 0; kb < R::KB; ++kb)
                        bulk_g2s(aw + kb * 16384, rec + R::WT + kb * 8192, 8192, &bars->fullE[p]);
                }
                if (prev) {
#pragma unroll
                    for (int kb = 0; kb < R::KB; ++kb)
                        tma_load_3d(aw + kb * 16384 + 8192, &tmq, kb * 64, (j - 1) * C, (int)bh,
                                    &bars->fullE[p]);
                }
                issued = j;
            }
            // never leave with copies into shared memory in flight
            for (int j = issued > 0 ? issued - 1 : 0; j <= issued; ++j)
                if (!wait(&bars->fullE[j & 1], (j >> 1) & 1)) ok = false;
        }
    } else if (warp == 3) {
        // ============================================= late-group loads
        int issued = -1;
        for (int j = 0; j <= nblk && ok; ++j) {
            const int p = j & 1;
            const bool prev = j >= 1;
            if (lane == 0) {
                if (j >= 2) ok = wait(&bars->emptyL[p], ((j >> 1) - 1) & 1);
                if (ok && fault && j == 1) {
                    issued = j;  // the test hook: stage 1 is never loaded
                } else if (ok) {
                    const uint8_t *rec = recs + (size_t)j * R::BYTES;
                    const bool cur = DELTA && j < nblk;
                    uint32_t bytes = 1024u + (DELTA ? 24576u : 0u) + (cur ? 8192u : 0u);
                    if (prev) bytes += (DELTA ? 0u : 8192u) + (uint32_t)R::KB * 8192u +
                                       (DELTA ? 0u : 8192u);
                    mbar_expect_tx(&bars->fullL[p], bytes);
                    bulk_g2s(sm + L::VEC + p * 1024, rec + R::VEC, 1024, &bars->fullL[p]);
                    if (DELTA)
                        bulk_g2s(sm + L::TZP + p * 24576, rec + R::TZP, 24576, &bars->fullL[p]);
                    if (cur)
                        tma_load_3d(sm + L::VR + p * 8192, &tmv, vx, j * TS, (int)bh, &bars->fullL[p]);
                    if (prev) {
                        if (!DELTA)
                            bulk_g2s(sm + L::TZP + p * 24576 + 16384, rec + R::TZP + 16384, 8192,
                                     &bars->fullL[p]);
#pragma unroll
                        for (int kb = 0; kb < R::KB; ++kb)
                            tma_load_3d(sm + L::KR + p * 16384 + kb * 8192, &tmk, kb * 64,
                                        (j - 1) * C, (int)bh, &bars->fullL[p]);
                        if (!DELTA)
                            tma_load_3d(sm + L::VR + p * 8192, &tmv, vx, (j - 1) * C, (int)bh,
                                        &bars->fullL[p]);
                    }
                    issued = j;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
        // never leave with copies into shared memory in flight
        if (lane == 0)
            for (int j = issued > 0 ? issued - 1 : 0; j <= issued; ++j)
                if (!wait(&bars->fullL[j & 1], (j >> 1) & 1)) ok = false;
    } else if (warp < 12 && (warp & 3) < 2) {
        // ============================================ U rows (TMEM lanes 0..63)
        const int r = 32 * (warp & 3) + lane;
        const int ch0 = (NV / 2) * ((warp - 4) >> 2);  // first value channel of this warp's half
        const uint32_t lb0 = (uint32_t)(32 * (warp & 3)) << 16;
        for (int j = 0; j <= nblk && ok; ++j) {
            const int p = j & 1;
            const uint32_t ph = (j >> 1) & 1, base = p * kParCols;
            ok = __all_sync(0xffffffffu, wait(&bars->fullL[p], ph));
            if (!ok) break;
            // with delta only the gates are read from the late group: take them
            // and release it now
            const float kdr = GEN ? 1.f : DELTA ? vec_of(p)[kVkd + r] : 0.f;
            // b's W rows carry -g_C' (the generalised rule folds its factors into W)
            const float gn = GEN ? 1.f : DELTA ? -vec_of(p)[kVgCPrev] : 0.f;
            if (DELTA) warp_arrive(&bars->emptyL[p]);
            if (DELTA && j < nblk) {
                ok = wait(&bars->dA[p], ph);
                ok = ok && wait(&bars->dB[p], ph);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int sub = 0; sub < NV / 32; ++sub) {  // 16 value channels at a time
                    const int ch = ch0 + 16 * sub;
                    const uint32_t lb = lb0 + (uint32_t)ch;
                    float x[16], y[16], z[16];
                    tmem_ld16(tmem + lb + base + kDa, x);
                    tmem_ld16(tmem + lb + base + kDb, y);
                    if (j > 0) {
                        tmem_ld16(tmem + lb + base + kDc, z);
                        tmem_ld_wait(x, y, z);
#pragma unroll
                        for (int c = 0; c < 16; ++c) x[c] += gn * y[c] + z[c];
                    } else {
                        tmem_ld_wait(x, y);
#pragma unroll
                        for (int c = 0; c < 16; ++c) x[c] += gn * y[c];
                    }
                    // kd U (for ds, on the state chain) and U (for c, on the U chain)
                    float xk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) xk[c] = x[c] * kdr;
#pragma unroll
                    for (int c8 = 0; c8 < 2; ++c8) {
                        *reinterpret_cast<uint4 *>(sm + L::UBK + p * 8192 +
                                                   sw128_offset(r, ch + c8 * 8, 64)) = pack8(xk + c8 * 8);
                        *reinterpret_cast<uint4 *>(sm + L::UB + sw128_offset(r, ch + c8 * 8, 64)) =
                            pack8(x + c8 * 8);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                warp_arrive(&bars->uk[p]);
                warp_arrive(&bars->u);
            } else {
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (!DELTA && j >= 1) {
                    // kd' V' (B operand of Delta S = K'^T diag(kd') V'): this warp's
                    // 16 token rows
                    const float *vec = vec_of(p);
                    const uint8_t *vr = sm + L::VR + p * 8192;
                    uint8_t *vk = sm + L::UBK + p * 8192;
                    const int rw = 16 * (((warp & 3) << 1) | ((warp - 4) >> 2));
                    for (int idx = lane; idx < 16 * (NV / 8); idx += 32) {
                        const int rr = rw + idx / (NV / 8), c8 = idx % (NV / 8);
                        const uint4 raw = *reinterpret_cast<const uint4 *>(
                            vr + sw128_offset(rr, (c0 & 63) + c8 * 8, 64));
                        const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
                        const float f = vec[kVkdPrev + rr];
                        float xv[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) xv[t] = f * __bfloat162float(e[t]);
                        *reinterpret_cast<uint4 *>(vk + sw128_offset(rr, c8 * 8, 64)) = pack8(xv);
                    }
                    fence_async_smem();
                }
                // one completion per stage (also the first) keeps the parities aligned
                if (!DELTA) warp_arrive(&bars->vkr[p]);
            }
            if (!DELTA) warp_arrive(&bars->emptyL[p]);
        }
    } else if (warp < 12) {
        // ===================================== output rows (TMEM lanes 64..127)
        const int r = 32 * (warp & 3) + lane - 64;
        const int half = (warp - 4) >> 2;
        const int ch = (NV / 2) * half;  // this warp's NV / 2 value channels
        const uint32_t lb = ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)ch;
        auto store_rows = [&](const float *rows, int blk) {
            const int t = blk * TS + r;
            if (r < TS && t < T) {
                uint4 *dst = reinterpret_cast<uint4 *>(o + (bh * T + t) * dv + c0 + ch);
#pragma unroll
                for (int i8 = 0; i8 < NV / 16; ++i8) dst[i8] = pack8(rows + i8 * 8);
            }
        };
        float *const ps = reinterpret_cast<float *>(sm + L::PS);
        for (int j = 0; j <= nblk && ok; ++j) {
            const int p = j & 1;
            const uint32_t ph = (j >> 1) & 1, base = p * kParCols;
            ok = __all_sync(0xffffffffu, wait(&bars->fullL[p], ph));
            if (!ok) break;
            // the late-group values read here: g' and, with row_scale, a factor
            // per token (mLSTM: 1 / max(|denominator|, e^-m))
            const float gr = GEN ? 1.f : vec_of(p)[kVgPrev + r];
            const float rsc = (!DELTA && row_scale) ? vec_of(p)[kVrs + r] : 1.f;
            warp_arrive(&bars->emptyL[p]);
            if (j >= 1) ok = __all_sync(0xffffffffu, wait(&bars->dA[p], ph));
            if (!ok) break;
            if (j >= 1) {
                tc_fence_after();
                float out[NV / 2];
#pragma unroll
                for (int sub = 0; sub < NV / 32; ++sub) {
                    float x[16], y[16];
                    tmem_ld16(tmem + lb + base + kDb + 16 * sub, x);
                    tmem_ld16(tmem + lb + base + kDc + 16 * sub, y);
                    tmem_ld_wait(x, y);
#pragma unroll
                    for (int c = 0; c < 16; ++c)  // (g' Q' S'^T + P' U') times the token's factor
                        out[16 * sub + c] = (gr * x[c] + y[c]) * rsc;
                }
                tc_fence_before();
                warp_arrive(&bars->tfree[p]);
                if (NORM) {
                    const int m = j - 1, sl = m & 1;  // this output block and its slot
                    float ss = 0.f;
#pragma unroll
                    for (int c = 0; c < NV / 2; ++c) ss = fmaf(out[c], out[c], ss);
                    // lanes 0..7 send the sums of rows 4 lane .. 4 lane + 3 of the warp
                    float g[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) g[i] = __shfl_sync(0xffffffffu, ss, 4 * (lane & 7) + i);
                    if (lane < 8) {
                        const uint32_t dst = smem_u32(ps + (sl * 8 + 2 * cluster_rank() + half) * 64 +
                                                      (r - lane) + 4 * lane);
                        const uint32_t bar = smem_u32(&bars->psfull[sl]);
                        for (uint32_t t = 0; t < gridDim.x; ++t)
                            st_async_v4(map_to_rank(dst, t), g[0], g[1], g[2], g[3],
                                        map_to_rank(bar, t));
                    }
                    if (!__all_sync(0xffffffffu, wait(&bars->psfull[sl], (m >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    // the slot's next use is block m + 2 (whose sums may already be arriving)
                    if (warp == 6 && lane == 0) mbar_expect_tx(&bars->psfull[sl], kPsBytes * gridDim.x);
                    float tot = 0.f;
                    for (uint32_t i = 0; i < 2 * gridDim.x; ++i) tot += ps[(sl * 8 + i) * 64 + r];
                    const float inv = rsqrtf(tot / (float)dv + norm_eps);
#pragma unroll
                    for (int c = 0; c < NV / 2; ++c)
                        out[c] *= inv * (norm_w ? __ldg(norm_w + c0 + ch + c) : 1.f);
                }
                store_rows(out, j - 1);
            } else {
                warp_arrive(&bars->tfree[p]);
            }
        }
    } else {
        // ========================== state (TMEM lanes 0..127 = key channels)
        constexpr int SC = NV / 2;  // value channels per warp
        const int kc = 32 * (warp & 3) + lane;
        const int ch = SC * ((warp - 12) >> 2);
        const uint32_t lb = ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)ch;
        float Sr[SC];
#pragma unroll
        for (int c = 0; c < SC; ++c)
            Sr[c] = (S0 && kc < DK) ? S0[(bh * dv + c0 + ch + c) * DK + kc] : 0.f;
        auto write_sb = [&](int i) {
            if (kc < DK) {
#pragma unroll
                for (int c8 = 0; c8 < SC / 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm + L::SB + i * L::SB_BYTES +
                                               sw128_offset(kc, ch + c8 * 8, DK)) = pack8(Sr + c8 * 8);
            }
        };
        // S_{-1} = S_0 in copy 0 (read by b_0), S_0 in copy 1 (read by b_1)
        write_sb(0);
        write_sb(1);
        fence_async_smem();
        warp_arrive(&bars->s[0]);
        warp_arrive(&bars->s[1]);
        // Without delta these warps also order two reuses that the U chain
        // orders with delta: the late group (and with it the Delta S
        // accumulator of this parity and its dsf barrier) is released only
        // after Delta S is read, and a bf16 state copy is rewritten only after
        // b_{j-1}, its last reader, is done (emptyE).
        for (int j = 0; j <= nblk && ok; ++j) {
            const int p = j & 1;
            const uint32_t ph = (j >> 1) & 1, base = p * kParCols;
            ok = __all_sync(0xffffffffu, wait(&bars->fullL[p], ph));
            if (!ok) break;
            // the only late-group value read here: g_C', per key channel with the diagonal gate
            const float gC = GEN    ? vec_of(p)[kVgCGen + (kc & 127)]
                             : DIAG ? vec_of(p)[kVgCDiag + (kc & 127)]
                                    : vec_of(p)[kVgCPrev];
            if (DELTA) warp_arrive(&bars->emptyL[p]);
            ok = __all_sync(0xffffffffu, wait(&bars->dsf[p], ph));
            if (!ok) break;
            if (j >= 1) {
                tc_fence_after();
                float d[SC];
#pragma unroll
                for (int h = 0; h < SC / 16; ++h)
                    tmem_ld16(tmem + lb + base + kDS + 16 * h, *reinterpret_cast<float(*)[16]>(d + 16 * h));
                tmem_ld_wait(d);
                tc_fence_before();
                if (!DELTA) warp_arrive(&bars->emptyL[p]);
#pragma unroll
                for (int c = 0; c < SC; ++c) Sr[c] = gC * Sr[c] + d[c];
                if (j < nblk) {  // S_j -> copy (j+1)&1, read by b_{j+1}
                    if (!DELTA)
                        ok = __all_sync(0xffffffffu,
                                        wait(&bars->emptyE[(j - 1) & 1], ((j - 1) >> 1) & 1));
                    if (!ok) break;
                    write_sb((j + 1) & 1);
                    fence_async_smem();
                    warp_arrive(&bars->s[(j + 1) & 1]);
                }
            } else if (!DELTA) {
                warp_arrive(&bars->emptyL[p]);
            }
        }
        if (ok && kc < DK) {
#pragma unroll
            for (int c = 0; c < SC; ++c) ST[(bh * dv + c0 + ch + c) * DK + kc] = Sr[c];
        }
    }

    if (!ok) atomicExch(&g_tc_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kScanCols);
    // no CTA leaves while another may still write its partial-sum slots or
    // arrive on its barriers
    if (NORM) cluster_sync_all();
}

// ============================================================ tensor maps

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
// zero fill outside (also the columns of a box wider than d).
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

}  // namespace
}  // namespace lr
