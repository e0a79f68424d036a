// Thin wrappers over the sm_100-family tensor-core (tcgen05), tensor-memory
// and mbarrier PTX used by the chunked kernel.  Every wait is bounded: after
// kSpinLimit polls it gives up and reports failure to the caller, which sets
// an error word and leaves the kernel cleanly.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace lr {
namespace tc {

#ifndef LR_SPIN_LIMIT_LOG2
#define LR_SPIN_LIMIT_LOG2 26  // polls of a bounded wait: 2^26 by default
#endif
constexpr uint32_t kSpinLimit = 1u << LR_SPIN_LIMIT_LOG2;
// Poll limit of a kernel run under the failure-detection test hook.
constexpr uint32_t kFaultSpinLimit = 1u << 12;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Plain arrive (count 1) on `bar`.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Wait until the phase with the given parity has completed.  Returns false
// if the bounded spin ran out (after `limit` polls).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint32_t limit = kSpinLimit) {
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// ------------------------------------------------------------- clusters
// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address, in the shared memory of CTA `rank` of this cluster, of the object
// at shared-memory address `local` of this CTA.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// Store 16 bytes at cluster address `addr` (possibly in another CTA) and count
// them as transaction bytes on the mbarrier at cluster address `bar`, in the
// same CTA as `addr`.  As with a TMA copy, the bytes are in that CTA's shared
// memory once the barrier's phase completes, and a plain (CTA-scope) wait on
// the barrier orders the waiter's reads after them.  (An acquire at cluster
// scope would also do, but even one per warp and block costs the scan about
// 7 %: it stalls the SM's memory pipeline.)
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
        : "memory");
}
// Every thread of every CTA of the cluster (all threads must execute it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------- tensor memory (TMEM)
// Executed by one whole warp.  The allocated base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (lane_base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives
// lane (lane_base + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Wait for this thread's tensor-memory loads, then pin every register they
// wrote (the arrays passed) behind the wait: tcgen05.ld's outputs hold their
// values only after tcgen05.wait::ld, but nothing in the load's own asm tells
// the compiler so, and it may otherwise schedule a use of them above the
// wait (seen as rows of the mLSTM output that changed from call to call).
// Each array gets an empty asm with the values as in-out operands, ordered
// after the wait like every volatile asm.
template <int N>
__device__ __forceinline__ void tmem_pin(float (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}
template <typename A, typename... R>
__device__ __forceinline__ void tmem_ld_wait(A &a, R &...rest) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    tmem_pin(a);
    (tmem_pin(rest), ...);
}

// ---------------------------------------------------- matrix descriptors
// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: 8-row x 128-byte atoms (row r of an atom at byte 128*r,
// its 16-byte chunk c at chunk position c ^ r), atoms stacked along M/N
// every `sbo` bytes.  Bits: [0,14) start>>4, [16,30) leading offset>>4
// (unused for this layout, set to 1), [32,46) stride offset>>4, [46,49)
// fixed 0b001, [61,64) layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand with the 128-byte
// swizzle: the stored tile's rows are the K index (each 128-byte row holds 64
// consecutive M/N elements, 16-byte chunk c of row r at chunk position
// c ^ (r & 7)), 8-row K groups every 1024 bytes, 64-wide M/N blocks every
// `lbo` bytes.  `saddr` points at the first K row of the slice.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D,
// shape M x N.  Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16),
// [10,13) B format (1 = bf16), 15/16 A/B major (0 = K), [17,23) N>>3,
// [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// The same with A and/or B MN-major (bits 15 and 16).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_mn(int M, int N, bool a_mn, bool b_mn) {
    return idesc_bf16_f32(M, N) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (K = 16 for bf16).
// Issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------ swizzled tiles
// Byte offset of element (row, k) of a bf16 K-major tile stored as
// 128-byte-swizzled atoms: K is split into blocks of 64 elements; block kb
// holds all `rows` rows (rows a multiple of 8) contiguously at
// kb * rows * 128 bytes.  Tiles must start on a 1024-byte boundary.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
    const int kb = k >> 6;
    const int kin = k & 63;
    const int chunk = (kin >> 3) ^ (row & 7);
    return (uint32_t)(kb * rows * 128 + row * 128 + chunk * 16 + (kin & 7) * 2);
}

// The same descriptors advanced by K slice `ks` from slice 0 (the start
// address field moves; nothing else changes).
__device__ __forceinline__ uint64_t kdesc_step(uint64_t d0, int rows, int ks) {
    return d0 + (uint64_t)(((uint32_t)(ks >> 2) * (uint32_t)rows * 128u + (uint32_t)(ks & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t mndesc_step(uint64_t d0, int ks) {
    return d0 + (uint64_t)((uint32_t)ks * 128u);
}

// Descriptor of K slice `ks` of an MN-major tile laid out by
// sw128_offset(k, mn, krows) (rows = K index, 64-wide M/N blocks every
// krows * 128 bytes).
__device__ __forceinline__ uint64_t tile_desc_mn(uint32_t tile_saddr, int krows, int ks) {
    return desc_mnmajor_sw128(tile_saddr + (uint32_t)ks * 2048u, (uint32_t)krows * 128u);
}

// ------------------------------------------------------------- bulk copies
// Expect `bytes` more transaction bytes on `bar` and arrive once.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Global -> shared bulk copy (16-byte aligned, size a multiple of 16),
// completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global bulk copy (both 16-byte aligned, size a multiple of 16),
// tracked by the issuing thread's bulk-async group; commit and wait below.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed shared -> global bulk copy of this thread is done.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiled TMA load of a 3-D box (coordinates x innermost) into shared memory,
// completion counted on `bar`.  `map` is a __grid_constant__ CUtensorMap.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// Tiled TMA store of a 3-D box from shared memory (box elements outside the
// tensor are not written), tracked by the issuing thread's bulk-async group.
__device__ __forceinline__ void tma_store_3d(const void *map, const void *src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
                     "l"(map), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// Wait until every committed bulk store of this thread has finished reading
// shared memory (the writes to global memory may still be in flight).
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Hint: bring [p, p + bytes) into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Descriptor of the 16-wide K slice `ks` (K elements [16*ks, 16*ks+16)) of a
// tile laid out as above, restricted to rows [row0, row0 + M) (row0 % 8 == 0).
__device__ __forceinline__ uint64_t tile_desc(uint32_t tile_saddr, int rows, int row0, int ks) {
    const uint32_t kb = (uint32_t)(ks >> 2);
    const uint32_t addr = tile_saddr + kb * (uint32_t)rows * 128u + (uint32_t)row0 * 128u +
                          (uint32_t)(ks & 3) * 32u;
    return desc_kmajor_sw128(addr, 1024u);
}

}  // namespace tc
}  // namespace lr
