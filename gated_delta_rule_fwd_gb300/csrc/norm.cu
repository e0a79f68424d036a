// Output RMSNorm of the chunked forward (LR_FUSE_O_RMSNORM): every read-out
// row o_t (d_v channels of one head) divided by sqrt(mean(o_t^2) + eps) and
// multiplied channel-wise by a weight shared by the heads (page "Scrivere
// meglio nella memoria: gate e delta rule": the read-out of DeltaNet is
// stabilised by an RMSNorm).
//
// In place, HBM-bound (read o once, write it once).  Each lane owns 16
// contiguous bytes of a row, so a row is d_v * size / 16 lanes (4 to 32) and a
// warp covers 32 / that rows per access; the row's sum of squares reduces over
// its lanes with xor shuffles.  Each warp keeps kUnroll row groups of loads in
// flight.
#include "lr_internal.cuh"

namespace lr {
namespace {

constexpr int kNormThreads = 256;
constexpr int kUnroll = 4;

template <typename Tin> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float (&x)[4]) {
        const float4 r = *reinterpret_cast<const float4 *>(p);
        x[0] = r.x, x[1] = r.y, x[2] = r.z, x[3] = r.w;
    }
    __device__ static void store(float *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float (&x)[8]) {
        const uint4 r = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&x)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            const uint32_t lo = __bfloat16_as_ushort(h2.x), hi = __bfloat16_as_ushort(h2.y);
            w[i] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <typename Tin, int DV>
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(Tin *__restrict__ o, const float *__restrict__ w, float eps, size_t rows) {
    using V = Vec16<Tin>;
    constexpr int EPL = V::N;             // elements per lane
    constexpr int LPR = DV / EPL;         // lanes per row
    constexpr int RPW = 32 / LPR;         // rows per warp access
    static_assert(LPR >= 1 && LPR <= 32 && RPW * LPR == 32, "d_v must be 32, 64 or 128");
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const size_t warp = (size_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
    const size_t row0 = warp * (RPW * kUnroll) + lane / LPR;

    float wl[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) wl[e] = w ? w[sub * EPL + e] : 1.f;

    float x[kUnroll][EPL];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t r = row0 + (size_t)u * RPW;
        if (r < rows) {
            V::load(o + r * DV + sub * EPL, x[u]);
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[u][e] = 0.f;
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t r = row0 + (size_t)u * RPW;
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) ss += x[u][e] * x[u][e];
#pragma unroll
        for (int d = LPR / 2; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        const float inv = rsqrtf(ss / (float)DV + eps);
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[u][e] *= inv * wl[e];
        if (r < rows) V::store(o + r * DV + sub * EPL, x[u]);
    }
}

template <typename Tin, int DV>
cudaError_t launch_dv(void *o, const float *w, float eps, size_t rows, cudaStream_t stream) {
    constexpr int RPW = 32 / (DV / Vec16<Tin>::N);
    constexpr size_t rows_per_block = (size_t)(kNormThreads / 32) * RPW * kUnroll;
    const size_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
    rmsnorm_kernel<Tin, DV><<<(unsigned)blocks, kNormThreads, 0, stream>>>(static_cast<Tin *>(o),
                                                                          w, eps, rows);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_typed(void *o, const float *w, float eps, size_t rows, int dv,
                         cudaStream_t stream) {
    switch (dv) {
    case 32: return launch_dv<Tin, 32>(o, w, eps, rows, stream);
    case 64: return launch_dv<Tin, 64>(o, w, eps, rows, stream);
    default: return launch_dv<Tin, 128>(o, w, eps, rows, stream);
    }
}

}  // namespace

cudaError_t launch_rmsnorm(void *o, const float *w, float eps, size_t rows, int dv, lr_dtype dt,
                           cudaStream_t stream) {
    if (dt == LR_DT_F32) return launch_typed<float>(o, w, eps, rows, dv, stream);
    return launch_typed<__nv_bfloat16>(o, w, eps, rows, dv, stream);
}

}  // namespace lr
