// Host side of the C ABI declared in include/lr.h: argument validation,
// dispatch to the kernels, status mapping.  Validation happens before any
// launch, so an error status means nothing was enqueued.
#include <atomic>

#include "lr_internal.cuh"

namespace lr {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSlots = 208;
std::atomic<int> g_smem_bytes[kMaxDevices][kMaxSlots];

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    uintptr_t lo = 0, hi = 0;  // [lo, hi)
};
Span span(const void *p, size_t bytes) {
    Span s;
    if (p && bytes) {
        s.lo = reinterpret_cast<uintptr_t>(p);
        s.hi = s.lo + bytes;
    }
    return s;
}
bool overlap(Span a, Span b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool uses_alpha(lr_mode m) {
    return m == LR_MODE_DECAY || m == LR_MODE_GATED_DELTA || m == LR_MODE_DIAG_DECAY;
}
// fp32 values of alpha per token: one, or one per key channel for the diagonal gate
size_t alpha_per_token(lr_mode m, int dk) { return m == LR_MODE_DIAG_DECAY ? (size_t)dk : 1; }
bool uses_beta(lr_mode m) { return m == LR_MODE_DELTA || m == LR_MODE_GATED_DELTA; }

constexpr unsigned kFuseAll = LR_FUSE_QK_SILU_L2 | LR_FUSE_BETA_SIGMOID | LR_FUSE_ALPHA_SIGMOID |
                              LR_FUSE_ALPHA_SOFTPLUS | LR_FUSE_O_RMSNORM |
                              LR_FUSE_ALPHA_SIGMOID_POW;

// at most one alpha map
bool alpha_maps_ok(unsigned fl) {
    const unsigned a = fl & kAlphaMaps;
    return (a & (a - 1)) == 0;
}

// The kernels' view of lr_fuse: flags validated, the gate maps dropped where
// the mode has no such gate.
lr_status to_fuse(const lr_fuse *f, lr_mode mode, Fuse *out) {
    *out = Fuse{};
    if (!f) return LR_OK;
    unsigned fl = f->flags;
    if (fl & ~kFuseAll) return LR_ERR_FUSE;
    if (!alpha_maps_ok(fl)) return LR_ERR_FUSE;
    if ((fl & LR_FUSE_O_RMSNORM) && !(f->norm_eps >= 0.f && f->norm_eps <= 3.4e38f))
        return LR_ERR_FUSE;
    if (!uses_alpha(mode)) fl &= ~kAlphaMaps;
    if (!uses_beta(mode)) fl &= ~LR_FUSE_BETA_SIGMOID;
    out->flags = fl;
    out->ascale = (fl & kScaledAlphaMaps) ? f->alpha_scale : nullptr;
    out->norm_w = (fl & LR_FUSE_O_RMSNORM) ? f->norm_weight : nullptr;
    out->norm_eps = f->norm_eps;
    return LR_OK;
}

// Element counts fit comfortably in 64 bits and in what one device can hold.
bool count_ok(long long a, long long b, long long c, long long d) {
    const long long lim = 1ll << 40;
    long long x = a;
    for (long long f : {b, c, d}) {
        if (f <= 0) return f == 0;
        if (x > lim / f) return false;
        x *= f;
    }
    return true;
}

__global__ void copy_state_kernel(const float *__restrict__ src, float *__restrict__ dst,
                                  size_t n, float fill = 0.f) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : fill;
}

cudaError_t copy_state(const float *src, float *dst, size_t n, cudaStream_t stream,
                       float fill = 0.f) {
    if (src == dst || n == 0) return cudaSuccess;
    const size_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    copy_state_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, dst, n, fill);
    return cudaGetLastError();
}

}  // namespace

cudaError_t ensure_smem_attr(const void *fn, int bytes, int slot) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kMaxSlots)
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (g_smem_bytes[dev][slot].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_bytes[dev][slot].store(bytes, std::memory_order_release);
    return e;
}

}  // namespace lr

using namespace lr;

extern "C" {

int lr_abi_version(void) { return 3; }

const char *lr_status_string(lr_status s) {
    switch (s) {
    case LR_OK: return "ok";
    case LR_ERR_NULL: return "a required pointer is NULL";
    case LR_ERR_SHAPE: return "invalid size (negative, zero where not allowed, or too large)";
    case LR_ERR_DTYPE: return "unknown element type";
    case LR_ERR_ALIGN: return "a base pointer is not 16-byte aligned";
    case LR_ERR_MODE: return "unknown mode";
    case LR_ERR_UNSUPPORTED: return "unsupported size: dk and dv must be 32, 64 or 128 and chunk 64";
    case LR_ERR_CUDA: return "CUDA runtime error at launch";
    case LR_ERR_ALIAS: return "an output overlaps an input";
    case LR_ERR_TIMEOUT: return "a kernel gave up a bounded wait; its outputs are incomplete";
    case LR_ERR_WORKSPACE: return "workspace is NULL or smaller than lr_fwd_chunked_workspace_size";
    case LR_ERR_TOO_LARGE: return "problem needs more scratch than the static workspace holds (LR_STATIC_WORKSPACE_BYTES)";
    case LR_ERR_FUSE: return "invalid lr_fuse: unknown flag, both alpha maps, or a negative or non-finite norm_eps";
    }
    return "unknown status";
}

static lr_status check_chunked_shape(int B, int H, int T, int dk, int dv, int chunk, lr_dtype dt,
                                     lr_mode mode) {
    if (mode < LR_MODE_LINEAR || mode > LR_MODE_DIAG_DECAY) return LR_ERR_MODE;
    if (dt != LR_DT_F32 && dt != LR_DT_BF16) return LR_ERR_DTYPE;
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1) return LR_ERR_SHAPE;
    if (!count_ok(B, H, T, dk > dv ? dk : dv) || !count_ok(B, H, dv, dk)) return LR_ERR_SHAPE;
    if (!supported_dim(dk) || !supported_dim(dv) || chunk != 64) return LR_ERR_UNSUPPORTED;
    return LR_OK;
}

size_t lr_fwd_chunked_fused_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                           lr_dtype dt, lr_mode mode, unsigned flags) {
    if (check_chunked_shape(B, H, T, dk, dv, chunk, dt, mode) != LR_OK) return 0;
    if ((flags & ~kFuseAll) || !alpha_maps_ok(flags))
        return 0;
    if (dt != LR_DT_BF16 || T == 0) return 0;
    return chunked_tc_workspace_bytes(B, H, T, dk, mode, flags);
}

size_t lr_fwd_chunked_workspace_size(int B, int H, int T, int dk, int dv, int chunk, lr_dtype dt,
                                     lr_mode mode) {
    return lr_fwd_chunked_fused_workspace_size(B, H, T, dk, dv, chunk, dt, mode, 0u);
}

lr_status lr_fwd_chunked_fused(const void *q, const void *k, const void *v, const float *alpha,
                               const float *beta, const float *S0, void *o, float *S_T, int B,
                               int H, int T, int dk, int dv, int chunk, lr_dtype dt, lr_mode mode,
                               const lr_fuse *fuse, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    const lr_status shape = check_chunked_shape(B, H, T, dk, dv, chunk, dt, mode);
    if (shape != LR_OK) return shape;
    Fuse fz;
    const lr_status fs = to_fuse(fuse, mode, &fz);
    if (fs != LR_OK) return fs;
    if (!S_T) return LR_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !o)) return LR_ERR_NULL;
    if (T > 0 && uses_alpha(mode) && !alpha) return LR_ERR_NULL;
    if (T > 0 && uses_beta(mode) && !beta) return LR_ERR_NULL;
    if (T > 0 && (fz.flags & kScaledAlphaMaps) && !fz.ascale) return LR_ERR_NULL;
    const size_t need =
        lr_fwd_chunked_fused_workspace_size(B, H, T, dk, dv, chunk, dt, mode, fz.flags);
    if (need > 0 && (!workspace || workspace_bytes < need)) return LR_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) ||
        !aligned16(beta) || !aligned16(S0) || !aligned16(o) || !aligned16(S_T) ||
        (need > 0 && !aligned16(workspace)) || !aligned16(fz.ascale) || !aligned16(fz.norm_w))
        return LR_ERR_ALIGN;

    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t bht = (size_t)B * H * T;
    const size_t state_bytes = (size_t)B * H * dv * dk * 4;
    const Span sq = span(q, bht * dk * es), sk = span(k, bht * dk * es),
               sv = span(v, bht * dv * es);
    const Span sa = span(uses_alpha(mode) ? alpha : nullptr, bht * alpha_per_token(mode, dk) * 4);
    const Span sb = span(uses_beta(mode) ? beta : nullptr, bht * 4);
    const Span s0 = span(S0, state_bytes), so = span(o, bht * dv * es),
               st = span(S_T, state_bytes);
    for (Span in : {sq, sk, sv, sa, sb, s0, st})
        if (overlap(so, in)) return LR_ERR_ALIAS;
    for (Span in : {sq, sk, sv, sa, sb})
        if (overlap(st, in)) return LR_ERR_ALIAS;
    if (S0 && S0 != S_T && overlap(s0, st)) return LR_ERR_ALIAS;
    const Span sw = span(need > 0 ? workspace : nullptr, need);
    for (Span other : {sq, sk, sv, sa, sb, s0, so, st})
        if (overlap(sw, other)) return LR_ERR_ALIAS;
    const Span sc = span(fz.ascale, (size_t)H * 4), sn = span(fz.norm_w, (size_t)dv * 4);
    for (Span out : {so, st, sw})
        if (overlap(out, sc) || overlap(out, sn)) return LR_ERR_ALIAS;

    cudaError_t e;
    if (T == 0) {
        if (S0 == S_T) return LR_OK;
        const size_t n = (size_t)B * H * dv * dk;
        copy_state_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0,
                            stream>>>(S0, S_T, n);
        e = cudaGetLastError();
    } else {
        e = dt == LR_DT_BF16
                ? launch_chunked_tc(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, mode, fz,
                                    workspace, stream)
                : launch_chunked_simt(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, dt, mode,
                                      fz, stream);
        const bool folded = dt == LR_DT_BF16 && chunked_tc_applies_norm(mode, B, H, dv);
        if (e == cudaSuccess && (fz.flags & LR_FUSE_O_RMSNORM) && !folded)
            e = launch_rmsnorm(o, fz.norm_w, fz.norm_eps, (size_t)B * H * T, dv, dt, stream);
    }
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_fwd_chunked(const void *q, const void *k, const void *v, const float *alpha,
                         const float *beta, const float *S0, void *o, float *S_T, int B, int H,
                         int T, int dk, int dv, int chunk, lr_dtype dt, lr_mode mode,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return lr_fwd_chunked_fused(q, k, v, alpha, beta, S0, o, S_T, B, H, T, dk, dv, chunk, dt, mode,
                                nullptr, workspace, workspace_bytes, stream);
}

size_t lr_fwd_chunked_mlstm_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                           lr_dtype dt) {
    if (check_chunked_shape(B, H, T, dk, dv, chunk, dt, LR_MODE_DECAY) != LR_OK) return 0;
    if (dt != LR_DT_BF16 || T == 0) return 0;
    return mlstm_workspace_bytes(B, H, T, dk);
}

lr_status lr_fwd_chunked_mlstm(const void *q, const void *k, const void *v, const float *fgate,
                               const float *igate, const float *C0, const float *n0,
                               const float *m0, void *h, float *C_T, float *n_T, float *m_T,
                               int B, int H, int T, int dk, int dv, int chunk, lr_dtype dt,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const lr_status shape = check_chunked_shape(B, H, T, dk, dv, chunk, dt, LR_MODE_DECAY);
    if (shape != LR_OK) return shape;
    if (!C_T || !n_T || !m_T) return LR_ERR_NULL;
    if ((C0 || n0 || m0) && !(C0 && n0 && m0)) return LR_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !h || !fgate || !igate)) return LR_ERR_NULL;
    const size_t need = lr_fwd_chunked_mlstm_workspace_size(B, H, T, dk, dv, chunk, dt);
    if (need > 0 && (!workspace || workspace_bytes < need)) return LR_ERR_WORKSPACE;
    for (const void *p : {q, k, v, (const void *)fgate, (const void *)igate, (const void *)C0,
                          (const void *)n0, (const void *)m0, (const void *)h, (const void *)C_T,
                          (const void *)n_T, (const void *)m_T})
        if (!aligned16(p)) return LR_ERR_ALIGN;
    if (need > 0 && !aligned16(workspace)) return LR_ERR_ALIGN;

    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t bh = (size_t)B * H, bht = bh * T;
    const Span sq = span(q, bht * dk * es), sk = span(k, bht * dk * es), sv = span(v, bht * dv * es);
    const Span sf = span(fgate, bht * 4), si = span(igate, bht * 4);
    const Span c0 = span(C0, bh * dv * dk * 4), n0s = span(n0, bh * dk * 4), m0s = span(m0, bh * 4);
    const Span sh = span(h, bht * dv * es), ct = span(C_T, bh * dv * dk * 4),
               nt = span(n_T, bh * dk * 4), mt = span(m_T, bh * 4);
    const Span sw = span(need > 0 ? workspace : nullptr, need);
    for (Span in : {sq, sk, sv, sf, si, c0, n0s, m0s, ct, nt, mt, sw})
        if (overlap(sh, in)) return LR_ERR_ALIAS;
    // each final state may be its own initial state, and overlaps nothing else
    const Span outs[3] = {ct, nt, mt};
    const void *own[3] = {C0, n0, m0};
    const void *outp[3] = {C_T, n_T, m_T};
    const Span ins[3] = {c0, n0s, m0s};
    for (int a = 0; a < 3; ++a) {
        for (Span in : {sq, sk, sv, sf, si, sw})
            if (overlap(outs[a], in)) return LR_ERR_ALIAS;
        for (int b = 0; b < 3; ++b) {
            if (b != a && overlap(outs[a], outs[b])) return LR_ERR_ALIAS;
            if (overlap(outs[a], ins[b]) && !(a == b && own[a] == outp[a])) return LR_ERR_ALIAS;
        }
    }
    for (Span in : {sq, sk, sv, sf, si, c0, n0s, m0s})
        if (overlap(sw, in)) return LR_ERR_ALIAS;

    cudaError_t e;
    if (T == 0) {
        e = copy_state(C0, C_T, bh * dv * dk, stream);
        if (e == cudaSuccess) e = copy_state(n0, n_T, bh * dk, stream);
        if (e == cudaSuccess) e = copy_state(m0, m_T, bh, stream, -INFINITY);
    } else {
        e = launch_mlstm_chunked(q, k, v, fgate, igate, C0, n0, m0, h, C_T, n_T, m_T, B, H, T, dk,
                                 dv, dt, workspace, stream);
    }
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_step_mlstm(const void *q, const void *k, const void *v, const float *fgate,
                        const float *igate, float *C, float *n, float *m, void *h, int N, int H,
                        int dk, int dv, lr_dtype dt, cudaStream_t stream) {
    if (dt != LR_DT_F32 && dt != LR_DT_BF16) return LR_ERR_DTYPE;
    if (N < 1 || H < 1 || dk < 1 || dv < 1) return LR_ERR_SHAPE;
    if (!count_ok(N, H, dv, dk) || (long long)N * H > 0x7fffffffll) return LR_ERR_SHAPE;
    if (!supported_dim(dk) || !supported_dim(dv)) return LR_ERR_UNSUPPORTED;
    if (!q || !k || !v || !fgate || !igate || !C || !n || !m || !h) return LR_ERR_NULL;
    for (const void *p : {q, k, v, (const void *)fgate, (const void *)igate, (const void *)C,
                          (const void *)n, (const void *)m, (const void *)h})
        if (!aligned16(p)) return LR_ERR_ALIGN;
    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t nh = (size_t)N * H;
    const Span sq = span(q, nh * dk * es), sk = span(k, nh * dk * es), sv = span(v, nh * dv * es);
    const Span sf = span(fgate, nh * 4), si = span(igate, nh * 4), sh = span(h, nh * dv * es);
    const Span sc = span(C, nh * dv * dk * 4), sn = span(n, nh * dk * 4), sm = span(m, nh * 4);
    for (Span in : {sq, sk, sv, sf, si, sc, sn, sm})
        if (overlap(sh, in)) return LR_ERR_ALIAS;
    for (Span st : {sc, sn, sm})
        for (Span in : {sq, sk, sv, sf, si})
            if (overlap(st, in)) return LR_ERR_ALIAS;
    if (overlap(sc, sn) || overlap(sc, sm) || overlap(sn, sm)) return LR_ERR_ALIAS;
    const cudaError_t e = launch_mlstm_step(q, k, v, fgate, igate, C, n, m, h, N, H, dk, dv, dt,
                                            stream);
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

size_t lr_fwd_chunked_gen_delta_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                               lr_dtype dt) {
    if (check_chunked_shape(B, H, T, dk, dv, chunk, dt, LR_MODE_DELTA) != LR_OK) return 0;
    if (dt != LR_DT_BF16 || T == 0) return 0;
    return gen_delta_tc_workspace_bytes(B, H, T, dk);
}

lr_status lr_fwd_chunked_gen_delta(const void *q, const void *kw, const void *v, const float *w,
                                   const float *kappa, const float *a, const float *S0, void *o,
                                   float *S_T, int B, int H, int T, int dk, int dv, int chunk,
                                   lr_dtype dt, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
    const lr_status shape = check_chunked_shape(B, H, T, dk, dv, chunk, dt, LR_MODE_DELTA);
    if (shape != LR_OK) return shape;
    if (!S_T) return LR_ERR_NULL;
    if (T > 0 && (!q || !kw || !v || !w || !kappa || !a || !o)) return LR_ERR_NULL;
    const size_t need = lr_fwd_chunked_gen_delta_workspace_size(B, H, T, dk, dv, chunk, dt);
    if (need > 0 && (!workspace || workspace_bytes < need)) return LR_ERR_WORKSPACE;
    for (const void *p : {q, kw, v, (const void *)w, (const void *)kappa, (const void *)a,
                          (const void *)S0, (const void *)o, (const void *)S_T})
        if (!aligned16(p)) return LR_ERR_ALIGN;
    if (need > 0 && !aligned16(workspace)) return LR_ERR_ALIGN;
    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t bht = (size_t)B * H * T, state = (size_t)B * H * dv * dk * 4;
    const Span sq = span(q, bht * dk * es), sk = span(kw, bht * dk * es), sv = span(v, bht * dv * es);
    const Span sw = span(w, bht * dk * 4), sc = span(kappa, bht * dk * 4), sa = span(a, bht * dk * 4);
    const Span s0 = span(S0, state), so = span(o, bht * dv * es), st = span(S_T, state);
    const Span sws = span(need > 0 ? workspace : nullptr, need);
    for (Span in : {sq, sk, sv, sw, sc, sa, s0, st, sws})
        if (overlap(so, in)) return LR_ERR_ALIAS;
    for (Span in : {sq, sk, sv, sw, sc, sa, sws})
        if (overlap(st, in)) return LR_ERR_ALIAS;
    for (Span in : {sq, sk, sv, sw, sc, sa, s0})
        if (overlap(sws, in)) return LR_ERR_ALIAS;
    if (S0 && S0 != S_T && overlap(s0, st)) return LR_ERR_ALIAS;
    cudaError_t e;
    if (T == 0)
        e = copy_state(S0, S_T, (size_t)B * H * dv * dk, stream);
    else if (dt == LR_DT_BF16)
        e = launch_gen_delta_tc(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dk, dv, workspace,
                                stream);
    else
        e = launch_gen_delta_chunked(q, kw, v, w, kappa, a, S0, o, S_T, B, H, T, dk, dv, dt,
                                     stream);
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_step_gen_delta(const void *q, const void *kw, const void *v, const float *w,
                            const float *kappa, const float *a, float *S, void *o, int N, int H,
                            int dk, int dv, lr_dtype dt, cudaStream_t stream) {
    if (dt != LR_DT_F32 && dt != LR_DT_BF16) return LR_ERR_DTYPE;
    if (N < 1 || H < 1 || dk < 1 || dv < 1) return LR_ERR_SHAPE;
    if (!count_ok(N, H, dv, dk) || (long long)N * H > 0x7fffffffll) return LR_ERR_SHAPE;
    if (!supported_dim(dk) || !supported_dim(dv)) return LR_ERR_UNSUPPORTED;
    if (!q || !kw || !v || !w || !kappa || !a || !S || !o) return LR_ERR_NULL;
    for (const void *p : {q, kw, v, (const void *)w, (const void *)kappa, (const void *)a,
                          (const void *)S, (const void *)o})
        if (!aligned16(p)) return LR_ERR_ALIGN;
    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t nh = (size_t)N * H;
    const Span sq = span(q, nh * dk * es), sk = span(kw, nh * dk * es), sv = span(v, nh * dv * es);
    const Span sw = span(w, nh * dk * 4), sc = span(kappa, nh * dk * 4), sa = span(a, nh * dk * 4);
    const Span ss = span(S, nh * dv * dk * 4), so = span(o, nh * dv * es);
    for (Span in : {sq, sk, sv, sw, sc, sa, ss})
        if (overlap(so, in)) return LR_ERR_ALIAS;
    for (Span in : {sq, sk, sv, sw, sc, sa})
        if (overlap(ss, in)) return LR_ERR_ALIAS;
    const cudaError_t e = launch_gen_delta_step(q, kw, v, w, kappa, a, S, o, N, H, dk, dv, dt,
                                                stream);
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return LR_ERR_CUDA;
    const int e = read_and_clear_tc_error(), eg = read_and_clear_gd_tc_error();
    if (e < 0 || eg < 0) return LR_ERR_CUDA;
    return (e || eg) ? LR_ERR_TIMEOUT : LR_OK;
}

lr_status lr_debug_inject_scan_timeout(int on) {
    if (cudaDeviceSynchronize() != cudaSuccess) return LR_ERR_CUDA;
    return set_scan_fault_tc(on ? 1u : 0u) == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_step_fused(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                        lr_dtype dt, lr_mode mode, const lr_fuse *fuse, cudaStream_t stream) {
    if (mode < LR_MODE_LINEAR || mode > LR_MODE_DIAG_DECAY) return LR_ERR_MODE;
    if (dt != LR_DT_F32 && dt != LR_DT_BF16) return LR_ERR_DTYPE;
    if (N < 1 || H < 1 || dk < 1 || dv < 1) return LR_ERR_SHAPE;
    if (!count_ok(N, H, dv, dk) || (long long)N * H > 0x7fffffffll) return LR_ERR_SHAPE;
    if (!supported_dim(dk) || !supported_dim(dv)) return LR_ERR_UNSUPPORTED;
    Fuse fz;
    const lr_status fs = to_fuse(fuse, mode, &fz);
    if (fs != LR_OK) return fs;
    if (!q || !k || !v || !S || !o) return LR_ERR_NULL;
    if (uses_alpha(mode) && !alpha) return LR_ERR_NULL;
    if (uses_beta(mode) && !beta) return LR_ERR_NULL;
    if ((fz.flags & kScaledAlphaMaps) && !fz.ascale) return LR_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) ||
        !aligned16(beta) || !aligned16(S) || !aligned16(o) || !aligned16(fz.ascale) ||
        !aligned16(fz.norm_w))
        return LR_ERR_ALIGN;

    const size_t es = dt == LR_DT_F32 ? 4 : 2;
    const size_t nh = (size_t)N * H;
    const Span sq = span(q, nh * dk * es), sk = span(k, nh * dk * es), sv = span(v, nh * dv * es);
    const Span sa = span(uses_alpha(mode) ? alpha : nullptr, nh * alpha_per_token(mode, dk) * 4);
    const Span sb = span(uses_beta(mode) ? beta : nullptr, nh * 4);
    const Span ss = span(S, nh * dv * dk * 4), so = span(o, nh * dv * es);
    for (Span in : {sq, sk, sv, sa, sb, ss})
        if (overlap(so, in)) return LR_ERR_ALIAS;
    for (Span in : {sq, sk, sv, sa, sb})
        if (overlap(ss, in)) return LR_ERR_ALIAS;
    const Span sc = span(fz.ascale, (size_t)H * 4), sn = span(fz.norm_w, (size_t)dv * 4);
    for (Span out : {so, ss})
        if (overlap(out, sc) || overlap(out, sn)) return LR_ERR_ALIAS;

    const cudaError_t e =
        launch_step(q, k, v, alpha, beta, S, o, N, H, dk, dv, dt, mode, fz, stream);
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

lr_status lr_step(const void *q, const void *k, const void *v, const float *alpha,
                  const float *beta, float *S, void *o, int N, int H, int dk, int dv,
                  lr_dtype dt, lr_mode mode, cudaStream_t stream) {
    return lr_step_fused(q, k, v, alpha, beta, S, o, N, H, dk, dv, dt, mode, nullptr, stream);
}

}  // extern "C"
