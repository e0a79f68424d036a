/*
 * lr.h -- C ABI of the GB300 (sm_103a) library for the fixed-size
 * linear-attention memory S_t (d_v x d_k) under the gated delta rule.
 *
 * The operation (page "Scrivere meglio nella memoria: gate e delta rule",
 * section "Unire oblio e correzione: Gated DeltaNet", and the summary table of
 * the same page):
 *
 *     S_t = S_{t-1} [ alpha_t (I - beta_t k_t k_t^T) ] + beta_t v_t k_t^T
 *     o_t = S_t q_t                     (read-out after the write of token t)
 *
 * and its special cases, selected by lr_mode.  S has value channels as rows
 * and key channels as columns, so o = S q (same page, gates section, on the
 * side from which a transition multiplies).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no memory at run time and keeps no state between calls other
 *     than per-device kernel attributes set once and the fixed scratch array
 *     used by lr_fwd_chunked_noalloc (part of the loaded module).
 *   - Tensors are contiguous and row-major with the shapes given below; base
 *     pointers must be 16-byte aligned (else LR_ERR_ALIGN).
 *   - alpha, beta and the state are always fp32; q, k, v and o have the
 *     element type given by lr_dtype.
 *   - Arguments are validated on the host, before any launch; a call that
 *     returns an error status launched nothing and wrote nothing.
 *   - Work is enqueued on `stream`; the call returns without synchronising.
 *     Faults inside a kernel surface at the caller's next synchronisation
 *     (LR_ERR_CUDA is returned only for launch failures reported at once).
 *   - Values are not validated.  The documented domain is alpha in (0, 1],
 *     beta in [0, 1]; NaN and Inf propagate.
 *   - No exceptions cross the ABI.  Calls on different streams are
 *     independent; calls that write the same buffers race.
 */
#ifndef LR_H_
#define LR_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LR_OK = 0,
    LR_ERR_NULL = 1,        /* a required pointer is NULL                         */
    LR_ERR_SHAPE = 2,       /* a size is negative, zero where it must not be, or
                               the element count overflows                          */
    LR_ERR_DTYPE = 3,       /* unknown lr_dtype                                    */
    LR_ERR_ALIGN = 4,       /* a base pointer is not 16-byte aligned               */
    LR_ERR_MODE = 5,        /* unknown lr_mode                                     */
    LR_ERR_UNSUPPORTED = 6, /* valid but not implemented: d_k or d_v outside
                               {32, 64, 128}, or chunk != 64                       */
    LR_ERR_CUDA = 7,        /* the CUDA runtime reported an error at launch        */
    LR_ERR_ALIAS = 8,       /* an output overlaps an input it must not overlap     */
    LR_ERR_TIMEOUT = 9,     /* a kernel gave up a bounded wait (see lr_device_status) */
    LR_ERR_WORKSPACE = 10,  /* workspace NULL or smaller than lr_fwd_chunked_workspace_size */
    LR_ERR_TOO_LARGE = 11,  /* lr_fwd_chunked_noalloc: the problem needs more scratch
                               than LR_STATIC_WORKSPACE_BYTES */
    LR_ERR_FUSE = 12        /* lr_fuse: unknown flag bits, two alpha maps at once,
                               or norm_eps negative or not finite */
} lr_status;

/* Which row of the family (summary table of the first page). */
typedef enum {
    /* S_t = S_{t-1} + v_t k_t^T  (plain accumulation, opening section).
       alpha and beta are ignored and may be NULL. */
    LR_MODE_LINEAR = 0,
    /* S_t = alpha_t S_{t-1} + v_t k_t^T  (scalar gate: RetNet with a fixed
       per-head gamma broadcast by the caller, or a Mamba-2-style data-dependent
       alpha; section "Dimenticare: i gate").  beta is ignored, may be NULL. */
    LR_MODE_DECAY = 1,
    /* S_t = S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T  (delta rule,
       section "Correggere: la delta rule").  alpha is ignored, may be NULL. */
    LR_MODE_DELTA = 2,
    /* S_t = S_{t-1} [alpha_t (I - beta_t k_t k_t^T)] + beta_t v_t k_t^T
       (Gated DeltaNet).  Both alpha and beta are required. */
    LR_MODE_GATED_DELTA = 3,
    /* S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T  (the diagonal gate of GLA,
       section "Dimenticare: i gate": one gate per key channel, multiplying
       from the right, so column c of S decays by alpha_t[c]).  alpha has one
       value per key channel: [B, H, T, dk] for lr_fwd_chunked, [N, H, dk] for
       lr_step.  beta is ignored, may be NULL.  The chunked form computes the
       scores of a 64-token block in 16-token sub-blocks (the second level of
       blocks GLA needs for numerical stability, summary of the same page):
       the per-channel decay across any 16 consecutive tokens of a block must
       stay above e^-80 (an average gate above 0.007), else those scores are
       inexact. */
    LR_MODE_DIAG_DECAY = 4
} lr_mode;

/* Element type of q, k, v and o. */
typedef enum {
    LR_DT_F32 = 0,  /* fp32 in and out; computed in fp32 on CUDA cores          */
    LR_DT_BF16 = 1  /* bf16 in and out; bf16 tensor-core products with fp32
                       accumulation, fp32 state                               */
} lr_dtype;

/*
 * Chunkwise forward over whole sequences (prefill).
 *
 * Computes, for every (b, h), the recurrence over t = 0..T-1 from S0 and
 * returns every read-out and the final state.  The sequence is processed in
 * blocks of `chunk` tokens: inside a block all tokens are computed together
 * (decay-masked scores and, for the delta rows, the pseudo-value triangular
 * system of the WY representation -- first page, section "Correggere: la
 * delta rule"); only the end-of-block state passes from one block to the next
 * (page "Le architetture lineari: RetNet, RWKV, xLSTM", section "RetNet: la
 * retention e le sue tre forme", chunkwise form).  The result equals the
 * sequential recurrence up to rounding.  A final block shorter than `chunk`
 * is handled.
 *
 *   q      [B, H, T, dk]   dtype dt
 *   k      [B, H, T, dk]   dtype dt
 *   v      [B, H, T, dv]   dtype dt
 *   alpha  [B, H, T]       fp32; required for DECAY and GATED_DELTA;
 *                          [B, H, T, dk] for DIAG_DECAY
 *   beta   [B, H, T]       fp32; required for DELTA and GATED_DELTA
 *   S0     [B, H, dv, dk]  fp32 initial state, or NULL for zeros
 *   o      [B, H, T, dv]   dtype dt, written; must not overlap any input
 *   S_T    [B, H, dv, dk]  fp32 final state, written; may be the same pointer
 *                          as S0 (in-place update), must not overlap anything
 *                          else
 *   B, H >= 1; T >= 0 (T == 0 copies S0, or zeros, to S_T);
 *   dk, dv in {32, 64, 128}; chunk == 64.
 *   workspace       device scratch of at least
 *                   lr_fwd_chunked_workspace_size(...) bytes, 16-byte aligned,
 *                   owned by the caller and not overlapping any argument; its
 *                   contents on entry do not matter and are undefined on exit.
 *                   May be NULL when that size is 0.
 *   workspace_bytes its size in bytes.
 *
 * The bf16 path runs two kernels on `stream`: a per-block pass over all
 * blocks in parallel (gate products, decay-masked scores, the UT inverse of
 * the delta rows, W = T diag(beta g) K and the block-to-block coupling
 * W K'^T of consecutive blocks), stored in the workspace, then the
 * sequential pass over blocks that carries the state.  The fp32 path needs no
 * workspace.  Calls that share a workspace must be ordered on one stream.
 *
 * q, k, v and o may be NULL when T == 0.
 */
lr_status lr_fwd_chunked(const void *q, const void *k, const void *v,
                         const float *alpha, const float *beta,
                         const float *S0, void *o, float *S_T,
                         int B, int H, int T, int dk, int dv, int chunk,
                         lr_dtype dt, lr_mode mode,
                         void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * Bytes of workspace lr_fwd_chunked needs for these arguments: 0 for the fp32
 * path and for T == 0; for bf16, 41 KB per (batch, head) for every 64-token
 * block plus one more, at dk = 128 (33 KB at dk = 32 or 64).  Returns 0 as well for arguments lr_fwd_chunked would
 * reject.
 */
size_t lr_fwd_chunked_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                     lr_dtype dt, lr_mode mode);

/*
 * One recurrent step for N independent sequences (decode).  Per (n, h) and
 * per value channel r independently, with s = S[r, :] (page "Le architetture
 * lineari", recurrent form, O(d^2) per token and fixed memory):
 *
 *     a   = alpha (1 for LINEAR and DELTA)
 *     u_r = beta (v_r - a s.k)   for DELTA / GATED_DELTA,   v_r otherwise
 *     S[r, :] <- a s + u_r k
 *     o_r     =  a (s.q) + u_r (k.q)        ( = S_new[r, :] . q )
 *
 *   q, k   [N, H, dk]       dtype dt
 *   v      [N, H, dv]       dtype dt
 *   alpha  [N, H]           fp32 (required for DECAY, GATED_DELTA);
 *                           [N, H, dk] for DIAG_DECAY (then a is the vector
 *                           alpha and S[r, :] <- a * s + v_r k, o_r = S[r,:] . q)
 *   beta   [N, H]           fp32 (required for DELTA, GATED_DELTA)
 *   S      [N, H, dv, dk]   fp32, read and updated IN PLACE
 *   o      [N, H, dv]       dtype dt, written; must not overlap S or inputs
 *   N, H >= 1; dk, dv in {32, 64, 128}.
 */
lr_status lr_step(const void *q, const void *k, const void *v,
                  const float *alpha, const float *beta, float *S, void *o,
                  int N, int H, int dk, int dv, lr_dtype dt, lr_mode mode,
                  cudaStream_t stream);

/*
 * Reports, then clears, the error word that kernels of this library set on
 * the current device when a bounded wait inside them gave up (a tensor-core
 * completion signal that never arrived); such a kernel stops early and its
 * outputs are incomplete.  Synchronises the current device first.
 * Returns LR_OK, LR_ERR_TIMEOUT, or LR_ERR_CUDA if the device cannot be
 * queried.
 */
lr_status lr_device_status(void);

/*
 * Failure-detection test hook (no counterpart on the pages).  While it is on
 * (on != 0), every launch of the chunked forward's bf16 sequential pass on
 * the current device polls each of its barriers at most a few thousand times
 * and its late-group load thread skips the tile loads of stage 1, so every
 * role's wait for that stage gives up: the kernel stops, waits for its own
 * copies and tensor-core products in flight, frees its tensor memory, sets
 * the error word and returns (lr_device_status then reports
 * LR_ERR_TIMEOUT).  Outputs of such a call are undefined.  Nothing faults and
 * nothing waits without a limit.  Synchronises the device; call with 0 to
 * restore normal operation.  Returns LR_OK, or LR_ERR_CUDA if the hook could
 * not be set.
 */
lr_status lr_debug_inject_scan_timeout(int on);

/*
 * Chunked forward without any allocation by the caller.  No counterpart on
 * the pages: this is a deployment variant of lr_fwd_chunked.
 *
 * For callers that cannot allocate device memory -- code inside a host
 * framework that owns all device memory and gives its plug-ins no allocator,
 * or code on a path where cudaMalloc must not run because it can synchronise
 * the device or fail at an unpredictable time.  Same arguments and result as
 * lr_fwd_chunked, without the workspace: the scratch comes from a fixed
 * array of LR_STATIC_WORKSPACE_BYTES in the library's own device memory,
 * which every GPU that loads the library holds until the process exits.
 *
 *   - Returns LR_ERR_TOO_LARGE, launching nothing, when
 *     lr_fwd_chunked_workspace_size(...) for the same arguments exceeds
 *     LR_STATIC_WORKSPACE_BYTES; that function is the rule for every mode.
 *     (For the modes with a scalar gate or none at dk = 128 the scratch is
 *     41 KB per (batch, head) for every 64-token block plus one, so
 *     B * H * (ceil(T / 64) + 1) <= 1598; LR_MODE_DIAG_DECAY also keeps
 *     its transformed q and k there, 2 * B * H * T * dk * 2 bytes more.)
 *   - The first call on a device looks up the array's device address (with
 *     cudaGetSymbolAddress, that device current) and keeps it for the rest
 *     of the process: make that first call before any stream capture, and do
 *     not reset the device (cudaDeviceReset) while the library is loaded.
 *   - Every call uses the same array: calls that may run at the same time on
 *     the GPU (other streams, other host threads) race and must be ordered by
 *     the caller.  No clearing is needed between calls.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define LR_STATIC_WORKSPACE_BYTES (64u << 20)

lr_status lr_fwd_chunked_noalloc(const void *q, const void *k, const void *v,
                                 const float *alpha, const float *beta,
                                 const float *S0, void *o, float *S_T,
                                 int B, int H, int T, int dk, int dv, int chunk,
                                 lr_dtype dt, lr_mode mode, cudaStream_t stream);

/*
 * Fused entry points: the maps that sit on either side of the recurrence,
 * applied inside the library's kernels, so that the caller passes
 * pre-activation values and receives the normalised read-out (page "Scrivere
 * meglio nella memoria: gate e delta rule"):
 *
 *   LR_FUSE_QK_SILU_L2      q_t <- SiLU(q_t) / max(||SiLU(q_t)||_2, 1e-12), the
 *                           same for k_t, per token over the d_k channels
 *                           (opening section: DeltaNet's feature map on keys
 *                           and queries, which keeps the eigenvalues of
 *                           I - beta k k^T in [0, 1])
 *   LR_FUSE_BETA_SIGMOID    beta_t <- sigmoid(beta_t)  (section "Correggere: la
 *                           delta rule": a write strength between 0 and 1)
 *   LR_FUSE_ALPHA_SIGMOID   alpha_t <- sigmoid(alpha_t)
 *   LR_FUSE_ALPHA_SOFTPLUS  alpha_t <- exp(-c_h softplus(alpha_t)), c_h =
 *                           alpha_scale[h]  (section "Dimenticare: i gate":
 *                           a decay computed from the input; the page leaves
 *                           the parametrisation open, these are the two in
 *                           common use)
 *   LR_FUSE_ALPHA_SIGMOID_POW  alpha_t <- sigmoid(alpha_t)^c_h, c_h =
 *                           alpha_scale[h]  (the same section: GLA's gate, a
 *                           sigmoid raised to 1/tau, tau = 16, per key channel)
 *   LR_FUSE_O_RMSNORM       o_t <- o_t / sqrt(mean_r o_t[r]^2 + norm_eps) *
 *                           norm_weight, per token over the d_v channels of a
 *                           head (same page, the read-out of DeltaNet is
 *                           stabilised by an RMSNorm)
 *
 * The alpha maps apply only in modes that use alpha, the beta map only in
 * modes that use beta; the other flags apply in every mode.  The state is
 * never normalised.  Gates are evaluated in fp32; ln alpha is formed directly
 * (-softplus(-a) or -c softplus(a)), not as the log of a rounded alpha.
 */
#define LR_FUSE_QK_SILU_L2 0x1u
#define LR_FUSE_BETA_SIGMOID 0x2u
#define LR_FUSE_ALPHA_SIGMOID 0x4u
#define LR_FUSE_ALPHA_SOFTPLUS 0x8u
#define LR_FUSE_O_RMSNORM 0x10u
#define LR_FUSE_ALPHA_SIGMOID_POW 0x20u

typedef struct {
    unsigned flags;            /* OR of LR_FUSE_* (0: the plain call)                */
    const float *alpha_scale;  /* [H] fp32 device, c_h of LR_FUSE_ALPHA_SOFTPLUS and
                                  LR_FUSE_ALPHA_SIGMOID_POW; required with them in
                                  modes using alpha                                 */
    const float *norm_weight;  /* [d_v] fp32 device, shared by all heads, or NULL
                                  for ones (LR_FUSE_O_RMSNORM)                      */
    float norm_eps;            /* >= 0, finite (LR_FUSE_O_RMSNORM)                  */
} lr_fuse;

/*
 * lr_fwd_chunked with the maps of `fuse` (NULL or flags 0: exactly
 * lr_fwd_chunked).  Arguments as for lr_fwd_chunked, except that alpha, beta,
 * q and k hold the pre-activation values of the maps selected, and the
 * workspace must hold lr_fwd_chunked_fused_workspace_size(..., flags) bytes.
 * alpha_scale and norm_weight must be 16-byte aligned and must not overlap o
 * or S_T.
 *
 * bf16: the per-block pass applies the gate maps to the gates it reads, and
 * SiLU to the q and k tiles it stages (fp32 through the hardware tanh
 * approximation: absolute error about 2^-12 |x|, then one rounding to bf16); the
 * rows' L2 norms are kept in fp32 and folded into the factors the products
 * are scaled by, so the result is that of the normalised vectors.  It writes
 * SiLU(q) and SiLU(k) (bf16, [B, H, T, dk] each) to the workspace, where the
 * sequential pass reads them instead of q and k (2 * B * H * T * dk * 2 more
 * bytes of workspace).  fp32: the single kernel applies the maps to what it
 * stages, in fp32.  Rows whose sum of squares overflows fp32 (entries beyond
 * about 1e19) normalise to zero.
 * With LR_FUSE_O_RMSNORM, bf16 in the lr modes, when a head's value channels
 * span at most two CTAs of the sequential pass (d_v <= 64, or d_v = 128 where
 * B * H is large enough for 64-channel CTAs): the pass launches those CTAs
 * as one thread-block cluster; they exchange each token's partial sums of
 * squares through distributed shared memory and store o normalised (fp32
 * sums and scaling, one rounding to bf16).  Otherwise (four CTAs per head,
 * fp32, or LR_MODE_DIAG_DECAY) one more kernel normalises o in place after
 * the chunked kernel.
 */
lr_status lr_fwd_chunked_fused(const void *q, const void *k, const void *v,
                               const float *alpha, const float *beta,
                               const float *S0, void *o, float *S_T,
                               int B, int H, int T, int dk, int dv, int chunk,
                               lr_dtype dt, lr_mode mode, const lr_fuse *fuse,
                               void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* Workspace bytes lr_fwd_chunked_fused needs with these flags (0 for
 * arguments it would reject). */
size_t lr_fwd_chunked_fused_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                           lr_dtype dt, lr_mode mode, unsigned flags);

/*
 * lr_step with the maps of `fuse` (NULL or flags 0: exactly lr_step), all
 * inside the one decode kernel: q and k normalised in registers (fp32, not
 * rounded), the gates mapped, and the d_v outputs of a head normalised
 * together before they are stored.  alpha_scale and norm_weight must be
 * 16-byte aligned and must not overlap o or S.
 */
lr_status lr_step_fused(const void *q, const void *k, const void *v,
                        const float *alpha, const float *beta, float *S, void *o,
                        int N, int H, int dk, int dv, lr_dtype dt, lr_mode mode,
                        const lr_fuse *fuse, cudaStream_t stream);

/*
 * mLSTM memory (page "Le architetture lineari: RetNet, RWKV, xLSTM", xLSTM
 * section, the matrix-memory cell): the scalar-gate row with an exponential
 * write factor and a normaliser,
 *
 *     C_t = f_t C_{t-1} + i_t v_t k_t^T,   n_t = f_t n_{t-1} + i_t k_t,   i_t = exp(igate_t),
 *     h_t = C_t q_t / max(|n_t^T q_t|, 1),
 *
 * computed in the stabilised form the page gives: m_t = max(log f_t +
 * m_{t-1}, igate_t), the memory kept as C~ = e^{-m} C and n~ = e^{-m} n, and
 * h_t = C~_t q_t / max(|n~_t^T q_t|, e^{-m_t}) (the same output).  The state
 * the caller passes in and gets back is that stabilised triple.
 *
 *   q, k   [B, H, T, dk]   dtype dt
 *   v      [B, H, T, dv]   dtype dt
 *   fgate  [B, H, T]       fp32 forget gate f_t in (0, 1]
 *   igate  [B, H, T]       fp32 input-gate pre-activation (any real)
 *   C0, n0, m0             [B, H, dv, dk], [B, H, dk], [B, H] fp32: the initial
 *                          (C~, n~, m), or all three NULL for the empty memory
 *                          (C = 0, n = 0, m = -inf: the first token's m is its igate)
 *   h      [B, H, T, dv]   dtype dt, written; must not overlap any input
 *   C_T, n_T, m_T          the final (C~, n~, m), written; each may be the same
 *                          pointer as its initial counterpart (in place)
 *   workspace              lr_fwd_chunked_mlstm_workspace_size(...) bytes (0 for fp32)
 *
 * Sizes and conventions as for lr_fwd_chunked (dk, dv in {32, 64, 128},
 * chunk == 64, T >= 0).  The bf16 path runs five kernels: the stabiliser at
 * every block start (it depends on the gates only, so one pass over f and
 * igate gives it), the per-block pass (scores weighted by
 * e^{F_t - F_s + igate_s - m_t}, F the cumulative log forget gate of the
 * block), the normaliser n~ at every block start, every token's factor
 * 1 / max(|n~_t^T q_t|, e^{-m_t}), and the sequential pass of lr_fwd_chunked
 * without delta, which scales each token's numerator by its factor in fp32
 * before the one rounding of h.  The fp32 path is one kernel.
 */
lr_status lr_fwd_chunked_mlstm(const void *q, const void *k, const void *v,
                               const float *fgate, const float *igate,
                               const float *C0, const float *n0, const float *m0,
                               void *h, float *C_T, float *n_T, float *m_T,
                               int B, int H, int T, int dk, int dv, int chunk, lr_dtype dt,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes lr_fwd_chunked_mlstm needs (0 for fp32, T == 0, or
 * arguments it would reject). */
size_t lr_fwd_chunked_mlstm_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                           lr_dtype dt);

/*
 * One mLSTM step for N sequences (decode), the state (C, n, m) [N, H, dv, dk],
 * [N, H, dk], [N, H] updated in place: m' = max(log f + m, igate),
 * C <- e^{log f + m - m'} C + e^{igate - m'} v k^T (n likewise with k),
 * h = C q / max(|n^T q|, e^{-m'}).  q, k [N, H, dk]; v, h [N, H, dv] (dtype dt);
 * fgate, igate [N, H] fp32.  An empty memory is C = 0, n = 0, m = -inf.
 */
lr_status lr_step_mlstm(const void *q, const void *k, const void *v, const float *fgate,
                        const float *igate, float *C, float *n, float *m, void *h, int N,
                        int H, int dk, int dv, lr_dtype dt, cudaStream_t stream);

/*
 * Generalised delta rule of RWKV-7 (page "Le architetture lineari: RetNet,
 * RWKV, xLSTM", RWKV section: a per-channel decay plus a rank-one correction
 * with a normalised removal key decoupled from the write key and a
 * per-channel in-context learning rate; eigenvalues anywhere in [-1, 1]).
 * The extracted page lost the equation; this library reads it, in the
 * convention of lr_mode (S is d_v x d_k, transitions multiply from the
 * right), as
 *
 *     S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) + v_t kw_t^T,   o_t = S_t q_t.
 *
 *   q, kw       [B, H, T, dk]   dtype dt (query and write key)
 *   v, o        [B, H, T, dv]   dtype dt
 *   w, kappa, a [B, H, T, dk]   fp32 (decay in (0, 1], removal key, rate)
 *   S0, S_T     [B, H, dv, dk]  fp32 (S0 NULL = zeros; S_T may be S0)
 *
 *   workspace   lr_fwd_chunked_gen_delta_workspace_size(...) bytes (0 for fp32),
 *               16-byte aligned, owned by the caller, not overlapping any argument
 *
 * Sizes and conventions as for lr_fwd_chunked (dk, dv in {32, 64, 128},
 * chunk == 64, T >= 0).  Both paths work in 32-token blocks with the
 * pseudo-values u_t = S_{t-1} kappa_t of a unit-lower-triangular system per
 * block, every decay factor e^{L_t - L_s} (t >= s, L the cumulative log decay)
 * at most 1.  The bf16 path runs two kernels: a per-block pass over all blocks
 * in parallel (the four decayed score matrices, the triangular solve, the
 * coupling to the previous block), stored in the workspace, then the
 * sequential pass of lr_fwd_chunked with values stacked on pseudo-values, on
 * the tensor cores.  Its score matrices split each decay at the last token of
 * the key's 16-token half: exact while the decay over any 16 consecutive
 * tokens stays above e^-80 (w >= 0.007 per token always satisfies it).  The
 * fp32 path is one kernel on the CUDA cores with every decay factor taken
 * directly.
 */
lr_status lr_fwd_chunked_gen_delta(const void *q, const void *kw, const void *v,
                                   const float *w, const float *kappa, const float *a,
                                   const float *S0, void *o, float *S_T,
                                   int B, int H, int T, int dk, int dv, int chunk, lr_dtype dt,
                                   void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes lr_fwd_chunked_gen_delta needs (0 for fp32, T == 0, or
 * arguments it would reject). */
size_t lr_fwd_chunked_gen_delta_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                               lr_dtype dt);

/* One step of the same rule for N sequences (decode): per value row r with
 * s = S[r, :], u = s . kappa, S[r, :] <- s * w - u (a * kappa) + v_r kw,
 * o_r = S[r, :] . q.  q, kw, w, kappa, a [N, H, dk] (q, kw in dtype dt, the
 * rest fp32); v, o [N, H, dv]; S [N, H, dv, dk] fp32 updated in place. */
lr_status lr_step_gen_delta(const void *q, const void *kw, const void *v, const float *w,
                            const float *kappa, const float *a, float *S, void *o, int N, int H,
                            int dk, int dv, lr_dtype dt, cudaStream_t stream);

/* Static English text for a status code (never NULL). */
const char *lr_status_string(lr_status s);

/* ABI version of this header: 3 (2 added the fused entry points, the
 * diagonal gate, the mLSTM entry points and LR_ERR_FUSE; 3 gave
 * lr_fwd_chunked_gen_delta a workspace and added its size query; every entry
 * point of 1 is unchanged). */
int lr_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LR_H_ */
