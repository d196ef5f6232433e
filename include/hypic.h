/*
 * hypic.h -- C ABI of the GB300 segment-scan and state-composition library
 * for position-independent caching (HYPIC) of hybrid linear-attention models.
 *
 * What the operations are (web pages about HYPIC):
 *   xix.ai/fr, "Xiaohongshu, l'Université de Pékin et l'Université Jiao Tong de
 *   Shanghai dévoilent HYPIC ...", paragraph on linear layers ("opérateurs de
 *   transition"): each segment C is prefilled once from a zero state; the cache
 *   keeps the pair (T_C, S(C|0)), T_C being the product of every per-token
 *   transition matrix of the segment; at reuse the running state is
 *   left-multiplied by T_C and S(C|0) is added:  S(C1.C2) = T(C2) S(C1) + S(C2).
 *   remio.ai/ja, "HYPIC ...", section "how HYPIC composes states": the
 *   composition costs the same whatever the segment length; section "cold
 *   requests become parallel": a combine step folds the pairs of many segments
 *   into the request's running state.
 *
 * The pages print no per-token rule.  This library reads the families named
 * there as (state S in R^{dk x dv}, fp32):
 *   S_t = T_t S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t  (state after token t)
 *     HYPIC_SCALAR : T_t = alpha_t I                       (RetNet, Mamba2)
 *     HYPIC_DIAG   : T_t = diag(alpha_t), alpha_t in R^dk  (GLA; gates the key axis)
 *     HYPIC_DENSE  : T_t = alpha_t (I - beta_t k_t k_t^T)  (gated delta rule)
 *     HYPIC_KDA    : T_t = diag(alpha_t) (I - beta_t k_t k_t^T), alpha_t in R^dk
 *                    (KDA-style: the gated delta rule with a gate per channel)
 *   T_C = T_L ... T_1,  S(C|0) = S_L from S_0 = 0.
 * T_C is stored in log-scaled form T_C = exp(lambda) * M, because the plain
 * product underflows fp32 (and fp64) at the segment lengths of long prompts:
 *   scalar: lambda [.., H] = sum_t log alpha_t;              M is 1 (not stored)
 *   diag  : lambda [.., H, dk] = sum_t log alpha_{t,i};      M is I (not stored)
 *   dense : lambda [.., H], M [.., H, dk, dk] with max|M| in [1, 2)
 *           (M == 0 exactly only for a product that is exactly zero).
 *   kda   : as dense, with the per-channel gates inside M (lambda holds only
 *           the power-of-two rescaling).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no memory and keeps no state between calls.  Every call is
 *     asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy default
 *     stream) and safe to issue from several host threads.
 *   - Layouts are dense row-major, innermost index last.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns a negative hypic_status and launches nothing.  A launch failure
 *     returns HYPIC_ECUDA.  Device-side problems (pool index out of range,
 *     segment offsets not ascending within [0, total_tokens]) never trap: the
 *     offending index is clamped or the segment treated as empty, and
 *     HYPIC_EINDEX is written to `d_err` when `d_err` is non-NULL (a device
 *     int the caller zeroes and reads after synchronising).
 *   - Supported head sizes: dk, dv in {32, 64, 128}.
 *   - Every gate alpha must be finite and > 0.
 */
#ifndef HYPIC_H
#define HYPIC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HYPIC_OK = 0,
    HYPIC_EINVAL = -1,       /* bad count, null required pointer, inconsistent options */
    HYPIC_EUNSUPPORTED = -2, /* head size or family/dtype combination not built */
    HYPIC_EALIGN = -3,       /* a pointer is not aligned as documented */
    HYPIC_ECUDA = -4,        /* a CUDA runtime call or kernel launch failed */
    HYPIC_EINDEX = -5,       /* device side: index out of range (written to d_err) */
    HYPIC_ETIMEOUT = -6      /* device side: a pipeline wait gave up after ~2 s (written to d_err);
                                the kernel left its outputs incomplete and released its resources */
} hypic_status;

typedef enum { HYPIC_SCALAR = 0, HYPIC_DIAG = 1, HYPIC_DENSE = 2, HYPIC_KDA = 3 } hypic_family;

typedef enum { HYPIC_BF16 = 0, HYPIC_F32 = 1 } hypic_dtype;

/*
 * hypic_segment_scan -- per segment C and head: (T_C, S(C|0)) and optionally
 * the per-token outputs o_t.  (xix.ai/fr, linear-layer paragraph: the pair is
 * built at the segment's first prefill from a zero state and depends only on
 * the segment's own tokens.)
 *
 * Segments are packed along the token axis and shared by all layers:
 * segment s of every layer covers tokens [seg_offsets[s], seg_offsets[s+1]).
 *   fam, in_dtype      family; element type of q, k, v and o_out
 *   n_layers, n_seg, total_tokens (N), n_heads (H), d_k, d_v   sizes
 *   seg_offsets        int64 [n_seg + 1], ascending, 0 .. N        (device)
 *   q                  [n_layers, N, H, d_k]; required iff o_out != NULL
 *   k                  [n_layers, N, H, d_k]
 *   v                  [n_layers, N, H, d_v]
 *   alpha   fp32       [n_layers, N, H] (scalar, dense) or [n_layers, N, H, d_k] (diag, kda)
 *   beta    fp32       [n_layers, N, H] or NULL (=> 1 for every token)
 *   lam_out fp32       [n_layers, n_seg, H] or [n_layers, n_seg, H, d_k] (diag)
 *   M_out   fp32       [n_layers, n_seg, H, d_k, d_k]; dense, kda: required; else NULL
 *   S_out   fp32       [n_layers, n_seg, H, d_k, d_v]
 *   o_out   in_dtype   [n_layers, N, H, d_v] or NULL; o_t = S_t^T q_t
 *   d_err              device int or NULL (see conventions)
 * An empty segment yields lambda = 0, M = I, S = 0.
 * Alignment: q, k, v, o_out, S_out, M_out, the diag / kda alpha and the diag
 * lambda must be 16-byte aligned; other pointers 4-byte (seg_offsets 8-byte).
 * Kernels: with bf16 inputs and d_k = d_v = 128 every family runs on the tensor
 * cores (scalar and diagonal with or without o_t, the gated delta rule with or
 * without o_t); without a workspace the KDA family runs on the token-by-token
 * fp32 kernel (CUDA cores), as do fp32 inputs, head sizes 32 / 64 and KDA with
 * o_t; hypic_segment_scan_ws takes KDA without o_t to the tensor cores.
 */
int hypic_segment_scan(int fam, int in_dtype, int n_layers, int n_seg,
                       int64_t total_tokens, int n_heads, int d_k, int d_v,
                       const int64_t *seg_offsets, const void *q, const void *k,
                       const void *v, const float *alpha, const float *beta,
                       float *lam_out, float *M_out, float *S_out, void *o_out,
                       int *d_err, void *cuda_stream);

/*
 * hypic_segment_scan_workspace_bytes -- bytes of device scratch that
 * hypic_segment_scan_ws needs for these sizes, or 0 when that call uses none
 * (then its workspace may be NULL).  A negative hypic_status on bad counts.
 * Today the scratch is used with bf16 inputs and d_k = d_v = 128 by
 *   the dense family: one record per (layer, head, 64-token chunk slot) of
 *     49424 bytes (50192 bytes with o_t), n_layers * n_heads * (n_seg +
 *     total_tokens / 64) records, then n_seg int32 (the segments ranked by
 *     length: the longest chains are started first), each part rounded up to
 *     256 bytes;
 *   the diagonal family without o_t and with n_seg <= 512: 2 x 512 partial
 *     states of 66048 bytes (67.6 MB), for a schedule that spreads all
 *     segments' chunks evenly over the GPU and then folds the pieces of
 *     segments split between CTAs with the composition rule;
 *   the KDA family without o_t: per (layer, 64-token chunk slot, head) the
 *     chunk's pair (M_c, S_c: 2 x 65536 bytes, lambda_c: 4 bytes), n_layers *
 *     (n_seg + total_tokens / 64) * n_heads of them, then as many int32 plus one
 *     (the list of chunks formed token by token, with its count), n_seg +
 *     total_tokens / 64 + 1 int64 chunk starts and 2 x n_layers * n_seg int32
 *     (each segment's first pair and count), each part rounded up to 256 bytes;
 *     above 64 GiB the token-by-token kernel is used and this is 0.
 */
int64_t hypic_segment_scan_workspace_bytes(int fam, int in_dtype, int n_layers, int n_seg,
                                           int64_t total_tokens, int n_heads, int d_k, int d_v,
                                           int with_o);

/*
 * hypic_segment_scan_ws -- hypic_segment_scan with caller-owned device
 * scratch; same arguments, layouts, results and error behaviour, plus
 *   workspace        device memory, 256-byte aligned, at least
 *                    hypic_segment_scan_workspace_bytes(...) bytes (NULL allowed
 *                    when that is 0).  Its contents on entry do not matter; the
 *                    call overwrites them, and two calls in flight at once
 *                    must not share it.
 *   workspace_bytes  its size; too small returns HYPIC_EINVAL.
 * With the scratch the dense scan runs in two passes: every 64-token chunk's
 * intra-chunk solve (Gram matrix, L, (I + L)^-1, decays) in parallel over all
 * chunks, then the ordered state pass (the chunked WY/UT form of the gated
 * delta rule; the pages give no chunked algorithm); the diagonal scan balances
 * its work over the GPU (results equal to hypic_segment_scan's up to rounding;
 * they depend on the batch's total work, not on a segment's position); the KDA
 * scan forms every 64-token chunk's pair (T_c, S(c|0)) on the tensor cores in
 * parallel (a chunk in which a channel decays by more than e^60 token by token)
 * and composes each segment's chunk pairs in order, T(C1.C2) = T(C2) T(C1)
 * (xix.ai/fr, paragraph on linear layers).  Other cases run exactly as
 * hypic_segment_scan.
 */
int hypic_segment_scan_ws(int fam, int in_dtype, int n_layers, int n_seg,
                          int64_t total_tokens, int n_heads, int d_k, int d_v,
                          const int64_t *seg_offsets, const void *q, const void *k,
                          const void *v, const float *alpha, const float *beta,
                          float *lam_out, float *M_out, float *S_out, void *o_out,
                          void *workspace, int64_t workspace_bytes, int *d_err,
                          void *cuda_stream);

/*
 * hypic_segment_scan_static -- the two-pass dense scan of hypic_segment_scan_ws
 * with its scratch taken from a fixed 64 MiB device array inside the library
 * instead of a caller workspace; the call allocates nothing.  The HYPIC pages
 * have no counterpart of this entry point.  It is meant for callers that cannot
 * allocate device memory at call time (an engine that gave all free memory to
 * its KV-cache pool at start-up; a host path that must not enter the allocator,
 * which can synchronise the device).
 *   Arguments as hypic_segment_scan without q / o_out.  Only fam = HYPIC_DENSE,
 *   in_dtype = HYPIC_BF16, d_k = d_v = 128 is served; another family, input type
 *   or head size, or a problem whose records need more than the 64 MiB
 *   (hypic_segment_scan_workspace_bytes gives the need; 64 MiB hold 1357 records
 *   of 49424 bytes), returns HYPIC_EUNSUPPORTED and launches nothing.  A batch
 *   whose segments are all empty (total_tokens = 0) needs no scratch and gets
 *   lambda = 0, M = I, S = 0 as from hypic_segment_scan.
 *   The scratch's contents never need to start at zero.  It is one array per
 *   device for the whole process: two calls in flight at the same time (other
 *   streams or host threads) race on it, so callers serialise them.
 *   The first call in each CUDA context (per device: its primary context, or
 *   a context the caller made current) looks up the array's address
 *   (cudaGetSymbolAddress, with that device current) and caches it under the
 *   context's id, so a context created later (after cudaDeviceReset, say) gets
 *   a fresh lookup; a caller that will later capture its stream makes one call
 *   in that context before capturing.
 */
int hypic_segment_scan_static(int fam, int in_dtype, int n_layers, int n_seg,
                              int64_t total_tokens, int n_heads, int d_k, int d_v,
                              const int64_t *seg_offsets, const void *k, const void *v,
                              const float *alpha, const float *beta, float *lam_out,
                              float *M_out, float *S_out, int *d_err, void *cuda_stream);

/*
 * hypic_compose -- S = T_C S_prev + S_C for n items x H heads, with
 * T_C = exp(lambda) M.  (xix.ai/fr, linear-layer paragraph:
 * S(C1.C2) = T(C2) S(C1) + S(C2); left-multiplication by the cached T then an
 * addition.)  Optionally also the operator of the concatenation,
 * T(C1.C2) = T(C2) T(C1), which makes compositions chainable in any grouping.
 *   lam     fp32  [n, H] (scalar, dense) or [n, H, d_k] (diag)   -- T(C2)
 *   M       fp32  [n, H, d_k, d_k] (dense, kda; must be NULL otherwise)
 *   S_prev  fp32  [n, H, d_k, d_v] or NULL (=> 0)                 -- S(C1)
 *   S_C     fp32  [n, H, d_k, d_v]                                -- S(C2)
 *   S_out   fp32  [n, H, d_k, d_v]; may be the same pointer as S_prev
 *                 (scalar, diag and dense); must not overlap S_C otherwise
 *   lam_prev, lam_out  like lam; both NULL or both given          -- T(C1), T(C1.C2)
 *                      lam_out must not overlap lam, lam_prev, S_out or M_out
 *                      (HYPIC_EINVAL): no in-place operator accumulation
 *   M_prev, M_out      like M (dense, kda; given iff lam_out is)
 * Dense M_out has max|M_out| in [1, 2) (exact power-of-two scaling into lam_out).
 * All pointers 16-byte aligned except scalar/dense lambdas (4-byte).
 */
int hypic_compose(int fam, int n, int n_heads, int d_k, int d_v, const float *lam,
                  const float *M, const float *S_prev, const float *S_C, float *S_out,
                  const float *lam_prev, const float *M_prev, float *lam_out,
                  float *M_out, void *cuda_stream);

/*
 * hypic_compose_chain -- the combine step: for every request r, layer l and
 * head h, starting from S_init (or 0), fold the cached pairs of the pool
 * entries seg_idx[r, 0 .. chain_len[r]-1] in that order:
 *   S <- T_p S + S_p
 * and write the final state once.  (xix.ai/fr: reuse under any prefix;
 * remio.ai/ja, "cold requests become parallel": the combine worker folds each
 * segment's transition and state into the running state.)
 *   chain_len  int32 [n_req]            0 <= chain_len[r] <= max_chain
 *   seg_idx    int32 [n_req, max_chain] pool indices in prompt order
 *   pool_lam   fp32  [pool_size, n_layers, H] or [pool_size, n_layers, H, d_k] (diag)
 *   pool_M     fp32  [pool_size, n_layers, H, d_k, d_k] (dense, kda; NULL otherwise)
 *   pool_S     fp32  [pool_size, n_layers, H, d_k, d_v]
 *   S_init     fp32  [n_req, n_layers, H, d_k, d_v] or NULL (=> 0)
 *   S_out      fp32  [n_req, n_layers, H, d_k, d_v]; may be S_init itself;
 *              must overlap neither the pool nor (another part of) S_init:
 *              HYPIC_EINVAL otherwise
 *   d_err      device int or NULL: an index outside [0, pool_size) or a
 *              chain length outside [0, max_chain] is clamped and reported.
 */
int hypic_compose_chain(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v,
                        int max_chain, const int32_t *chain_len, const int32_t *seg_idx,
                        int pool_size, const float *pool_lam, const float *pool_M,
                        const float *pool_S, const float *S_init, float *S_out,
                        int *d_err, void *cuda_stream);

/*
 * hypic_compose_chain_ws -- hypic_compose_chain with caller-owned device scratch,
 * used when few (request, layer, head) units carry long chains (fewer units than
 * twice the SM count, chains of 8 or more entries): a chain then runs on few SMs
 * one entry after another.  Because T(C1.C2) = T(C2) T(C1) (xix.ai/fr,
 * linear-layer paragraph), consecutive entries can be folded into one cached pair
 * first: the call folds groups of consecutive entries of every chain in parallel
 * (composed prefixes, as hypic_compose_prefix), then each chain's group pairs in
 * order into S_init -- a two-level tree.  Results equal hypic_compose_chain's up
 * to rounding (the fp32 additions are regrouped).  Other shapes run exactly as
 * hypic_compose_chain and need no scratch.
 *   Arguments as hypic_compose_chain, plus
 *   workspace        device scratch, 256-byte aligned, at least
 *                    hypic_compose_chain_workspace_bytes(...) bytes (may be NULL when
 *                    that is 0); it may overlap no other argument.  Caller-owned;
 *                    its contents need not be initialised and are garbage after.
 *   workspace_bytes  its size; too small -> HYPIC_EINVAL before any launch.
 */
int64_t hypic_compose_chain_workspace_bytes(int fam, int n_req, int n_layers, int n_heads,
                                            int d_k, int d_v, int max_chain);
int hypic_compose_chain_ws(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v,
                           int max_chain, const int32_t *chain_len, const int32_t *seg_idx,
                           int pool_size, const float *pool_lam, const float *pool_M,
                           const float *pool_S, const float *S_init, float *S_out,
                           void *workspace, int64_t workspace_bytes, int *d_err,
                           void *cuda_stream);

/*
 * hypic_compose_prefix -- a composed prefix: for every request r, layer l and
 * head h, the cached pair of the concatenation of the pool entries
 * seg_idx[r, 0 .. chain_len[r]-1] (in that order):
 *   T = T_{p_n} ... T_{p_1},   S = S(C_{p_1} ... C_{p_n} | 0).
 * (xix.ai/fr, linear-layer paragraph: T(C1.C2) = T(C2) T(C1) makes the
 * composition chainable in any grouping, so a popular ordered group of cached
 * segments can itself be cached as one pair and used as a pool entry.)
 *   Arguments as hypic_compose_chain without S_init, plus
 *   lam_out  fp32  [n_req, n_layers, H] or [n_req, n_layers, H, d_k] (diag)
 *   M_out    fp32  [n_req, n_layers, H, d_k, d_k] (dense, kda; NULL otherwise),
 *            max|M_out| in [1, 2) (exact power-of-two scaling into lam_out)
 *   S_out    fp32  [n_req, n_layers, H, d_k, d_v]
 * The outputs must not overlap one another or the pool.  An empty group gives
 * lambda = 0, M = I, S = 0.  Dense and KDA run the operator chain M_pn ... M_p1 on
 * the same kernels as the state's chain (then a pass that folds the power of two).
 */
int hypic_compose_prefix(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v,
                         int max_chain, const int32_t *chain_len, const int32_t *seg_idx,
                         int pool_size, const float *pool_lam, const float *pool_M,
                         const float *pool_S, float *lam_out, float *M_out, float *S_out,
                         int *d_err, void *cuda_stream);

/*
 * hypic_seam_compose -- reuse of a cached segment whose first w tokens (the
 * seam window) were left out of its cache.  (xix.ai/fr, paragraph on
 * full-attention layers: at reuse the seam tokens are recomputed under the full
 * prefix; the linear layers advance the running state through them and hand
 * each seam token's output to the layer above.  The rest of the segment then
 * enters by its cached pair, as in hypic_compose.)  For n items x H heads:
 *   S = S_prev;  for t = 0 .. w-1:  S = T_t S + beta_t k_t v_t^T,  o_t = S^T q_t;
 *   S_out = T_body S + S_body,  T_body = exp(lambda) M.
 *   in_dtype  HYPIC_BF16 or HYPIC_F32: q, k, v and o_out
 *   q, k    [n, w, H, d_k];  v [n, w, H, d_v]      -- the seam tokens (q may be
 *                                                   NULL when o_out is NULL)
 *   alpha   fp32 [n, w, H] (scalar, dense) or [n, w, H, d_k] (diag, kda)
 *   beta    fp32 [n, w, H] or NULL (=> 1)
 *   lam     fp32 [n, H] or [n, H, d_k] (diag)     -- T_body of the cached rest
 *   M       fp32 [n, H, d_k, d_k] (dense, kda; NULL otherwise)
 *   S_prev  fp32 [n, H, d_k, d_v] or NULL (=> 0)   -- state before the segment
 *   S_C     fp32 [n, H, d_k, d_v]                  -- S_body of the cached rest
 *   S_out   fp32 [n, H, d_k, d_v]; may be the same pointer as S_prev, must not
 *           overlap any other argument
 *   o_out   [n, w, H, d_v] or NULL
 * 0 <= w <= 4096; w = 0 is hypic_compose.  The window runs on CUDA cores in
 * fp32; the dense family writes the advanced state to S_out and then composes
 * it in place (so S_out holds the intermediate state between two launches on
 * the stream).  Pointers 16-byte aligned (alpha, beta, scalar/dense lam:
 * 4-byte; bf16 q, k, v, o_out: 2-byte with rows of 16-byte multiples).
 */
int hypic_seam_compose(int fam, int in_dtype, int n, int w, int n_heads, int d_k, int d_v,
                       const void *q, const void *k, const void *v, const float *alpha,
                       const float *beta, const float *lam, const float *M, const float *S_prev,
                       const float *S_C, float *S_out, void *o_out, void *cuda_stream);

/* Human-readable name of a hypic_status value (static string, never NULL). */
const char *hypic_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int hypic_version(void);

/* Diagnostic: the bounded pipeline wait that every kernel above uses, on its own.
 * One thread waits on a fresh shared-memory mbarrier for at most limit_cycles SM
 * cycles (0 <= limit_cycles <= 4e9, the kernels' own limit).  With arrive != 0 it
 * arrives on the barrier first and the wait completes at once; with arrive == 0
 * nothing arrives, the wait gives up after the limit and HYPIC_ETIMEOUT is written
 * to *d_err -- the status a pipeline kernel leaves when one of its waits runs out.
 *   d_err     device int32, nullable, 4-byte aligned
 *   d_cycles  device int64, nullable, 8-byte aligned: the cycles the wait took
 * Nothing faults or traps and the context stays usable.  Returns HYPIC_EINVAL for
 * a limit out of range, HYPIC_EALIGN for a misaligned pointer, HYPIC_ECUDA when
 * the launch fails; asynchronous on the stream like the other entry points. */
int hypic_selftest_wait(long long limit_cycles, int arrive, int *d_err, long long *d_cycles,
                        void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* HYPIC_H */
