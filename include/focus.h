/*
 * focus.h - C ABI of the Focus centroid-gated sparse attention forward pass
 *           (libfocus.so, sm_103a).
 *
 * The method: "Why Attend to Everything? Focus is the Key" (Yao, Chen et al.).
 *   - gist.science technical summary, section 2 "Core Architecture": K learnable
 *     centroids C in R^{K x d_g}; tokens are projected into centroid space and
 *     grouped; a local window of w tokens attends with exact softmax; distant
 *     tokens attend only within a shared group.
 *   - same section, "Inference Efficiency (Top-k)": at inference each token joins
 *     its top-k highest-scoring groups and distant tokens interact only when they
 *     share at least one group.
 *   - same summary, "Key Technical Innovation: Sinkhorn Normalization": Sinkhorn
 *     balancing of the token-to-group assignment.
 *   - jindou-blog deep read, method bullets: routing dimension d_g = 16, scoring by
 *     dot product, exact softmax inside the window and inside each group.
 *
 * What is computed, per batch b and query head h (readings where the pages are
 * silent: logits scale * q.k with scale 1/sqrt(d) by default; window pairs are
 * j <= i with i - j < w; long-range pairs are j <= i - w whose group bitmasks
 * intersect; ONE softmax runs over the union, each key counted once):
 *
 *   A_i   = { j <= i : i - j < w } U { j <= i - w : mask_i & mask_j != 0 }
 *   LSE_i = log sum_{j in A_i} exp(scale q_i.k_j)          (natural log)
 *   O_i   = sum_{j in A_i} exp(scale q_i.k_j - LSE_i) v_j
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device, caller
 *     owned, contiguous, row-major in the stated layout, 16-byte aligned (the
 *     workspace 256-byte aligned). bf16 tensors are passed as uint16_t bit patterns.
 *   - The library allocates no device memory and keeps no state between calls;
 *     scratch lives in the caller's workspace (focus_workspace_size bytes).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t, NULL = legacy
 *     default stream). Nothing is synchronised except by focus_get_status.
 *   - Return value: FOCUS_OK (0) or a negative FOCUS_ERR_* code. Argument errors
 *     are detected on the host before anything is launched. Nothing is thrown
 *     across the ABI.
 *
 * Index conventions: B batch, N tokens, H query heads, H_kv key/value heads
 * (H % H_kv == 0), R routing heads (R divides H_kv; R = 1 is one routing vector
 * per token per layer, R = H_kv one per KV-head group), K groups (centroids),
 * top_k groups per token, w window. Query head h reads KV head
 * kvh = h / (H / H_kv) and routing head rho = kvh / (H_kv / R).
 */
#ifndef FOCUS_H_
#define FOCUS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FOCUS_D_G 16            /* routing dimension */
#define FOCUS_MAX_K 32          /* groups representable in a uint32 bitmask */
#define FOCUS_MAX_SEGMENTS 1024 /* C(K, top_k) limit of the mask-value bucketing */

/* Long-range schedule (focus_params.schedule).
 *   SEGMENTS: tokens sorted by their exact group set (C(K, top_k) segments); a
 *             query segment attends to every segment its set intersects, so each
 *             key is met once.  Needs C(K, top_k) <= FOCUS_MAX_SEGMENTS.
 *   GROUPS:   one position-ordered list per group (each token in top_k lists); a
 *             query in list g counts key j only when g is the LOWEST group the two
 *             share, so each key is still counted once; the top_k partial results
 *             of a token are merged with the window's by log-sum-exp.  Any K, top_k.
 *   AUTO:     the one with the smaller estimated tensor-core work (fractions of
 *             dense causal attention): SEGMENTS ~ (1 - C(K-k,k)/C(K,k)) *
 *             (1 + 2 C(K,k) 256 / N), the chance that two sets meet times the
 *             raggedness of C(K,k) segments over N tokens; GROUPS ~ 1.15 k^2 / K.
 *             SEGMENTS when top_k = 1 (the same partition), GROUPS when
 *             C(K, top_k) > FOCUS_MAX_SEGMENTS.  focus_bucket_shape reports it. */
enum focus_schedule {
  FOCUS_SCHEDULE_AUTO = 0,
  FOCUS_SCHEDULE_SEGMENTS = 1,
  FOCUS_SCHEDULE_GROUPS = 2
};

enum focus_status {
  FOCUS_OK = 0,
  FOCUS_ERR_INVALID_ARG = -1, /* null pointer, bad size or inconsistent shape */
  FOCUS_ERR_UNSUPPORTED = -2, /* valid but not implemented (d_head; C(K,top_k) with SEGMENTS) */
  FOCUS_ERR_WORKSPACE = -3,   /* ws_bytes < focus_workspace_size() */
  FOCUS_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
  FOCUS_ERR_TIMEOUT = -5,     /* a bounded device-side wait ran out */
  FOCUS_ERR_BOUNDS = -6,      /* device-side index check failed (bad mask_in) */
  FOCUS_ERR_ALIGNMENT = -7,   /* a pointer is not suitably aligned */
  FOCUS_ERR_NONFINITE = -8    /* a routing score was NaN or infinite (non-finite r or C) */
};

typedef struct focus_params {
  int32_t B, N, H, H_kv, d_head; /* d_head in {64, 128} */
  int32_t R;                     /* routing heads, divides H_kv */
  int32_t K, top_k;              /* 1 <= top_k <= K <= 32 */
  int32_t w;                     /* window, >= 1 */
  int32_t sinkhorn_iters;        /* 0 = plain top-k on the scores */
  float sinkhorn_eps;            /* score temperature for Sinkhorn, > 0 (1.0 typical) */
  float softmax_scale;           /* <= 0 selects 1 / sqrt(d_head) */
  int32_t schedule;              /* enum focus_schedule; 0 = AUTO */
} focus_params;

/* Bytes of device workspace needed by focus_route, focus_bucket and
 * focus_attn_fwd for these parameters; 0 if the parameters are invalid. */
size_t focus_workspace_size(const focus_params* p);

/*
 * Group membership: scoring, optional Sinkhorn balancing, hard top-k.
 *   r          [B, N, R, 16] fp32  routing vectors
 *   C          [K, 16] fp32        centroids
 *   mask_out   [B, R, N] uint32    bit g set iff group g is among the token's
 *                                  top_k; ties go to the lower group index
 *   margin_out [B, R, N] fp32 or NULL: kappa_(top_k) - kappa_(top_k+1)
 *                                  (+inf when top_k == K)
 * Score s_ig = r_i . c_g as a fused multiply-add chain over t = 0..15 in fp32.
 * With sinkhorn_iters = T > 0 the log-domain iteration runs T times over all N
 * tokens of each (b, routing head): column step beta_g = log(N/K) -
 * LSE_i(s_ig/eps + alpha_i), then row step alpha_i = -LSE_g(s_ig/eps + beta_g);
 * the ranking key is kappa_ig = s_ig/eps + beta_g. With T = 0, kappa = s.
 * A ranking key that is not finite (NaN or +-inf, e.g. from NaN in r or C) sets
 * FOCUS_ERR_NONFINITE in the workspace's status word (read it with
 * focus_get_status); a NaN key ranks below every number, so such a token still
 * gets exactly top_k groups (the lowest-indexed ones when all its keys are NaN)
 * and nothing reads out of bounds. Its margin is then unspecified.
 */
int focus_route(const focus_params* p, const float* r, const float* C, uint32_t* mask_out,
                float* margin_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Shape of the bucketing for these parameters: the schedule that runs
 * (FOCUS_SCHEDULE_SEGMENTS or FOCUS_SCHEDULE_GROUPS, AUTO resolved), the number
 * of segments (C(K, top_k) or K) and the rows per (b, routing head) (N or
 * N * top_k).  Either output pointer may be NULL.  Returns the schedule, or a
 * negative FOCUS_ERR_* code for invalid parameters.
 */
int focus_bucket_shape(const focus_params* p, int32_t* n_segments, int32_t* rows);

/*
 * Bucketing of tokens by group bitmask (exposed for inspection and tests).
 *   mask        [B, R, N] uint32, exactly top_k of the low K bits set per token
 *   perm_out    [B, R, rows] int32 (rows from focus_bucket_shape):
 *               SEGMENTS: token positions stably sorted by the colex rank of
 *               their mask's k-subset (positions ascend inside a segment);
 *               GROUPS: the K group lists one after another, each the ascending
 *               positions of the tokens whose mask has that bit
 *   seg_off_out [B, R, n_segments + 1] int32: segment start offsets into perm_out
 * Either output may be NULL (the result then stays in the workspace only).
 * A mask with the wrong number of bits sets FOCUS_ERR_BOUNDS in the status word
 * (GROUPS then files such a token under groups 0..top_k-1).
 */
int focus_bucket(const focus_params* p, const uint32_t* mask, int32_t* perm_out,
                 int32_t* seg_off_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Forward pass of Focus attention over the union set A_i defined above.
 *   q        [B, N, H, d_head] bf16
 *   k, v     [B, N, H_kv, d_head] bf16
 *   r, C     routing inputs as in focus_route (may be NULL when mask_in is given)
 *   mask_in  [B, R, N] uint32 or NULL: precomputed membership; NULL routes
 *            internally (focus_route's result, kept in the workspace)
 *   o        [B, N, H, d_head] bf16 out
 *   lse      [B, H, N] fp32 out (natural log of the scaled logits), may be NULL
 * Steps on `stream`: route (if mask_in is NULL), bucket, permuted copies of
 * Q/K/V, window attention, long-range attention over compatible segments with
 * the union merge (SEGMENTS), or over the group lists followed by a merge of the
 * window part with each token's top_k list parts (GROUPS).
 */
int focus_attn_fwd(const focus_params* p, const uint16_t* q, const uint16_t* k,
                   const uint16_t* v, const float* r, const float* C, const uint32_t* mask_in,
                   uint16_t* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * focus_attn_fwd with stage timing: identical work and results, plus CUDA events
 * recorded on `stream` at the stage boundaries, so a caller can time each stage
 * without adding any synchronisation.
 *   stage_events  array of FOCUS_N_STAGE_EVENTS cudaEvent_t handles (cast to
 *                 void*) created by the caller, or NULL (then this is exactly
 *                 focus_attn_fwd). Recorded in order: [0] start, [1] after routing,
 *                 [2] after bucketing, the long-range schedule and its plans, [3]
 *                 after the permuted Q/K/V copies, [4] after window attention, [5]
 *                 after long-range attention and the union merge.
 */
#define FOCUS_N_STAGE_EVENTS 6
int focus_attn_fwd_ev(const focus_params* p, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const float* r, const float* C,
                      const uint32_t* mask_in, uint16_t* o, float* lse, void* ws,
                      size_t ws_bytes, void* stream, void* const* stage_events);

/*
 * focus_route without a workspace argument, for callers that cannot allocate
 * device memory on their call path: for example a custom op or plugin inside an
 * inference engine that hands all device memory to its own pool at start-up and
 * forbids cudaMalloc afterwards (cudaMalloc can also synchronise the device,
 * which such hosts must not do mid-stream). The paper has no counterpart; this is
 * a deployment variant of focus_route with identical results.
 *   Arguments and outputs as in focus_route (r, C, mask_out, optional margin_out,
 *   stream); the caller still owns every input and output buffer. Parameter
 *   errors give the same codes as focus_route.
 *   Scratch: only the Sinkhorn step needs any. It lives in a file-scope device
 *   array of focus_route_static_limit() bytes (4 MiB) inside the library, held by
 *   every GPU that loads the library until the process exits. A Sinkhorn problem
 *   needing more (256 * ceil(B*R*K*4 / 256) + B*R*ceil(N/256)*K*8 bytes) returns
 *   FOCUS_ERR_WORKSPACE before anything else is checked or launched; without
 *   Sinkhorn (sinkhorn_iters = 0) there is no size limit and the array is unused.
 *   The array's device address is looked up (cudaGetSymbolAddress) by the first
 *   Sinkhorn call on each device, and again by the first call under a new CUDA
 *   context of that device (e.g. after cudaDeviceReset); make that first call
 *   before any stream capture.
 *   All calls share the one array and nothing in it needs clearing between calls
 *   (every value is written before it is read), but Sinkhorn calls that overlap on
 *   the GPU (concurrent streams, several host threads) race on it: serialise them.
 *   Non-finite routing scores are handled as in focus_route, but there is no
 *   status word to report them.
 *   No device memory is allocated or freed by this call.
 */
int focus_route_static(const focus_params* p, const float* r, const float* C,
                       uint32_t* mask_out, float* margin_out, void* stream);

/* Size in bytes of focus_route_static's device scratch array (host only). */
size_t focus_route_static_limit(void);

/*
 * Forward pass on HOST buffers, with host-device copies overlapped with compute.
 * The heads are split into groups of consecutive KV heads (with their query heads
 * and, when R > 1, their routing heads: a group holds whole routing heads); group
 * g+1's inputs are copied in while group g computes, and group g's outputs are
 * copied out meanwhile.
 * Each group is an independent problem (attention never mixes heads), so the
 * result equals focus_attn_fwd on the whole problem.
 *   q_h, k_h, v_h, r_h, C_h  host inputs, layouts as in focus_attn_fwd (r and C
 *                            are required: routing runs inside, per group)
 *   o_h [B, N, H, d] bf16, lse_h [B, H, N] fp32 or NULL: host outputs
 *   n_groups   > 0: that many equal groups (it must divide H_kv and, when R > 1,
 *              R); 0 = automatic: the first group's inputs and the last group's
 *              outputs cannot overlap any compute, so those two groups are small
 *              (about an eighth of the KV heads each) and the others about a
 *              quarter each (focus_host_groups lists the sizes)
 *   ws         device workspace of focus_host_workspace_size(p, n_groups) bytes
 *   compute_stream, copy_stream  two different streams (NULL = legacy default)
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister), else the
 * copies are staged synchronously by CUDA. Returns after enqueuing: the outputs are
 * complete once copy_stream has been synchronised.
 */
size_t focus_host_workspace_size(const focus_params* p, int n_groups);
/* The groups focus_attn_fwd_host uses for (p, n_groups): writes the KV heads of
 * each group, in order, to kv_heads[0 .. min(count, max_groups)) (kv_heads may be
 * NULL) and returns the number of groups, or a negative FOCUS_ERR_* code. */
int focus_host_groups(const focus_params* p, int n_groups, int32_t* kv_heads, int max_groups);
int focus_attn_fwd_host(const focus_params* p, const uint16_t* q_h, const uint16_t* k_h,
                        const uint16_t* v_h, const float* r_h, const float* C_h, uint16_t* o_h,
                        float* lse_h, int n_groups, void* ws, size_t ws_bytes,
                        void* compute_stream, void* copy_stream);

/* Synchronises `stream` and returns the device status word of the last call
 * that used this workspace (FOCUS_OK, FOCUS_ERR_TIMEOUT, FOCUS_ERR_BOUNDS,
 * FOCUS_ERR_NONFINITE), or
 * FOCUS_ERR_CUDA if the synchronisation itself failed. */
int focus_get_status(const void* ws, void* stream);

/*
 * Decode step: the newest token of each sequence (position N - 1) attends to its
 * cache over the same union set as focus_attn_fwd (window keys i - j < w, plus
 * keys whose group bitmask meets the token's).
 *   q        [B, H, d_head] bf16: queries of the newest tokens
 *   k_cache, v_cache  [B, N, H_kv, d_head] bf16: all N cached tokens, the newest
 *            token's key and value included at position N - 1
 *   mask     [B, R, N] uint32: group bitmasks of all N tokens (the newest included;
 *            e.g. from focus_route on its routing vector)
 *   o        [B, H, d_head] bf16 out;  lse [B, H] fp32 out or NULL
 *   ws       focus_decode_workspace_size(p) bytes
 * p->N is the cache length including the newest token. Split over the keys in
 * slices (one warp per slice, KV head and up to 8 of its query heads, streaming the
 * slice's allowed K and V rows through shared memory), then an LSE merge of the
 * slices. The workspace holds the slices' partial results only.
 */
size_t focus_decode_workspace_size(const focus_params* p);
int focus_decode(const focus_params* p, const uint16_t* q, const uint16_t* k_cache,
                 const uint16_t* v_cache, const uint32_t* mask, uint16_t* o, float* lse,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * Backward pass of focus_attn_fwd with the group masks held fixed (hard top-k):
 * gradients of the loss with respect to q, k and v, given its gradient dO with
 * respect to o.  With P_ij = exp(scale q_i.k_j - LSE_i) over the same union set
 * A_i:  dP_ij = dO_i.v_j,  D_i = dO_i.o_i,  dS_ij = P_ij (dP_ij - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i,
 * where a KV head sums over the query heads that read it.  The masks are piecewise
 * constant in r and C, so the routing inputs get no gradient (none is returned).
 *   q, o, d_o  [B, N, H, d_head] bf16 (o: the forward output)
 *   k, v       [B, N, H_kv, d_head] bf16
 *   mask       [B, R, N] uint32: the masks the forward used (e.g. focus_route's)
 *   lse        [B, H, N] fp32: the forward's LSE
 *   dq         [B, N, H, d_head] bf16 out;  dk, dv [B, N, H_kv, d_head] bf16 out
 *   ws         focus_bwd_workspace_size(p) bytes
 * The long-range schedule is chosen as for the forward (focus_bucket_shape).
 * Steps on `stream`: bucket, block schedule and backward plans, permuted copies
 * of Q/K/V/dO, D, then per pass (window, long-range) a query-major dQ kernel and
 * a key-major dK/dV kernel on the tensor cores; with group lists the long-range
 * pass writes each list's part of a token's gradients to one of top_k slots and a
 * last kernel sums them with the window part.  Deterministic: no atomics.
 */
size_t focus_bwd_workspace_size(const focus_params* p);
int focus_attn_bwd(const focus_params* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const uint32_t* mask, const uint16_t* o, const float* lse, const uint16_t* d_o,
                   uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * focus_attn_bwd with stage timing (as focus_attn_fwd_ev): FOCUS_BWD_STAGE_EVENTS
 * caller-created cudaEvent_t handles (or NULL), recorded on `stream` at [0] start,
 * [1] after bucketing, plans, permuted copies and D, [2] after the window pass
 * (dQ and dK/dV kernels), [3] after the long-range dQ kernel, [4] after the
 * long-range dK/dV kernel.
 */
#define FOCUS_BWD_STAGE_EVENTS 5
int focus_attn_bwd_ev(const focus_params* p, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const uint32_t* mask, const uint16_t* o, const float* lse,
                      const uint16_t* d_o, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws,
                      size_t ws_bytes, void* stream, void* const* stage_events);

/*
 * Diagnostic of the device-side failure path (no counterpart in the paper): runs
 * the attention kernel on a tiny problem with its TMA producer held back and
 * ~10 ms wait limits, so the tensor-core issuer's first bounded wait runs out. The
 * kernel must raise FOCUS_ERR_TIMEOUT, abort every role, free its tensor memory
 * and exit, leaving the CUDA context usable. Synchronises `stream` and returns
 * the status word (FOCUS_ERR_TIMEOUT when the failure path works).
 *   ws  device buffer of at least 1 MiB, 256-byte aligned (contents overwritten)
 */
int focus_selftest_timeout(void* ws, size_t ws_bytes, void* stream);

/* Static, human-readable text for a status code. */
const char* focus_strerror(int code);

/* Text of the last CUDA error behind a FOCUS_ERR_CUDA returned to this host thread
 * (cudaGetErrorString), or "no CUDA error". */
const char* focus_cuda_error_string(void);

/* ABI version, (major << 16) | minor. */
int focus_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FOCUS_H_ */
