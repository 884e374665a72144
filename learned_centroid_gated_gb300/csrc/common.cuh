// Shared device/host definitions of the Focus CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/focus.h"

namespace focus {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- workspace --
// Header at the start of the workspace: device status word and counters.
struct WsHeader {
  int status;       // first error code raised by a kernel, 0 if none
  int qtab_count;   // number of query blocks in the long-range schedule
  int item_counter[4];  // next work item of each persistent attention kernel of a call
  int pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Query-block entry of the long-range schedule: routing problem (b * R + rho),
// segment, first permuted row, number of rows.
struct QBlock {
  int br, seg, row0, rows;
};

// Long-range plan of one query block: its compatible key segments, in segment
// order, each as (first permuted row, keys with pos <= p_hi - w, leading tiles
// whose keys all satisfy pos <= p_lo - w), and the total number of key tiles.
struct PlanHead {
  int n_ent, n_tiles, pad0, pad1;
};
struct PlanEnt {
  int start, cnt, nfull, pad;
};

constexpr int kKeyTile = 128;     // keys per attention key tile
constexpr int kChunk = 1024;      // tokens per bucketing chunk (one warp)
constexpr int kSinkBlock = 256;   // tokens per Sinkhorn partial-reduction block
constexpr int kAttnBM = 256;      // query rows per long-range work item
constexpr int kBwdBlock = 128;    // backward: query rows (dQ) or key rows (dK, dV) per item
constexpr int kBwdKeyTile = 128;  // backward dQ: keys per tile
constexpr int kBwdQryTile = 128;  // backward dK, dV: queries per tile

// Workspace layout.  Segment schedule: nseg = C(K, top_k) segments over NR = N rows
// per (b, rho).  Group schedule: nseg = K lists over NR = N * top_k rows, plus the
// permuted masks (pmask) and top_k per-list partial results per token (oslot,
// lseslot: [top_k][B, N, H, d] fp32 and [top_k][B, H, N]).
struct WsLayout {
  size_t hdr, mask, beta, skpart, hist, segoff, cbase, perm, pmask, entoff, qtab, plan_head,
      plan_ent, qp, kp, vp, olr, lselr, oslot, lseslot;
  size_t total;
  int nseg, nchunk, nblk_sk, qtab_cap;
  int group;  // 1: group-list schedule
  int NR;     // permuted rows per (b, rho)
};

// Backward workspace: the exact-set bucketing and the 128-row block schedule (in
// L), the backward plans (query-major and key-major), the permuted dO, D = dO . O
// and the window pass's fp32 partial gradients.
struct BwdPlan {
  WsLayout L;
  size_t qhead, qent, rhead, rent, dop, dvec, dqw, dkw, dvw;
  size_t dqs, dks, dvs;  // group lists: [top_k][...] fp32 list parts of dq, dk, dv
};

// Binomial coefficient C(n, r) for n <= 32 (fits uint32 for all r).
__host__ __device__ inline uint32_t binom(int n, int r) {
  if (r < 0 || r > n) return 0;
  if (r > n - r) r = n - r;
  uint64_t c = 1;
  for (int i = 1; i <= r; ++i) c = c * (uint64_t)(n - r + i) / (uint64_t)i;
  return (uint32_t)c;
}

// Raise a device status code (the first one raised wins).
__device__ inline void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

// Index checks of the debug build (compiled with FOCUS_DEBUG_BOUNDS, see build.py): an
// index read from device data that falls outside its array raises FOCUS_ERR_BOUNDS on
// the status word and the access is skipped.  In the default build the check is
// `true` and costs nothing.
#ifdef FOCUS_DEBUG_BOUNDS
__device__ inline bool in_bounds(bool ok, int* status) {
  if (!ok && status) raise_status(status, FOCUS_ERR_BOUNDS);
  return ok;
}
#define FOCUS_IN_BOUNDS(cond, status) ::focus::in_bounds((cond), (status))
#else
#define FOCUS_IN_BOUNDS(cond, status) true
#endif

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ kernel launchers --
// route.cu
// status: device status word for FOCUS_ERR_NONFINITE, or nullptr
cudaError_t launch_route(const focus_params& p, const WsLayout& L, const float* r, const float* C,
                         char* ws, uint32_t* mask_out, float* margin_out, int* status,
                         cudaStream_t s);
// focus_api.cu: shape checks shared by every entry point (host only)
int check_params(const focus_params* p);
// bucket.cu
cudaError_t launch_bucket(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                          cudaStream_t s);
cudaError_t launch_qtab(const focus_params& p, const WsLayout& L, char* ws, int block_rows,
                        cudaStream_t s);
cudaError_t launch_plan(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                        int block_rows, cudaStream_t s);
cudaError_t launch_permute(const focus_params& p, const WsLayout& L, const bf16* q, const bf16* k,
                           const bf16* v, char* ws, cudaStream_t s);
cudaError_t launch_plan_bwd(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                            PlanHead* qheads, PlanEnt* qents, PlanHead* rheads, PlanEnt* rents,
                            cudaStream_t s);
// merge.cu (group schedule)
cudaError_t launch_merge_slots(const focus_params& p, const WsLayout& L, const char* ws, bf16* o,
                               float* lse, cudaStream_t s);
// attn_bwd.cu (backward)
cudaError_t launch_bwd_rowdot(const focus_params& p, const bf16* o, const bf16* d_o, float* dvec,
                              cudaStream_t s);
cudaError_t launch_permute_rows(const focus_params& p, const WsLayout& L, const bf16* src, bf16* dst,
                                const char* ws, cudaStream_t s);
cudaError_t launch_attn_bwd(const focus_params& p, const BwdPlan& bp, const bf16* q, const bf16* k,
                            const bf16* v, const bf16* d_o, const float* lse, bf16* dq, bf16* dk,
                            bf16* dv, char* ws, float scale, bool long_pass, bool dq_kernel,
                            cudaStream_t s);
cudaError_t launch_bwd_merge_slots(const focus_params& p, const BwdPlan& bp, const char* ws, bf16* dq,
                                   bf16* dk, bf16* dv, cudaStream_t s);
// decode.cu
size_t decode_workspace_bytes(const focus_params& p);
cudaError_t launch_decode(const focus_params& p, const bf16* q, const bf16* k, const bf16* v,
                          const uint32_t* mask, bf16* o, float* lse, char* ws, float scale,
                          cudaStream_t s);
// attn_tc.cu (tcgen05 engine)
int tc_block_rows();
cudaError_t launch_timeout_selftest(char* ws, size_t ws_bytes, cudaStream_t s);
cudaError_t launch_attn_long_tc(const focus_params& p, const WsLayout& L, char* ws, bf16* o,
                                float* lse, float scale, cudaStream_t s);
// attn_pair.cu (long-range pass on CTA pairs: d = 128, exact-set segments)
bool pair_engine_supported(const focus_params& p, const WsLayout& L);
cudaError_t launch_attn_long_pair(const focus_params& p, const WsLayout& L, char* ws, bf16* o,
                                  float* lse, float scale, cudaStream_t s);
cudaError_t launch_attn_window_tc(const focus_params& p, const WsLayout& L, const bf16* q,
                                  const bf16* k, const bf16* v, char* ws, float scale,
                                  cudaStream_t s);

}  // namespace focus
