// C ABI of the Focus attention library: argument validation, workspace layout
// and the launch sequence on the caller's stream.  See include/focus.h.
#include <math.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

namespace focus {
namespace {

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

// The schedule that runs.  AUTO compares estimates of the tensor-core work, as a
// fraction of dense causal attention:
//   segments:    P(two uniform top_k-sets of K intersect) = 1 - C(K-k, k) / C(K, k),
//                times (1 + 2 * C(K, k) * 256 / N) for the ragged query blocks and
//                key tiles of C(K, k) segments over N tokens;
//   group lists: 1.15 * k^2 / K (K lists of N k / K rows, each a dense causal
//                problem; 15 % for the lowest-group test, list imbalance, the merge).
// top_k = 1 makes both the same partition, so segments (no merge pass).
bool use_groups(const focus_params& p) {
  if (p.schedule == FOCUS_SCHEDULE_GROUPS) return true;
  if (p.schedule == FOCUS_SCHEDULE_SEGMENTS) return false;
  if (p.top_k == 1) return false;
  const double sets = (double)binom(p.K, p.top_k);
  if (sets > (double)FOCUS_MAX_SEGMENTS) return true;
  const double meet = 1.0 - (double)binom(p.K - p.top_k, p.top_k) / sets;
  const double seg = meet * (1.0 + 2.0 * sets * (double)kAttnBM / (double)p.N);
  const double grp = 1.15 * (double)p.top_k * (double)p.top_k / (double)p.K;
  return grp < seg;
}

}  // namespace

// Shape checks shared by every entry point (host only, nothing launched).
int check_params(const focus_params* p) {
  if (!p) return FOCUS_ERR_INVALID_ARG;
  if (p->B < 1 || p->N < 1 || p->H < 1 || p->H_kv < 1 || p->R < 1 || p->K < 1 || p->top_k < 1 ||
      p->w < 1 || p->sinkhorn_iters < 0)
    return FOCUS_ERR_INVALID_ARG;
  if (p->H % p->H_kv != 0 || p->H_kv % p->R != 0) return FOCUS_ERR_INVALID_ARG;
  if (p->K > FOCUS_MAX_K || p->top_k > p->K) return FOCUS_ERR_INVALID_ARG;
  if (p->sinkhorn_iters > 0 && !(p->sinkhorn_eps > 0.0f)) return FOCUS_ERR_INVALID_ARG;
  if (p->schedule < FOCUS_SCHEDULE_AUTO || p->schedule > FOCUS_SCHEDULE_GROUPS)
    return FOCUS_ERR_INVALID_ARG;
  if (p->d_head != 64 && p->d_head != 128) return FOCUS_ERR_UNSUPPORTED;
  const bool group = use_groups(*p);
  if (!group && binom(p->K, p->top_k) > (uint32_t)FOCUS_MAX_SEGMENTS) return FOCUS_ERR_UNSUPPORTED;
  // 32-bit row indices: B * max(H, R) * (permuted rows per problem) must fit in int32
  const int64_t rows = (int64_t)p->B * (p->H > p->R ? p->H : p->R) * p->N * (group ? p->top_k : 1);
  if (rows >= (int64_t)INT32_MAX) return FOCUS_ERR_UNSUPPORTED;
  return FOCUS_OK;
}

namespace {

// NVTX ranges that name the stages of a call for a profiler (a no-op unless one is
// attached): at(i) closes the previous stage's range and opens stage i's.
class StageRanges {
 public:
  explicit StageRanges(const char* const* names, int count) : names_(names), count_(count) {}
  void at(int i) {
    if (open_) nvtxRangePop();
    open_ = i < count_;
    if (open_) nvtxRangePushA(names_[i]);
  }
  ~StageRanges() {
    if (open_) nvtxRangePop();
  }

 private:
  const char* const* names_;
  int count_;
  bool open_ = false;
};

WsLayout layout(const focus_params& p) {
  WsLayout L{};
  const int BR = p.B * p.R;
  L.group = use_groups(p) ? 1 : 0;
  L.nseg = L.group ? p.K : (int)binom(p.K, p.top_k);
  L.NR = L.group ? p.N * p.top_k : p.N;
  L.nchunk = (p.N + kChunk - 1) / kChunk;
  L.nblk_sk = (p.N + kSinkBlock - 1) / kSinkBlock;
  L.qtab_cap = BR * ((L.NR + kAttnBM - 1) / kAttnBM + L.nseg);
  const size_t A = 256;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, A);
    return at;
  };
  L.hdr = take(sizeof(WsHeader));
  L.mask = take(sizeof(uint32_t) * (size_t)BR * p.N);
  L.beta = take(sizeof(float) * (size_t)BR * p.K);
  L.skpart = take(sizeof(float2) * (size_t)BR * L.nblk_sk * p.K);
  L.hist = take(sizeof(int) * (size_t)BR * L.nchunk * L.nseg);
  L.segoff = take(sizeof(int) * (size_t)BR * (L.nseg + 1));
  L.cbase = take(sizeof(int) * (size_t)BR * L.nchunk * L.nseg);
  L.perm = take(sizeof(int) * (size_t)BR * L.NR);
  L.pmask = take(L.group ? sizeof(uint32_t) * (size_t)BR * L.NR : 0);
  L.entoff = take(sizeof(int) * ((size_t)BR * L.nseg + 1));
  L.qtab = take(sizeof(QBlock) * (size_t)L.qtab_cap);
  L.plan_head = take(sizeof(PlanHead) * (size_t)L.qtab_cap);
  L.plan_ent = take(sizeof(PlanEnt) * (size_t)L.qtab_cap * L.nseg);
  L.qp = take(sizeof(uint16_t) * (size_t)p.B * p.H * L.NR * p.d_head);
  L.kp = take(sizeof(uint16_t) * (size_t)p.B * p.H_kv * L.NR * p.d_head);
  L.vp = take(sizeof(uint16_t) * (size_t)p.B * p.H_kv * L.NR * p.d_head);
  L.olr = take(sizeof(float) * (size_t)p.B * p.N * p.H * p.d_head);
  L.lselr = take(sizeof(float) * (size_t)p.B * p.H * p.N);
  const size_t slots = L.group ? (size_t)p.top_k : 0;
  L.oslot = take(sizeof(float) * slots * p.B * p.N * p.H * p.d_head);
  L.lseslot = take(sizeof(float) * slots * p.B * p.H * p.N);
  L.total = off;
  return L;
}

// Backward: the same schedule choice as the forward (exact-set segments or group
// lists) over 128-row blocks.
int check_bwd_params(const focus_params* p) { return check_params(p); }

BwdPlan bwd_layout(const focus_params& p) {
  BwdPlan bp{};
  WsLayout& L = bp.L;
  const int BR = p.B * p.R;
  L.group = use_groups(p) ? 1 : 0;
  L.nseg = L.group ? p.K : (int)binom(p.K, p.top_k);
  L.NR = L.group ? p.N * p.top_k : p.N;
  L.nchunk = (p.N + kChunk - 1) / kChunk;
  L.nblk_sk = (p.N + kSinkBlock - 1) / kSinkBlock;
  L.qtab_cap = BR * ((L.NR + kBwdBlock - 1) / kBwdBlock + L.nseg);
  const size_t A = 256;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, A);
    return at;
  };
  const size_t BHN = (size_t)p.B * p.H * p.N, BKN = (size_t)p.B * p.H_kv * p.N;
  const size_t rep = L.group ? (size_t)p.top_k : 1;  // permuted rows per token
  L.hdr = take(sizeof(WsHeader));
  L.hist = take(sizeof(int) * (size_t)BR * L.nchunk * L.nseg);
  L.segoff = take(sizeof(int) * (size_t)BR * (L.nseg + 1));
  L.cbase = take(sizeof(int) * (size_t)BR * L.nchunk * L.nseg);
  L.perm = take(sizeof(int) * (size_t)BR * L.NR);
  L.pmask = take(L.group ? sizeof(uint32_t) * (size_t)BR * L.NR : 0);
  L.entoff = take(sizeof(int) * ((size_t)BR * L.nseg + 1));
  L.qtab = take(sizeof(QBlock) * (size_t)L.qtab_cap);
  L.qp = take(sizeof(uint16_t) * BHN * rep * p.d_head);
  L.kp = take(sizeof(uint16_t) * BKN * rep * p.d_head);
  L.vp = take(sizeof(uint16_t) * BKN * rep * p.d_head);
  bp.qhead = take(sizeof(PlanHead) * (size_t)L.qtab_cap);
  bp.qent = take(sizeof(PlanEnt) * (size_t)L.qtab_cap * L.nseg);
  bp.rhead = take(sizeof(PlanHead) * (size_t)L.qtab_cap);
  bp.rent = take(sizeof(PlanEnt) * (size_t)L.qtab_cap * L.nseg);
  bp.dop = take(sizeof(uint16_t) * BHN * rep * p.d_head);
  bp.dvec = take(sizeof(float) * BHN);
  bp.dqw = take(sizeof(float) * BHN * p.d_head);
  bp.dkw = take(sizeof(float) * BKN * p.d_head);
  bp.dvw = take(sizeof(float) * BKN * p.d_head);
  const size_t slots = L.group ? (size_t)p.top_k : 0;
  bp.dqs = take(sizeof(float) * slots * BHN * p.d_head);
  bp.dks = take(sizeof(float) * slots * BKN * p.d_head);
  bp.dvs = take(sizeof(float) * slots * BKN * p.d_head);
  L.total = off;
  return bp;
}

int check_ws(const WsLayout& L, const void* ws, size_t ws_bytes) {
  if (!ws) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return FOCUS_ERR_ALIGNMENT;
  if (ws_bytes < L.total) return FOCUS_ERR_WORKSPACE;
  return FOCUS_OK;
}

// The last CUDA error an entry point met on this host thread (focus_cuda_error_string).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return FOCUS_OK;
  g_last_cuda_error = e;
  return FOCUS_ERR_CUDA;
}

// Clears the status word and the schedule counter at the start of a call.
cudaError_t reset_header(char* ws, cudaStream_t s) {
  return cudaMemsetAsync(ws, 0, sizeof(WsHeader), s);
}

}  // namespace
}  // namespace focus

using namespace focus;

extern "C" {

size_t focus_workspace_size(const focus_params* p) {
  if (check_params(p) != FOCUS_OK) return 0;
  return layout(*p).total;
}

int focus_bucket_shape(const focus_params* p, int32_t* n_segments, int32_t* rows) {
  const int rc = check_params(p);
  if (rc) return rc;
  const WsLayout L = layout(*p);
  if (n_segments) *n_segments = L.nseg;
  if (rows) *rows = L.NR;
  return L.group ? FOCUS_SCHEDULE_GROUPS : FOCUS_SCHEDULE_SEGMENTS;
}

int focus_route(const focus_params* p, const float* r, const float* C, uint32_t* mask_out,
                float* margin_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!r || !C || !mask_out) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(r, 16) || !aligned(C, 4) || !aligned(mask_out, 4) || !aligned(margin_out, 4))
    return FOCUS_ERR_ALIGNMENT;
  const WsLayout L = layout(*p);
  if ((rc = check_ws(L, ws, ws_bytes))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  if ((rc = cuda_rc(reset_header(w, s)))) return rc;
  return cuda_rc(launch_route(*p, L, r, C, w, mask_out, margin_out,
                              &reinterpret_cast<WsHeader*>(w)->status, s));
}

int focus_bucket(const focus_params* p, const uint32_t* mask, int32_t* perm_out,
                 int32_t* seg_off_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!mask) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(mask, 4) || !aligned(perm_out, 4) || !aligned(seg_off_out, 4))
    return FOCUS_ERR_ALIGNMENT;
  const WsLayout L = layout(*p);
  if ((rc = check_ws(L, ws, ws_bytes))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  if ((rc = cuda_rc(reset_header(w, s)))) return rc;
  if ((rc = cuda_rc(launch_bucket(*p, L, mask, w, s)))) return rc;
  const size_t BR = (size_t)p->B * p->R;
  if (perm_out &&
      (rc = cuda_rc(cudaMemcpyAsync(perm_out, w + L.perm, sizeof(int) * BR * L.NR,
                                    cudaMemcpyDeviceToDevice, s))))
    return rc;
  if (seg_off_out &&
      (rc = cuda_rc(cudaMemcpyAsync(seg_off_out, w + L.segoff, sizeof(int) * BR * (L.nseg + 1),
                                    cudaMemcpyDeviceToDevice, s))))
    return rc;
  return FOCUS_OK;
}

int focus_attn_fwd_ev(const focus_params* p, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const float* r, const float* C,
                      const uint32_t* mask_in, uint16_t* o, float* lse, void* ws,
                      size_t ws_bytes, void* stream, void* const* stage_events) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!q || !k || !v || !o) return FOCUS_ERR_INVALID_ARG;
  if (!mask_in && (!r || !C)) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(mask_in, 4) || !aligned(r, 16) || !aligned(C, 4))
    return FOCUS_ERR_ALIGNMENT;
  const WsLayout L = layout(*p);
  if ((rc = check_ws(L, ws, ws_bytes))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const float scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / sqrtf((float)p->d_head);
  const bf16* qb = reinterpret_cast<const bf16*>(q);
  const bf16* kb = reinterpret_cast<const bf16*>(k);
  const bf16* vb = reinterpret_cast<const bf16*>(v);
  static const char* const kStageNames[] = {"focus fwd: routing", "focus fwd: bucketing",
                                            "focus fwd: permuted copies", "focus fwd: window",
                                            "focus fwd: long-range"};
  StageRanges ranges(kStageNames, 5);
  auto mark = [&](int i) -> int {
    ranges.at(i);
    if (!stage_events) return FOCUS_OK;
    return cuda_rc(cudaEventRecord((cudaEvent_t)stage_events[i], s));
  };

  if ((rc = mark(0))) return rc;
  if ((rc = cuda_rc(reset_header(w, s)))) return rc;
  const uint32_t* mask = mask_in;
  if (!mask) {
    uint32_t* m = reinterpret_cast<uint32_t*>(w + L.mask);
    if ((rc = cuda_rc(launch_route(*p, L, r, C, w, m, nullptr,
                                   &reinterpret_cast<WsHeader*>(w)->status, s))))
      return rc;
    mask = m;
  }
  if ((rc = mark(1))) return rc;
  if ((rc = cuda_rc(launch_bucket(*p, L, mask, w, s)))) return rc;
  if ((rc = cuda_rc(launch_qtab(*p, L, w, tc_block_rows(), s)))) return rc;
  if ((rc = cuda_rc(launch_plan(*p, L, mask, w, tc_block_rows(), s)))) return rc;
  if ((rc = mark(2))) return rc;
  if ((rc = cuda_rc(launch_permute(*p, L, qb, kb, vb, w, s)))) return rc;
  if ((rc = mark(3))) return rc;
  if ((rc = cuda_rc(launch_attn_window_tc(*p, L, qb, kb, vb, w, scale, s)))) return rc;
  if ((rc = mark(4))) return rc;
  if ((rc = cuda_rc(launch_attn_long_tc(*p, L, w, reinterpret_cast<bf16*>(o), lse, scale, s))))
    return rc;
  if (L.group &&
      (rc = cuda_rc(launch_merge_slots(*p, L, w, reinterpret_cast<bf16*>(o), lse, s))))
    return rc;
  return mark(5);
}

int focus_attn_fwd(const focus_params* p, const uint16_t* q, const uint16_t* k,
                   const uint16_t* v, const float* r, const float* C, const uint32_t* mask_in,
                   uint16_t* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return focus_attn_fwd_ev(p, q, k, v, r, C, mask_in, o, lse, ws, ws_bytes, stream, nullptr);
}

// ------------------------------------------------------------ host buffers --
namespace {

// Head groups of the host-buffer entry: runs of consecutive KV heads (with their
// query heads and, when R > 1, their routing heads), as (first KV head, KV heads).
// A group must hold whole routing heads when R > 1, so sizes are multiples of
// unit = H_kv / R (1 when R = 1).
struct HostGroups {
  int n = 0;
  int off[64], cnt[64];
  int max_cnt = 0;
};

// n_groups > 0: that many equal groups (it must divide H_kv and, when R > 1, R).
// n_groups == 0: automatic.  The first group's inputs and the last group's outputs
// cannot overlap any compute, so those two groups are small (about an eighth of
// the heads each) and the rest is split into groups of about a quarter; problems
// with fewer than four units use equal groups of one unit.
bool host_groups(const focus_params& p, int n_groups, HostGroups* G) {
  const int unit = p.R == 1 ? 1 : p.H_kv / p.R;
  const int U = p.H_kv / unit;  // units of whole routing heads
  G->n = 0;
  auto add = [&](int units) {
    G->off[G->n] = (G->n ? G->off[G->n - 1] + G->cnt[G->n - 1] : 0);
    G->cnt[G->n] = units * unit;
    if (G->cnt[G->n] > G->max_cnt) G->max_cnt = G->cnt[G->n];
    ++G->n;
  };
  if (n_groups > 0) {
    if (n_groups > 64 || p.H_kv % n_groups != 0 || (p.R != 1 && p.R % n_groups != 0)) return false;
    const int per = p.H_kv / n_groups;
    for (int g = 0; g < n_groups; ++g) {
      G->off[g] = g * per;
      G->cnt[g] = per;
    }
    G->n = n_groups;
    G->max_cnt = per;
    return true;
  }
  if (U < 4) {
    for (int g = 0; g < U; ++g) add(1);
    return true;
  }
  const int edge = U / 8 > 1 ? U / 8 : 1;
  const int mid = U - 2 * edge;
  const int quarter = U / 4 > 1 ? U / 4 : 1;
  const int n_mid = (mid + quarter - 1) / quarter;
  if (2 + n_mid > 64) return false;
  add(edge);
  for (int g = 0, left = mid; g < n_mid; ++g) {
    const int take = left / (n_mid - g);  // near-equal middle groups
    add(take);
    left -= take;
  }
  add(edge);
  return true;
}

focus_params group_params(const focus_params& p, int kv_cnt) {
  focus_params q = p;
  const int gq = p.H / p.H_kv;
  q.H = kv_cnt * gq;
  q.H_kv = kv_cnt;
  q.R = p.R == 1 ? 1 : kv_cnt / (p.H_kv / p.R);
  return q;
}

struct HostLayout {
  size_t q, k, v, o, lse, r, set_bytes, C, attn, attn_bytes, total;
};

HostLayout host_layout(const focus_params& p, const HostGroups& G) {
  const focus_params g = group_params(p, G.max_cnt);
  HostLayout H{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  const size_t BN = (size_t)p.B * p.N;
  H.q = take(BN * g.H * p.d_head * 2);
  H.k = take(BN * g.H_kv * p.d_head * 2);
  H.v = take(BN * g.H_kv * p.d_head * 2);
  H.o = take(BN * g.H * p.d_head * 2);
  H.lse = take((size_t)p.B * g.H * p.N * 4);
  H.r = take(BN * g.R * FOCUS_D_G * 4);
  H.set_bytes = off;
  off = 2 * H.set_bytes;  // two staging sets
  H.C = take((size_t)p.K * FOCUS_D_G * 4);
  H.attn_bytes = layout(g).total;  // the largest group's workspace serves every group
  H.attn = take(H.attn_bytes);
  H.total = off;
  return H;
}

}  // namespace

size_t focus_host_workspace_size(const focus_params* p, int n_groups) {
  if (check_params(p) != FOCUS_OK) return 0;
  HostGroups G;
  if (!host_groups(*p, n_groups, &G)) return 0;
  return host_layout(*p, G).total;
}

int focus_host_groups(const focus_params* p, int n_groups, int32_t* kv_heads, int max_groups) {
  int rc = check_params(p);
  if (rc) return rc;
  HostGroups G;
  if (!host_groups(*p, n_groups, &G)) return FOCUS_ERR_INVALID_ARG;
  for (int g = 0; kv_heads && g < G.n && g < max_groups; ++g) kv_heads[g] = G.cnt[g];
  return G.n;
}

int focus_attn_fwd_host(const focus_params* p, const uint16_t* q_h, const uint16_t* k_h,
                        const uint16_t* v_h, const float* r_h, const float* C_h, uint16_t* o_h,
                        float* lse_h, int n_groups, void* ws, size_t ws_bytes,
                        void* compute_stream, void* copy_stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!q_h || !k_h || !v_h || !r_h || !C_h || !o_h) return FOCUS_ERR_INVALID_ARG;
  HostGroups G;
  if (!host_groups(*p, n_groups, &G)) return FOCUS_ERR_INVALID_ARG;
  if (compute_stream == copy_stream) return FOCUS_ERR_INVALID_ARG;
  const HostLayout HL = host_layout(*p, G);
  if (!ws) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return FOCUS_ERR_ALIGNMENT;
  if (ws_bytes < HL.total) return FOCUS_ERR_WORKSPACE;
  cudaStream_t cs = (cudaStream_t)compute_stream, xs = (cudaStream_t)copy_stream;
  char* w = (char*)ws;
  const size_t d2 = (size_t)p->d_head * 2;
  const size_t BN = (size_t)p->B * p->N;
  const int gq = p->H / p->H_kv;                   // query heads per KV head
  const int kv_per_rho = p->H_kv / p->R;           // KV heads per routing head

  cudaEvent_t ev_in[2], ev_comp[2];
  for (int i = 0; i < 2; ++i) {
    if (cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev_comp[i], cudaEventDisableTiming) != cudaSuccess)
      return FOCUS_ERR_CUDA;
  }
  auto cleanup = [&](int code) {
    for (int i = 0; i < 2; ++i) {
      cudaEventDestroy(ev_in[i]);
      cudaEventDestroy(ev_comp[i]);
    }
    return code;
  };
  auto set_ptr = [&](int g, size_t off) { return w + (g & 1) * HL.set_bytes + off; };
  // inputs of group g into staging set g % 2 (strided 2-D copies out of the host layout)
  auto copy_in = [&](int g) -> cudaError_t {
    const focus_params gp = group_params(*p, G.cnt[g]);
    const size_t kv0 = (size_t)G.off[g], h0 = kv0 * gq;
    cudaError_t e;
    if (g >= 2 && (e = cudaStreamWaitEvent(xs, ev_comp[g & 1], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpy2DAsync(set_ptr(g, HL.q), gp.H * d2, q_h + h0 * p->d_head, p->H * d2,
                               gp.H * d2, BN, cudaMemcpyHostToDevice, xs)))
      return e;
    if ((e = cudaMemcpy2DAsync(set_ptr(g, HL.k), gp.H_kv * d2, k_h + kv0 * p->d_head,
                               p->H_kv * d2, gp.H_kv * d2, BN, cudaMemcpyHostToDevice, xs)))
      return e;
    if ((e = cudaMemcpy2DAsync(set_ptr(g, HL.v), gp.H_kv * d2, v_h + kv0 * p->d_head,
                               p->H_kv * d2, gp.H_kv * d2, BN, cudaMemcpyHostToDevice, xs)))
      return e;
    const size_t rw = (size_t)gp.R * FOCUS_D_G * 4;
    const float* rsrc = r_h + (p->R == 1 ? 0 : (kv0 / kv_per_rho) * FOCUS_D_G);
    if ((e = cudaMemcpy2DAsync(set_ptr(g, HL.r), rw, rsrc, (size_t)p->R * FOCUS_D_G * 4, rw, BN,
                               cudaMemcpyHostToDevice, xs)))
      return e;
    return cudaEventRecord(ev_in[g & 1], xs);
  };
  auto copy_out = [&](int g) -> cudaError_t {
    const focus_params gp = group_params(*p, G.cnt[g]);
    const size_t h0 = (size_t)G.off[g] * gq;
    cudaError_t e;
    if ((e = cudaStreamWaitEvent(xs, ev_comp[g & 1], 0))) return e;
    if ((e = cudaMemcpy2DAsync(o_h + h0 * p->d_head, p->H * d2, set_ptr(g, HL.o), gp.H * d2,
                               gp.H * d2, BN, cudaMemcpyDeviceToHost, xs)))
      return e;
    if (lse_h &&
        (e = cudaMemcpy2DAsync(lse_h + h0 * p->N, (size_t)p->H * p->N * 4, set_ptr(g, HL.lse),
                               (size_t)gp.H * p->N * 4, (size_t)gp.H * p->N * 4, p->B,
                               cudaMemcpyDeviceToHost, xs)))
      return e;
    return cudaSuccess;
  };

  if ((rc = cuda_rc(cudaMemcpyAsync(w + HL.C, C_h, (size_t)p->K * FOCUS_D_G * 4,
                                    cudaMemcpyHostToDevice, xs))))
    return cleanup(rc);
  if ((rc = cuda_rc(copy_in(0)))) return cleanup(rc);
  for (int g = 0; g < G.n; ++g) {
    if (g + 1 < G.n && (rc = cuda_rc(copy_in(g + 1)))) return cleanup(rc);
    // compute of group g: inputs landed; staging outputs of set g % 2 were copied out
    // (copy_out(g - 2) precedes copy_in(g) on the copy stream, which the event covers)
    if ((rc = cuda_rc(cudaStreamWaitEvent(cs, ev_in[g & 1], 0)))) return cleanup(rc);
    const focus_params gp = group_params(*p, G.cnt[g]);
    rc = focus_attn_fwd(&gp, reinterpret_cast<const uint16_t*>(set_ptr(g, HL.q)),
                        reinterpret_cast<const uint16_t*>(set_ptr(g, HL.k)),
                        reinterpret_cast<const uint16_t*>(set_ptr(g, HL.v)),
                        reinterpret_cast<const float*>(set_ptr(g, HL.r)),
                        reinterpret_cast<const float*>(w + HL.C), nullptr,
                        reinterpret_cast<uint16_t*>(set_ptr(g, HL.o)),
                        reinterpret_cast<float*>(set_ptr(g, HL.lse)), w + HL.attn, HL.attn_bytes,
                        cs);
    if (rc) return cleanup(rc);
    if ((rc = cuda_rc(cudaEventRecord(ev_comp[g & 1], cs)))) return cleanup(rc);
    if ((rc = cuda_rc(copy_out(g)))) return cleanup(rc);
  }
  return cleanup(FOCUS_OK);
}

size_t focus_bwd_workspace_size(const focus_params* p) {
  if (check_bwd_params(p) != FOCUS_OK) return 0;
  return bwd_layout(*p).L.total;
}

int focus_attn_bwd_ev(const focus_params* p, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const uint32_t* mask, const uint16_t* o, const float* lse,
                      const uint16_t* d_o, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws,
                      size_t ws_bytes, void* stream, void* const* stage_events) {
  int rc = check_bwd_params(p);
  if (rc) return rc;
  if (!q || !k || !v || !mask || !o || !lse || !d_o || !dq || !dk || !dv)
    return FOCUS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(d_o, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(mask, 4) || !aligned(lse, 4))
    return FOCUS_ERR_ALIGNMENT;
  const BwdPlan bp = bwd_layout(*p);
  const WsLayout& L = bp.L;
  if ((rc = check_ws(L, ws, ws_bytes))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const float scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / sqrtf((float)p->d_head);
  const bf16* qb = reinterpret_cast<const bf16*>(q);
  const bf16* kb = reinterpret_cast<const bf16*>(k);
  const bf16* vb = reinterpret_cast<const bf16*>(v);
  const bf16* gb = reinterpret_cast<const bf16*>(d_o);
  bf16* dqb = reinterpret_cast<bf16*>(dq);
  bf16* dkb = reinterpret_cast<bf16*>(dk);
  bf16* dvb = reinterpret_cast<bf16*>(dv);
  static const char* const kStageNames[] = {"focus bwd: prepare", "focus bwd: window",
                                            "focus bwd: long-range dq", "focus bwd: long-range dk dv"};
  StageRanges ranges(kStageNames, 4);
  auto mark = [&](int i) -> int {
    ranges.at(i);
    if (!stage_events) return FOCUS_OK;
    return cuda_rc(cudaEventRecord((cudaEvent_t)stage_events[i], s));
  };
  auto pass = [&](bool long_pass, bool dq_kernel) {
    return cuda_rc(launch_attn_bwd(*p, bp, qb, kb, vb, gb, lse, dqb, dkb, dvb, w, scale, long_pass,
                                   dq_kernel, s));
  };
  if ((rc = mark(0))) return rc;
  if ((rc = cuda_rc(reset_header(w, s)))) return rc;
  if ((rc = cuda_rc(launch_bucket(*p, L, mask, w, s)))) return rc;
  if ((rc = cuda_rc(launch_qtab(*p, L, w, kBwdBlock, s)))) return rc;
  if ((rc = cuda_rc(launch_plan_bwd(*p, L, mask, w, reinterpret_cast<PlanHead*>(w + bp.qhead),
                                    reinterpret_cast<PlanEnt*>(w + bp.qent),
                                    reinterpret_cast<PlanHead*>(w + bp.rhead),
                                    reinterpret_cast<PlanEnt*>(w + bp.rent), s))))
    return rc;
  if ((rc = cuda_rc(launch_permute(*p, L, qb, kb, vb, w, s)))) return rc;
  if ((rc = cuda_rc(launch_permute_rows(*p, L, gb, reinterpret_cast<bf16*>(w + bp.dop), w, s))))
    return rc;
  if ((rc = cuda_rc(launch_bwd_rowdot(*p, reinterpret_cast<const bf16*>(o), gb,
                                      reinterpret_cast<float*>(w + bp.dvec), s))))
    return rc;
  if ((rc = mark(1))) return rc;
  if ((rc = pass(false, true)) || (rc = pass(false, false))) return rc;
  if ((rc = mark(2))) return rc;
  if ((rc = pass(true, true))) return rc;
  if ((rc = mark(3))) return rc;
  if ((rc = pass(true, false))) return rc;
  if (L.group && (rc = cuda_rc(launch_bwd_merge_slots(*p, bp, w, dqb, dkb, dvb, s)))) return rc;
  return mark(4);
}

int focus_attn_bwd(const focus_params* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const uint32_t* mask, const uint16_t* o, const float* lse, const uint16_t* d_o,
                   uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws, size_t ws_bytes,
                   void* stream) {
  return focus_attn_bwd_ev(p, q, k, v, mask, o, lse, d_o, dq, dk, dv, ws, ws_bytes, stream, nullptr);
}

size_t focus_decode_workspace_size(const focus_params* p) {
  if (check_params(p) != FOCUS_OK) return 0;
  return decode_workspace_bytes(*p);
}

int focus_decode(const focus_params* p, const uint16_t* q, const uint16_t* k_cache,
                 const uint16_t* v_cache, const uint32_t* mask, uint16_t* o, float* lse,
                 void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!q || !k_cache || !v_cache || !mask || !o) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(mask, 4) || !aligned(lse, 4))
    return FOCUS_ERR_ALIGNMENT;
  if (!ws) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return FOCUS_ERR_ALIGNMENT;
  if (ws_bytes < decode_workspace_bytes(*p)) return FOCUS_ERR_WORKSPACE;
  const float scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / sqrtf((float)p->d_head);
  return cuda_rc(launch_decode(*p, reinterpret_cast<const bf16*>(q),
                               reinterpret_cast<const bf16*>(k_cache),
                               reinterpret_cast<const bf16*>(v_cache), mask,
                               reinterpret_cast<bf16*>(o), lse, (char*)ws, scale,
                               (cudaStream_t)stream));
}

int focus_selftest_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return FOCUS_ERR_ALIGNMENT;
  if (ws_bytes < ((size_t)1 << 20)) return FOCUS_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  int rc;
  if ((rc = cuda_rc(reset_header(w, s)))) return rc;
  if ((rc = cuda_rc(launch_timeout_selftest(w, ws_bytes, s)))) return rc;
  return focus_get_status(ws, stream);
}

int focus_get_status(const void* ws, void* stream) {
  if (!ws) return FOCUS_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int status = 0;
  if (cudaMemcpyAsync(&status, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FOCUS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FOCUS_ERR_CUDA;
  return status;
}

const char* focus_strerror(int code) {
  switch (code) {
    case FOCUS_OK: return "ok";
    case FOCUS_ERR_INVALID_ARG: return "invalid argument";
    case FOCUS_ERR_UNSUPPORTED: return "unsupported parameters";
    case FOCUS_ERR_WORKSPACE: return "workspace too small";
    case FOCUS_ERR_CUDA: return "CUDA error";
    case FOCUS_ERR_TIMEOUT: return "device wait timed out";
    case FOCUS_ERR_BOUNDS: return "device index check failed (mask with wrong bit count?)";
    case FOCUS_ERR_ALIGNMENT: return "misaligned pointer";
    case FOCUS_ERR_NONFINITE: return "non-finite routing score (NaN or inf in r or C)";
    default: return "unknown status";
  }
}

int focus_version(void) { return (1 << 16) | 0; }

const char* focus_cuda_error_string(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

}  // extern "C"
