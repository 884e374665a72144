// Focus attention backward on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// "Why Attend to Everything? Focus is the Key", gist.science technical summary,
// section 2 "Core Architecture" and "Inference Efficiency (Top-k)": one exact
// softmax over the window keys and the distant keys that share a group.  With the
// hard mask held fixed, the gradients of that softmax are (s = scale q.k over the
// attended set A_i, P = exp(s - LSE)):
//   dP_ij = dO_i . v_j,  D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
// (Section 5 "Significance and Implications" of the same summary notes that
// training with the soft gate still visits all pairs; this is the hard-mask form.)
//
// Two persistent kernels, each in a window pass (token order, keys (i - w, i])
// and a long-range pass (compatible exact-set segments, permuted copies); no
// atomics, so the result is deterministic.  Every tensor-core product has N = 128
// (narrower products ran at a fraction of the rate), so each kernel keeps one
// 128 x 128 tile of S and dP in TMEM at a time:
//   bwd_dq<D, LONG>    query-major: 128 query rows of one head per item (Q resident
//                      in shared memory, dO staged in TMEM); per 128-key tile:
//                      S = Q K^T and dP = dO V^T; the warps read them (and release
//                      them at once, so the next tile's S and dP are computed
//                      meanwhile), write dS (bf16) to TMEM, dQ += dS K.
//   bwd_dkdv<D, LONG>  key-major: 128 key rows of one KV head per item (K and V
//                      resident in shared memory), every query head of its group;
//                      per 128-query tile: S^T = K Q^T, dP^T = V dO^T, P^T and dS^T
//                      (bf16) written over them, dV += P^T dO, dK += dS^T Q (each
//                      warpgroup hands over its first 16 query columns before the
//                      other 16, so half of the dV, dK products overlap the rest).
// TMEM (512 columns): dQ kernel S | dP | dS | dO | dQ, dK/dV kernel S^T | dP^T | dK | dV.
// The window pass writes fp32 partials; the long-range pass adds them and writes
// the bf16 gradients (the two key sets are disjoint, so the sums are the totals).
//
// Warps: 0-15 elementwise (four warpgroups, each 32 columns of every tile, lane =
// TMEM row), 16 producer (TMA; in bwd_dkdv the whole warp also stages the tile's
// per-query LSE, D and position; it also draws the work items from a global counter
// and passes them to the other warps through a shared-memory ring), 17 MMA issuer.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace focus {
namespace {

using namespace ptx;

constexpr int EW_WARPS = 16;             // elementwise warps: four warpgroups
constexpr int EW_THREADS = 32 * EW_WARPS;
constexpr int NTHREADS = EW_THREADS + 64;
constexpr int PRODUCER_WARP = EW_WARPS;
constexpr int MMA_WARP = EW_WARPS + 1;
constexpr int BM = kBwdBlock;       // rows per item
constexpr int NK = kBwdKeyTile;     // keys per dQ tile
constexpr int NQ = kBwdQryTile;     // queries per dK/dV tile
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMinSmem = 116 * 1024;  // > half the SM's shared memory: one CTA per SM

// Kernel modes: window pass, long range over exact-set segments, over group lists.
enum : int { kWin = 0, kSeg = 1, kGrp = 2 };

// Barrier block shared by both kernels: full[NST], empty[NST], then sdp, ds, dqc,
// rd, a, fin, drain, kv_full, kv_empty (8 bytes each), the TMEM address word and
// the abort flag.  (In bwd_dq kv_full / kv_empty guard the item's Q tile.)
constexpr int NRING = 4;            // work-item ring entries
constexpr int RING_CONSUMERS = 1 + EW_WARPS;  // MMA issuer + one lane per elementwise warp
template <int NST>
struct Bars {
  static constexpr int FULL = 0, EMPTY = 8 * NST, SDP = 16 * NST, DS = SDP + 8, DQC = DS + 8;
  static constexpr int RD = DQC + 8, A = RD + 8, FIN = A + 8, DRAIN = FIN + 8, KVF = DRAIN + 8;
  static constexpr int KVE = KVF + 8;
  static constexpr int TMEM_SLOT = KVE + 8, ABORT = TMEM_SLOT + 4;
  // work-item ring: full[NRING], empty[NRING] barriers and the item indices
  static constexpr int RF = (ABORT + 4 + 7) / 8 * 8, RE = RF + 8 * NRING, RING_X = RE + 8 * NRING;
  static constexpr int BYTES = 256;
  static_assert(RING_X + 4 * NRING <= BYTES, "barrier block overflow");
};

// Work items reach the MMA issuer and the elementwise warps through a small ring
// filled by the producer warp from a global counter, so the CTAs share the items
// dynamically in order (a static round-robin share left the average SM idle ~3.5% of
// a long-range launch while the most loaded one finished).  Each item writes only
// its own rows, so the result does not depend on which CTA takes it.
__device__ __forceinline__ bool ring_put(uint32_t rf, uint32_t re, volatile int* rx, int kr, int* counter,
                                         int& x, volatile int* abort_flag, int* status, long long tlim) {
  const int rs = kr % NRING;
  if (!mbar_wait(re + 8 * rs, (uint32_t)(((kr / NRING) & 1) ^ 1), abort_flag, status, tlim)) return false;
  x = atomicAdd(counter, 1);
  rx[rs] = x;
  mbar_arrive(rf + 8 * rs);
  return true;
}
__device__ __forceinline__ bool ring_get(uint32_t rf, uint32_t re, volatile int* rx, int kr, int& x,
                                         volatile int* abort_flag, int* status, long long tlim) {
  const int rs = kr % NRING;
  if (!mbar_wait(rf + 8 * rs, (uint32_t)((kr / NRING) & 1), abort_flag, status, tlim)) return false;
  x = rx[rs];
  mbar_arrive(re + 8 * rs);
  return true;
}
// Whole-warp consumer: every lane waits, lane 0 releases the slot.
__device__ __forceinline__ bool ring_get_warp(uint32_t rf, uint32_t re, volatile int* rx, int kr, int& x,
                                              volatile int* abort_flag, int* status, long long tlim) {
  const int rs = kr % NRING;
  const bool ok = mbar_wait(rf + 8 * rs, (uint32_t)((kr / NRING) & 1), abort_flag, status, tlim);
  if (!__all_sync(0xffffffffu, ok)) return false;
  x = rx[rs];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(re + 8 * rs);
  return true;
}

constexpr int BOX = 128 * 128;  // one TMA box: 128 rows x 128 bytes (64 bf16)

template <int D>
struct DqLayout {
  static constexpr int NST = 3;
  static constexpr int TILE = (D / 64) * BOX;    // one 128-row tile of Q, K or V
  static constexpr int QT = 0;                   // the item's Q tile
  static constexpr int RING = QT + TILE;         // [NST][K tile, V tile]
  static constexpr int KM = RING + NST * 2 * TILE;  // group lists: [NST][NK] key masks
  static constexpr int BAR = KM + NST * NK * 4;
  static constexpr int SMEM = BAR + Bars<NST>::BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  // S | dP | dS (bf16 pairs) | dO (bf16 pairs, A operand of dP) | dQ
  static constexpr int COL_S = 0, COL_DP = NK, COL_DS = 2 * NK, COL_DO = 2 * NK + NK / 2;
  static constexpr int COL_DQ = COL_DO + D / 2;
  static_assert(COL_DQ + D <= (int)TMEM_COLS, "tensor memory budget");
};

template <int D>
struct DkvLayout {
  static constexpr int NST = 2;
  static constexpr int TILE = (D / 64) * BOX;    // one 128-row tile of K, V, Q or dO
  static constexpr int KV = 0;                   // K tile, V tile of the item
  static constexpr int RING = KV + 2 * TILE;     // [NST][Q tile, dO tile]
  static constexpr int SCAL = RING + NST * 2 * TILE;  // [NST][lse2, D, pos, mask][NQ]
  static constexpr int BAR = SCAL + NST * 4 * NQ * 4;
  static constexpr int SMEM = BAR + Bars<NST>::BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr int COL_ST = 0, COL_DPT = NQ, COL_DK = 2 * NQ, COL_DV = 2 * NQ + D;
  static_assert(COL_DV + D <= (int)TMEM_COLS, "tensor memory budget");
};

struct BwdArgs {
  int B, N, H, H_kv, R, w, nseg, qtab_cap, NR;
  float sl2;    // softmax scale * log2(e)
  float scale;  // softmax scale
  const int* perm;
  const QBlock* qtab;
  const int* qtab_count;
  const PlanHead* qhead;
  const PlanEnt* qent;
  const PlanHead* rhead;
  const PlanEnt* rent;
  const bf16* q;
  const bf16* k;
  const bf16* v;
  const bf16* dout;
  const float* lse;   // [B, H, N]
  const float* dvec;  // [B, H, N]: D = dO . O
  float* dq_w;        // window partials, fp32, token order
  float* dk_w;
  float* dv_w;
  bf16* dq;           // gradients, bf16, token order
  bf16* dk;
  bf16* dv;
  const uint32_t* pmask;  // group lists: mask of each permuted row
  float* dq_s;            // group lists: [top_k][B, N, H, d] list parts
  float* dk_s;            // group lists: [top_k][B, N, H_kv, d]
  float* dv_s;
  int* status;
  int* item_counter;  // next work item of this launch (zero before it)
  long long timeout_cycles;
};

struct BItem {
  bool valid;
  int b, h, kvh, br, u, row0, rows, seg;
  int n;     // tiles
  int nsub;  // dK/dV: tiles per query head
  int lo, hi;
};

// dQ items: (query head, 128-row block).  Long: heads sharing a KV head adjacent.
template <bool LONG>
__device__ __forceinline__ BItem dq_item(const BwdArgs& a, int x) {
  BItem it{};
  const int gq = a.H / a.H_kv;
  if constexpr (LONG) {
    const int nkv = a.H_kv / a.R;
    const int jq = x % gq;
    const int rest = x / gq;
    const int u = rest % a.qtab_cap, kvl = rest / a.qtab_cap;
    it.valid = u < *a.qtab_count;
    if (!it.valid) return it;
    const QBlock e = a.qtab[u];
    it.u = u;
    it.br = e.br;
    it.seg = e.seg;
    it.b = e.br / a.R;
    it.kvh = (e.br % a.R) * nkv + kvl;
    it.h = it.kvh * gq + jq;
    it.row0 = e.row0;
    it.rows = e.rows;
    it.n = a.qhead[u].n_tiles;
  } else {
    const int nqb = (a.N + BM - 1) / BM;
    const int bh = x / nqb;
    it.valid = true;
    it.h = bh % a.H;
    it.b = bh / a.H;
    it.kvh = it.h / gq;
    it.row0 = (x % nqb) * BM;
    it.rows = min(BM, a.N - it.row0);
    it.lo = max(0, it.row0 - a.w + 1);
    it.hi = it.row0 + it.rows;
    it.n = (it.hi - it.lo + NK - 1) / NK;
  }
  return it;
}

// dK/dV items: (KV head, 128-row key block).  Long: key blocks of early positions
// (the most queries) first.
template <bool LONG>
__device__ __forceinline__ BItem dkv_item(const BwdArgs& a, int x) {
  BItem it{};
  const int gq = a.H / a.H_kv;
  if constexpr (LONG) {
    const int nkv = a.H_kv / a.R;
    const int ur = x % a.qtab_cap, kvl = x / a.qtab_cap;
    const int cnt = *a.qtab_count;
    it.valid = ur < cnt;
    if (!it.valid) return it;
    const int u = cnt - 1 - ur;
    const QBlock e = a.qtab[u];
    it.u = u;
    it.br = e.br;
    it.seg = e.seg;
    it.b = e.br / a.R;
    it.kvh = (e.br % a.R) * nkv + kvl;
    it.row0 = e.row0;
    it.rows = e.rows;
    it.nsub = a.rhead[u].n_tiles;
    it.n = gq * it.nsub;
  } else {
    const int nkb = (a.N + BM - 1) / BM;
    const int bk = x / nkb;
    it.valid = true;
    it.kvh = bk % a.H_kv;
    it.b = bk / a.H_kv;
    it.row0 = (x % nkb) * BM;
    it.rows = min(BM, a.N - it.row0);
    it.lo = it.row0;
    it.hi = min(a.N, it.row0 + it.rows + a.w - 1);
    it.nsub = (it.hi - it.lo + NQ - 1) / NQ;
    it.n = gq * it.nsub;
  }
  return it;
}

// Walks the key tiles of a dQ item: first key row (permuted row in the long pass,
// token in the window pass), keys in the tile, and whether every key of the tile
// is allowed for every row of the block (long pass).
struct DqWalk {
  int e, t_in;
  PlanEnt pe;
  __device__ __forceinline__ void init(const BwdArgs& a, const BItem& it, bool LONG) {
    e = 0;
    t_in = 0;
    pe = PlanEnt{0, 0, 0, 0};
    if (LONG && it.n > 0) pe = a.qent[(int64_t)it.u * a.nseg];
  }
  // fills (start, cnt, full) of tile t and moves on
  __device__ __forceinline__ void next(const BwdArgs& a, const BItem& it, bool LONG, int t,
                                       int& start, int& cnt, bool& full) {
    if (LONG) {
      start = pe.start + t_in * NK;
      cnt = min(NK, pe.cnt - t_in * NK);
      full = t_in * NK + cnt <= pe.nfull;
      if (++t_in * NK >= pe.cnt && ++e < a.nseg) {
        t_in = 0;
        pe = a.qent[(int64_t)it.u * a.nseg + e];
      }
    } else {
      start = it.lo + t * NK;
      cnt = min(NK, it.hi - start);
      full = false;
    }
  }
};

// Walks the query tiles of a dK/dV item: query head, first query row, count.
struct DkvWalk {
  int jq, e, t_in, n_ent;
  PlanEnt pe;
  __device__ __forceinline__ void init(const BwdArgs& a, const BItem& it, bool LONG) {
    jq = e = t_in = 0;
    n_ent = 0;
    pe = PlanEnt{0, 0, 0, 0};
    if (LONG && it.n > 0) {
      n_ent = a.rhead[it.u].n_ent;
      pe = a.rent[(int64_t)it.u * a.nseg];
    }
  }
  __device__ __forceinline__ void next(const BwdArgs& a, const BItem& it, bool LONG, int t,
                                       int& h, int& start, int& cnt) {
    const int gq = a.H / a.H_kv;
    if (LONG) {
      h = it.kvh * gq + jq;
      start = pe.start + t_in * NQ;
      cnt = min(NQ, pe.cnt - t_in * NQ);
      if (++t_in * NQ >= pe.cnt) {
        t_in = 0;
        if (++e >= n_ent) {
          e = 0;
          ++jq;
        }
        pe = a.rent[(int64_t)it.u * a.nseg + e];
      }
    } else {
      const int s = t % it.nsub;
      h = it.kvh * gq + t / it.nsub;
      start = it.lo + s * NQ;
      cnt = min(NQ, it.hi - start);
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// First index in [lo, hi) with P[index] > x (P ascending), or hi.
__device__ __forceinline__ int upper_bound_g(const int* __restrict__ P, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Stages one bf16 row of D values (src, 16-byte aligned; zeros when src is null)
// into TMEM columns [col, col + D/2) of this thread's lane as bf16 pairs.
template <int D>
__device__ __forceinline__ void stage_row(uint32_t taddr, const bf16* src) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t r[32];
    if (src) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src) + c * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 x = __ldg(s4 + i);
        r[4 * i] = x.x;
        r[4 * i + 1] = x.y;
        r[4 * i + 2] = x.z;
        r[4 * i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
    tmem_st32(taddr + 32 * c, r);
  }
}

// Epilogue helper: 32 fp32 accumulator columns of this lane -> window partial
// (fp32) or, in the long pass, partial + these -> bf16 gradient.
template <bool LONG>
__device__ __forceinline__ void emit32(const uint32_t (&y)[32], float mul, float* part,
                                       bf16* out) {
  if constexpr (!LONG) {
    float4* dst = reinterpret_cast<float4*>(part);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dst[i] = make_float4(__uint_as_float(y[4 * i]) * mul, __uint_as_float(y[4 * i + 1]) * mul,
                           __uint_as_float(y[4 * i + 2]) * mul, __uint_as_float(y[4 * i + 3]) * mul);
  } else {
    const float4* src = reinterpret_cast<const float4*>(part);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 w = src[i];
      pk[2 * i] = pack_bf16(w.x + __uint_as_float(y[4 * i]) * mul, w.y + __uint_as_float(y[4 * i + 1]) * mul);
      pk[2 * i + 1] =
          pack_bf16(w.z + __uint_as_float(y[4 * i + 2]) * mul, w.w + __uint_as_float(y[4 * i + 3]) * mul);
    }
    uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

// 16-column form of emit32.
template <bool LONG>
__device__ __forceinline__ void emit16(const uint32_t (&y)[16], float mul, float* part, bf16* out) {
  if constexpr (!LONG) {
    float4* dst = reinterpret_cast<float4*>(part);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i] = make_float4(__uint_as_float(y[4 * i]) * mul, __uint_as_float(y[4 * i + 1]) * mul,
                           __uint_as_float(y[4 * i + 2]) * mul, __uint_as_float(y[4 * i + 3]) * mul);
  } else {
    const float4* src = reinterpret_cast<const float4*>(part);
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 w = src[i];
      pk[2 * i] = pack_bf16(w.x + __uint_as_float(y[4 * i]) * mul, w.y + __uint_as_float(y[4 * i + 1]) * mul);
      pk[2 * i + 1] =
          pack_bf16(w.z + __uint_as_float(y[4 * i + 2]) * mul, w.w + __uint_as_float(y[4 * i + 3]) * mul);
    }
    uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
    for (int i = 0; i < 2; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

// Common prologue: TMEM allocation, barrier initialisation.
template <int NST>
__device__ __forceinline__ void init_cta(uint8_t* bar, int warp, uint32_t full_count) {
  using BB = Bars<NST>;
  const uint32_t base = smem_u32(bar);
  if (warp == MMA_WARP) {
    tmem_alloc(base + BB::TMEM_SLOT, TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(base + BB::FULL + 8 * s, full_count);
      mbar_init(base + BB::EMPTY + 8 * s, 1);
    }
    mbar_init(base + BB::SDP, 1);
    mbar_init(base + BB::DS, EW_THREADS);
    mbar_init(base + BB::DQC, 1);
    mbar_init(base + BB::RD, EW_THREADS);
    mbar_init(base + BB::A, EW_THREADS);
    mbar_init(base + BB::FIN, 1);
    mbar_init(base + BB::DRAIN, 1);
    mbar_init(base + BB::KVF, 1);
    mbar_init(base + BB::KVE, 1);
    for (int r = 0; r < NRING; ++r) {
      mbar_init(base + BB::RF + 8 * r, 1);
      mbar_init(base + BB::RE + 8 * r, RING_CONSUMERS);
    }
    *reinterpret_cast<volatile int*>(bar + BB::ABORT) = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// ================================================================ dQ kernel ==
// Per 128-key tile t: the tensor core computes S(t), dP(t); the warps load them
// (and signal "read" at once, so S(t+1), dP(t+1) can overwrite them), form
// dS(t) = P (dP - D) and, once dQ(t-1) has consumed the previous one, store it as
// bf16; then dQ += dS(t) K(t).
template <int D, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
bwd_dq(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
       const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
       const BwdArgs a, const int n_items) {
  constexpr bool LONG = MODE != kWin;
  constexpr bool GROUP = MODE == kGrp;
  using L = DqLayout<D>;
  using BB = Bars<L::NST>;
  constexpr int NST = L::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* bar = sm + L::BAR;
  const uint32_t bb = smem_u32(bar);
  const uint32_t b_full = bb + BB::FULL, b_empty = bb + BB::EMPTY, b_sdp = bb + BB::SDP;
  const uint32_t b_ds = bb + BB::DS, b_rd = bb + BB::RD, b_a = bb + BB::A, b_fin = bb + BB::FIN;
  const uint32_t b_dqc = bb + BB::DQC;
  const uint32_t b_drain = bb + BB::DRAIN, b_qf = bb + BB::KVF, b_qe = bb + BB::KVE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + BB::ABORT);
  uint32_t* kmask = reinterpret_cast<uint32_t*>(sm + L::KM);  // [NST][NK] (group lists)
  init_cta<NST>(bar, warp, GROUP ? 2 : 1);
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(bar + BB::TMEM_SLOT);
  int* status = a.status;
  const long long tlim = a.timeout_cycles;
  const uint32_t b_rf = bb + BB::RF, b_re = bb + BB::RE;
  volatile int* ring_x = reinterpret_cast<volatile int*>(bar + BB::RING_X);

  if (warp == PRODUCER_WARP) {
    // lane 0 waits and issues the copies; with group lists every lane also stages
    // four keys' masks of the tile
    if (lane == 0) {
      tma_prefetch(&mk);
      tma_prefetch(&mv);
      tma_prefetch(&mq);
    }
    int last_par[NST];
    for (int s = 0; s < NST; ++s) last_par[s] = -1;
    int g = 0, qc = 0, q_par = -1;
    bool ok = true;
    for (int kr = 0;; ++kr) {
      int x = 0;
      if (lane == 0) ok = ring_put(b_rf, b_re, ring_x, kr, a.item_counter, x, abort_flag, status, tlim);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      x = __shfl_sync(0xffffffffu, x, 0);
      if (!ok || x >= n_items) break;
      const BItem it = dq_item<LONG>(a, x);
      if (!it.valid || it.n == 0) continue;
      // the item's Q rows, once the previous item's products are done
      if (lane == 0) {
        ok = mbar_wait(b_qe, (uint32_t)((qc & 1) ^ 1), abort_flag, status, tlim);
        if (ok) {
          mbar_expect_tx(b_qf, L::TILE);
          for (int bx = 0; bx < D / 64; ++bx) {
            const uint32_t dst = smem_u32(sm + L::QT + bx * BOX);
            if constexpr (LONG)
              tma_load_2d(dst, &mq, 64 * bx, (it.b * a.H + it.h) * a.NR + it.row0, b_qf);
            else
              tma_load_3d(dst, &mq, 64 * bx, it.h, it.b * a.N + it.row0, b_qf);
          }
          q_par = qc & 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++qc;
      DqWalk wk;
      wk.init(a, it, LONG);
      for (int t = 0; t < it.n; ++t, ++g) {
        int start, cnt;
        bool full;
        wk.next(a, it, LONG, t, start, cnt, full);
        const int slot = g % NST;
        const uint32_t par = (uint32_t)((g / NST) & 1);
        if (lane == 0) ok = mbar_wait(b_empty + 8 * slot, par ^ 1, abort_flag, status, tlim);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t fb = b_full + 8 * slot;
        if (lane == 0) {
          mbar_expect_tx(fb, 2 * L::TILE);
          for (int kv = 0; kv < 2; ++kv)
            for (int bx = 0; bx < D / 64; ++bx) {
              const uint32_t dst = smem_u32(sm + L::RING + (slot * 2 + kv) * L::TILE + bx * BOX);
              const CUtensorMap* m = kv ? &mv : &mk;
              if constexpr (LONG)
                tma_load_2d(dst, m, 64 * bx, (it.b * a.H_kv + it.kvh) * a.NR + start, fb);
              else
                tma_load_3d(dst, m, 64 * bx, it.kvh, it.b * a.N + start, fb);
            }
        }
        if constexpr (GROUP) {  // masks of the tile's keys (0 past its count)
          const uint32_t* PM = a.pmask + (int64_t)it.br * a.NR;
#pragma unroll
          for (int i = 0; i < NK / 32; ++i) {
            const int kc = 32 * i + lane;
            kmask[slot * NK + kc] = kc < cnt ? __ldg(PM + start + kc) : 0u;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(fb);
        }
        last_par[slot] = (int)par;
      }
      if (!ok) break;
    }
    if (lane == 0 && *abort_flag) {
      if (q_par >= 0) mbar_drain(b_qf, (uint32_t)q_par);
      for (int s = 0; s < NST; ++s)
        if (last_par[s] >= 0) mbar_drain(b_full + 8 * s, (uint32_t)last_par[s]);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t ISD = idesc_bf16(128, NK, 0);  // S = Q K^T, dP = dO V^T
      constexpr uint32_t IDQ = idesc_bf16(128, D, 1);   // dQ += dS K (K MN-major)
      const uint32_t q_base = smem_u32(sm + L::QT);
      const uint32_t r_base = smem_u32(sm + L::RING);
      auto kaddr = [&](int g) { return r_base + (g % NST) * 2 * L::TILE; };
      auto ring_wait = [&](int g) {
        return mbar_wait(b_full + 8 * (g % NST), (uint32_t)((g / NST) & 1), abort_flag, status, tlim);
      };
      auto issue_sdp = [&](int g) {
        const uint32_t ka = kaddr(g), va = ka + L::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * BOX + (kk % 4) * 32;
          umma_ss(tmem + L::COL_S, sw128_desc(q_base + off, 16, 1024), sw128_desc(ka + off, 16, 1024), ISD,
                  kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * BOX + (kk % 4) * 32;
          umma_ts(tmem + L::COL_DP, tmem + L::COL_DO + 8 * kk, sw128_desc(va + off, 16, 1024), ISD, kk > 0);
        }
        umma_commit(b_sdp);
      };
      int g = 0, ac = 0, qc = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        int x = 0;
        if (!(ok = ring_get(b_rf, b_re, ring_x, kr, x, abort_flag, status, tlim)) || x >= n_items) break;
        const BItem it = dq_item<LONG>(a, x);
        if (!it.valid || it.n == 0) continue;
        // Q landed; the warps staged dO (and read the previous item's dQ)
        if (!(ok = mbar_wait(b_qf, (uint32_t)(qc & 1), abort_flag, status, tlim) &&
                   mbar_wait(b_a, (uint32_t)(ac & 1), abort_flag, status, tlim) && ring_wait(g)))
          break;
        ++qc;
        ++ac;
        tc_fence_after();
        issue_sdp(g);
        for (int t = 0; t < it.n; ++t) {
          const int gc = g + t;
          // S(gc), dP(gc) are in registers: the next tile's products may overwrite them
          if (!(ok = mbar_wait(b_rd, (uint32_t)(gc & 1), abort_flag, status, tlim))) break;
          if (t + 1 < it.n) {
            if (!(ok = ring_wait(gc + 1))) break;
            tc_fence_after();
            issue_sdp(gc + 1);
          }
          if (!(ok = mbar_wait(b_ds, (uint32_t)(gc & 1), abort_flag, status, tlim))) break;
          tc_fence_after();
          const uint32_t ka = kaddr(gc);
#pragma unroll
          for (int kk = 0; kk < NK / 16; ++kk)
            umma_ts(tmem + L::COL_DQ, tmem + L::COL_DS + 8 * kk, sw128_desc(ka + kk * 2048, BOX, 1024), IDQ,
                    (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(b_empty + 8 * (gc % NST));
          umma_commit(b_dqc);
        }
        if (!ok) break;
        umma_commit(b_fin);
        umma_commit(b_qe);
        g += it.n;
      }
      umma_commit(b_drain);
      mbar_drain(b_drain, 0);
    }
    __syncwarp();
  } else if (warp < EW_WARPS) {
    // ---------------------------------------------------------- elementwise --
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tl = tmem + lane_off;
    const float sl2 = a.sl2;
    int g = 0, ac = 0;
    bool ok = true;
    for (int kr = 0;; ++kr) {
      int x = 0;
      if (!(ok = ring_get_warp(b_rf, b_re, ring_x, kr, x, abort_flag, status, tlim)) || x >= n_items) break;
      const BItem it = dq_item<LONG>(a, x);
      if (!it.valid) continue;
      const bool row_ok = r < it.rows;
      const int rr = min(r, it.rows - 1);
      const int* P = LONG ? a.perm + (int64_t)it.br * a.NR : nullptr;
      const int qp = LONG ? __ldg(P + it.row0 + rr) : it.row0 + rr;
      const int64_t grow = ((int64_t)it.b * a.N + qp) * a.H + it.h;  // [B, N, H] row
      if (it.n > 0) {
        // the previous item's dQ has been read and its products are done: stage dO
        if (wg == 0) {
          stage_row<D>(tl + L::COL_DO, row_ok ? a.dout + grow * D : nullptr);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(b_a);
        ++ac;
      }
      const int64_t li = ((int64_t)it.b * a.H + it.h) * a.N + qp;
      const float lse2 = __ldg(a.lse + li) * kLog2e;
      const float Dr = __ldg(a.dvec + li);
      // group lists: the row's groups below list g (keys sharing one of them are
      // counted in a lower list) and its slot
      uint32_t m_low = 0u;
      if constexpr (GROUP)
        m_low = __ldg(a.pmask + (int64_t)it.br * a.NR + it.row0 + rr) & ((1u << it.seg) - 1u);
      const bool dedup = GROUP && __any_sync(0xffffffffu, m_low != 0u);
      DqWalk wk;
      wk.init(a, it, LONG);
      for (int t = 0; t < it.n; ++t) {
        const int gc = g + t;
        int start, cnt;
        bool full;
        wk.next(a, it, LONG, t, start, cnt, full);
        // every (row, key) pair of the tile allowed?  (uniform over the CTA; rows past
        // the block are never stored, so they need no mask)
        bool need_mask;
        int c_lo = 0, c_hi = cnt;
        if constexpr (LONG) {
          need_mask = !(full && cnt == NK);
          if (need_mask && !full) c_hi = upper_bound_g(P + start, 0, cnt, qp - a.w);
        } else {
          need_mask = !(cnt == NK && start + NK - 1 <= it.row0 && it.row0 + BM - 1 - start < a.w);
          c_lo = max(0, qp - a.w + 1 - start);
          c_hi = min(cnt, qp - start + 1);
        }
        const uint32_t width = (uint32_t)max(c_hi - c_lo, 0);
        ok = mbar_wait(b_sdp, (uint32_t)(gc & 1), abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[2][16], dpv[2][16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld16(tl + L::COL_S + 32 * wg + 16 * hh, sv[hh]);
          tmem_ld16(tl + L::COL_DP + 32 * wg + 16 * hh, dpv[hh]);
        }
        tmem_ld_wait(sv[0]);
        tie16(sv[1]);
        tie16(dpv[0]);
        tie16(dpv[1]);
        tc_fence_before();
        mbar_arrive(b_rd);
        // dS of keys 2i, 2i + 1 of the tile goes to column i of the dS region
        const uint32_t dsc = tl + L::COL_DS + 16 * wg;
        const uint32_t* km = kmask + (gc % NST) * NK;
        if (GROUP && dedup) {  // the tile's key masks (staged with its K and V)
          ok = mbar_wait(b_full + 8 * (gc % NST), (uint32_t)((gc / NST) & 1), abort_flag, status, tlim);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        uint32_t pkv[2][8];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = 32 * wg + 16 * hh;  // first key column of this half
          const uint32_t(&s)[16] = sv[hh];
          const uint32_t(&dp)[16] = dpv[hh];
          uint32_t(&pk)[8] = pkv[hh];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float y0, y1, t0, t1, d0, d1;
            ffma2(y0, y1, __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]), sl2, sl2, -lse2, -lse2);
            float p0 = ex2(y0), p1 = ex2(y1);
            if (need_mask) {
              if ((uint32_t)(c + 2 * i - c_lo) >= width) p0 = 0.0f;
              if ((uint32_t)(c + 2 * i + 1 - c_lo) >= width) p1 = 0.0f;
            }
            if (GROUP && dedup) {
              if (m_low & km[c + 2 * i]) p0 = 0.0f;
              if (m_low & km[c + 2 * i + 1]) p1 = 0.0f;
            }
            fadd2(t0, t1, __uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1]), -Dr, -Dr);
            fmul2(d0, d1, p0, p1, t0, t1);
            pk[i] = pack_bf16(d0, d1);
          }
        }
        if (gc > 0) {  // dQ(gc - 1) has read the previous dS
          ok = mbar_wait(b_dqc, (uint32_t)((gc - 1) & 1), abort_flag, status, tlim);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st8(dsc, pkv[0]);
        tmem_st8(dsc + 8, pkv[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds);
      }
      if (!ok) break;
      // ---- epilogue: dQ = scale * (dS K), window partial or final ----
      if (it.n > 0) {
        ok = mbar_wait(b_fin, (uint32_t)((ac - 1) & 1), abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      g += it.n;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = wg * (D / 4) + 16 * c;
        uint32_t y[16];
        if (it.n > 0) {
          tmem_ld16(tl + L::COL_DQ + col, y);
          tmem_ld_wait(y);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = 0u;
        }
        if constexpr (GROUP) {  // list part into the row's slot
          if (row_ok)
            emit16<false>(y, a.scale, a.dq_s + (int64_t)__popc(m_low) * a.B * a.N * a.H * D + grow * D + col,
                          nullptr);
        } else if (row_ok) {
          emit16<LONG>(y, a.scale, a.dq_w + grow * D + col, a.dq + grow * D + col);
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ============================================================= dK/dV kernel ==
template <int D, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
bwd_dkdv(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
         const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
         const BwdArgs a, const int n_items) {
  constexpr bool LONG = MODE != kWin;
  constexpr bool GROUP = MODE == kGrp;
  using L = DkvLayout<D>;
  using BB = Bars<L::NST>;
  constexpr int NST = L::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* bar = sm + L::BAR;
  const uint32_t bb = smem_u32(bar);
  const uint32_t b_full = bb + BB::FULL, b_empty = bb + BB::EMPTY, b_sdp = bb + BB::SDP;
  const uint32_t b_ds = bb + BB::DS, b_a = bb + BB::A, b_fin = bb + BB::FIN, b_drain = bb + BB::DRAIN;
  const uint32_t b_kvf = bb + BB::KVF, b_kve = bb + BB::KVE;
  const uint32_t b_ds0 = bb + BB::RD;  // first half of dS^T / P^T written (RD is the dQ kernel's)
  const uint32_t b_rf = bb + BB::RF, b_re = bb + BB::RE;
  volatile int* ring_x = reinterpret_cast<volatile int*>(bar + BB::RING_X);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + BB::ABORT);
  float* scal = reinterpret_cast<float*>(sm + L::SCAL);  // [NST][4][NQ]
  init_cta<NST>(bar, warp, 2);
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(bar + BB::TMEM_SLOT);
  int* status = a.status;
  const long long tlim = a.timeout_cycles;

  if (warp == PRODUCER_WARP) {
    // whole warp: lane 0 issues the copies, every lane stages four queries' scalars
    if (lane == 0) {
      tma_prefetch(&mk);
      tma_prefetch(&mv);
      tma_prefetch(&mq);
      tma_prefetch(&mdo);
    }
    int last_par[NST];
    for (int s = 0; s < NST; ++s) last_par[s] = -1;
    int g = 0, kc = 0, kv_par = -1;
    bool ok = true;
    for (int kr = 0;; ++kr) {
      int x = 0;
      if (lane == 0) ok = ring_put(b_rf, b_re, ring_x, kr, a.item_counter, x, abort_flag, status, tlim);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      x = __shfl_sync(0xffffffffu, x, 0);
      if (!ok || x >= n_items) break;
      const BItem it = dkv_item<LONG>(a, x);
      if (!it.valid || it.n == 0) continue;
      // the item's K and V rows, once the previous item's products are done
      if (lane == 0) {
        ok = mbar_wait(b_kve, (uint32_t)((kc & 1) ^ 1), abort_flag, status, tlim);
        if (ok) {
          mbar_expect_tx(b_kvf, 2 * L::TILE);
          for (int kv = 0; kv < 2; ++kv)
            for (int bx = 0; bx < D / 64; ++bx) {
              const uint32_t dst = smem_u32(sm + L::KV + kv * L::TILE + bx * BOX);
              const CUtensorMap* m = kv ? &mv : &mk;
              if constexpr (LONG)
                tma_load_2d(dst, m, 64 * bx, (it.b * a.H_kv + it.kvh) * a.NR + it.row0, b_kvf);
              else
                tma_load_3d(dst, m, 64 * bx, it.kvh, it.b * a.N + it.row0, b_kvf);
            }
          kv_par = kc & 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++kc;
      DkvWalk wk;
      wk.init(a, it, LONG);
      const int* P = LONG ? a.perm + (int64_t)it.br * a.NR : nullptr;
      for (int t = 0; t < it.n; ++t, ++g) {
        int h, start, cnt;
        wk.next(a, it, LONG, t, h, start, cnt);
        const int slot = g % NST;
        const uint32_t par = (uint32_t)((g / NST) & 1);
        if (lane == 0) ok = mbar_wait(b_empty + 8 * slot, par ^ 1, abort_flag, status, tlim);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t fb = b_full + 8 * slot;
        if (lane == 0) {
          mbar_expect_tx(fb, 2 * L::TILE);
          for (int kv = 0; kv < 2; ++kv)
            for (int bx = 0; bx < D / 64; ++bx) {
              const uint32_t dst = smem_u32(sm + L::RING + (slot * 2 + kv) * L::TILE + bx * BOX);
              const CUtensorMap* m = kv ? &mdo : &mq;
              if constexpr (LONG)
                tma_load_2d(dst, m, 64 * bx, (it.b * a.H + h) * a.NR + start, fb);
              else
                tma_load_3d(dst, m, 64 * bx, h, it.b * a.N + start, fb);
            }
        }
        // query scalars: LSE * log2(e) (+inf marks "no query"), D, position and,
        // with group lists, the query's mask
        float* sc = scal + slot * 4 * NQ;
#pragma unroll
        for (int i = 0; i < NQ / 32; ++i) {
          const int qc = 32 * i + lane;
          float lse2 = INFINITY, dd = 0.0f;
          int pos = 0;
          uint32_t qm = 0u;
          if (qc < cnt) {
            pos = LONG ? __ldg(P + start + qc) : start + qc;
            const int64_t li = ((int64_t)it.b * a.H + h) * a.N + pos;
            lse2 = __ldg(a.lse + li) * kLog2e;
            dd = __ldg(a.dvec + li);
            if constexpr (GROUP) qm = __ldg(a.pmask + (int64_t)it.br * a.NR + start + qc);
          }
          sc[qc] = lse2;
          sc[NQ + qc] = dd;
          reinterpret_cast<int*>(sc)[2 * NQ + qc] = pos;
          reinterpret_cast<uint32_t*>(sc)[3 * NQ + qc] = qm;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(fb);
        last_par[slot] = (int)par;
      }
      if (!ok) break;
    }
    if (lane == 0 && *abort_flag) {
      if (kv_par >= 0) mbar_drain(b_kvf, (uint32_t)kv_par);
      for (int s = 0; s < NST; ++s)
        if (last_par[s] >= 0) mbar_drain(b_full + 8 * s, (uint32_t)last_par[s]);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t IST = idesc_bf16(128, NQ, 0);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t IKV = idesc_bf16(128, D, 1);   // dV += P^T dO, dK += dS^T Q
      const uint32_t k_base = smem_u32(sm + L::KV), v_base = k_base + L::TILE;
      const uint32_t r_base = smem_u32(sm + L::RING);
      auto qaddr = [&](int g) { return r_base + (g % NST) * 2 * L::TILE; };
      auto ring_wait = [&](int g) {
        return mbar_wait(b_full + 8 * (g % NST), (uint32_t)((g / NST) & 1), abort_flag, status, tlim);
      };
      auto issue_st = [&](int g) {
        const uint32_t qa = qaddr(g), da = qa + L::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * BOX + (kk % 4) * 32;
          umma_ss(tmem + L::COL_ST, sw128_desc(k_base + off, 16, 1024), sw128_desc(qa + off, 16, 1024),
                  IST, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * BOX + (kk % 4) * 32;
          umma_ss(tmem + L::COL_DPT, sw128_desc(v_base + off, 16, 1024), sw128_desc(da + off, 16, 1024),
                  IST, kk > 0);
        }
        umma_commit(b_sdp);
      };
      int g = 0, ac = 0, kc = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        int x = 0;
        if (!(ok = ring_get(b_rf, b_re, ring_x, kr, x, abort_flag, status, tlim)) || x >= n_items) break;
        const BItem it = dkv_item<LONG>(a, x);
        if (!it.valid || it.n == 0) continue;
        if (!(ok = mbar_wait(b_kvf, (uint32_t)(kc & 1), abort_flag, status, tlim) && ring_wait(g))) break;
        ++kc;
        tc_fence_after();
        issue_st(g);
        // the previous item's epilogue has read dK and dV before they restart
        if (!(ok = mbar_wait(b_a, (uint32_t)(ac & 1), abort_flag, status, tlim))) break;
        ++ac;
        for (int t = 0; t < it.n; ++t) {
          const int gc = g + t;
          const uint32_t qa = qaddr(gc), da = qa + L::TILE;
          // P^T (dS^T) of queries 32w + 16h + 2i, +1 sits in column 32w + 8h + i.  The
          // elementwise warps hand over the first 16 queries of each warpgroup (h = 0,
          // barrier DS0) before the second (h = 1, barrier DS), so the products of the
          // first half run while the second half is computed.
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (!(ok = mbar_wait(hh ? b_ds : b_ds0, (uint32_t)(gc & 1), abort_flag, status, tlim))) break;
            tc_fence_after();
#pragma unroll
            for (int w4 = 0; w4 < NQ / 32; ++w4) {
              const int kk = 2 * w4 + hh;
              const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
              const uint32_t col = 32 * w4 + 8 * hh;
              umma_ts(tmem + L::COL_DV, tmem + L::COL_ST + col, sw128_desc(da + kk * 2048, BOX, 1024), IKV,
                      acc);
              umma_ts(tmem + L::COL_DK, tmem + L::COL_DPT + col, sw128_desc(qa + kk * 2048, BOX, 1024), IKV,
                      acc);
            }
          }
          if (!ok) break;
          umma_commit(b_empty + 8 * (gc % NST));
          if (t + 1 < it.n) {
            if (!(ok = ring_wait(gc + 1))) break;
            tc_fence_after();
            issue_st(gc + 1);
          }
        }
        if (!ok) break;
        umma_commit(b_fin);
        umma_commit(b_kve);
        g += it.n;
      }
      umma_commit(b_drain);
      mbar_drain(b_drain, 0);
    }
    __syncwarp();
  } else if (warp < EW_WARPS) {
    // ---------------------------------------------------------- elementwise --
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tl = tmem + lane_off;
    const float sl2 = a.sl2;
    const int w = a.w;
    int g = 0, ac = 0;
    bool ok = true;
    for (int kr = 0;; ++kr) {
      int x = 0;
      if (!(ok = ring_get_warp(b_rf, b_re, ring_x, kr, x, abort_flag, status, tlim)) || x >= n_items) break;
      const BItem it = dkv_item<LONG>(a, x);
      if (!it.valid) continue;
      const bool row_ok = r < it.rows;
      const int rr = min(r, it.rows - 1);
      const int pj = LONG ? __ldg(a.perm + (int64_t)it.br * a.NR + it.row0 + rr) : it.row0 + rr;
      const int64_t grow = ((int64_t)it.b * a.N + pj) * a.H_kv + it.kvh;  // [B, N, H_kv] row
      // last key position of the block (keys ascend in it)
      const int p_hi = LONG ? __ldg(a.perm + (int64_t)it.br * a.NR + it.row0 + it.rows - 1)
                            : it.row0 + it.rows - 1;
      // group lists: the key's groups below list g (queries sharing one of them count
      // it in a lower list) and its slot
      uint32_t m_low = 0u;
      if constexpr (GROUP)
        m_low = __ldg(a.pmask + (int64_t)it.br * a.NR + it.row0 + rr) & ((1u << it.seg) - 1u);
      const bool dedup = GROUP && __any_sync(0xffffffffu, m_low != 0u);
      if (it.n > 0) {
        tc_fence_before();
        mbar_arrive(b_a);  // the previous item's dK, dV have been read
        ++ac;
      }
      for (int t = 0; t < it.n; ++t) {
        const int gc = g + t, slot = gc % NST;
        ok = mbar_wait(b_full + 8 * slot, (uint32_t)((gc / NST) & 1), abort_flag, status, tlim) &&
             mbar_wait(b_sdp, (uint32_t)(gc & 1), abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* sc = scal + slot * 4 * NQ;
        // every (key, query) pair of the tile allowed?  Queries past the tile's count
        // carry LSE = +inf (P = 0) and keys past the block are never stored, so only
        // the position rule needs a mask: long range, the first (lowest) query
        // position against the last key; window, both window edges.
        const int q_first = reinterpret_cast<const int*>(sc)[2 * NQ];
        const bool need_mask =
            LONG ? q_first < p_hi + w : !(q_first >= it.row0 + BM - 1 && q_first + NQ - 1 - it.row0 < w);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = 32 * wg + 16 * hh;  // first query column of this half
          uint32_t st[16], dpt[16];
          tmem_ld16(tl + L::COL_ST + c, st);
          tmem_ld16(tl + L::COL_DPT + c, dpt);
          tmem_ld_wait(st);
          tie16(dpt);
          uint32_t pp[8], pd[8];
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(sc + c + i);
            const float4 d4 = *reinterpret_cast<const float4*>(sc + NQ + c + i);
            const float ls[4] = {l4.x, l4.y, l4.z, l4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
            float pv[4], dv4[4], y[4], tt[4];
            ffma2(y[0], y[1], __uint_as_float(st[i]), __uint_as_float(st[i + 1]), sl2, sl2, -ls[0], -ls[1]);
            ffma2(y[2], y[3], __uint_as_float(st[i + 2]), __uint_as_float(st[i + 3]), sl2, sl2, -ls[2], -ls[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = ex2(y[e]);
            if (need_mask) {
              const int4 q4 = *reinterpret_cast<const int4*>(reinterpret_cast<const int*>(sc) + 2 * NQ + c + i);
              const int pq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int dpos = pq[e] - pj;
                if (!(LONG ? dpos >= w : (uint32_t)dpos < (uint32_t)w)) pv[e] = 0.0f;
              }
            }
            if (GROUP && dedup) {
              const uint4 m4 = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(sc) + 3 * NQ + c + i);
              if (m_low & m4.x) pv[0] = 0.0f;
              if (m_low & m4.y) pv[1] = 0.0f;
              if (m_low & m4.z) pv[2] = 0.0f;
              if (m_low & m4.w) pv[3] = 0.0f;
            }
            fadd2(tt[0], tt[1], __uint_as_float(dpt[i]), __uint_as_float(dpt[i + 1]), -dd[0], -dd[1]);
            fadd2(tt[2], tt[3], __uint_as_float(dpt[i + 2]), __uint_as_float(dpt[i + 3]), -dd[2], -dd[3]);
            fmul2(dv4[0], dv4[1], pv[0], pv[1], tt[0], tt[1]);
            fmul2(dv4[2], dv4[3], pv[2], pv[3], tt[2], tt[3]);
            pp[i / 2] = pack_bf16(pv[0], pv[1]);
            pp[i / 2 + 1] = pack_bf16(pv[2], pv[3]);
            pd[i / 2] = pack_bf16(dv4[0], dv4[1]);
            pd[i / 2 + 1] = pack_bf16(dv4[2], dv4[3]);
          }
          tmem_st8(tl + L::COL_ST + 32 * wg + 8 * hh, pp);   // over columns already read
          tmem_st8(tl + L::COL_DPT + 32 * wg + 8 * hh, pd);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(hh ? b_ds : b_ds0);
        }
      }
      if (!ok) break;
      // ---- epilogue: dK = scale * (dS^T Q) (warpgroups 0, 1), dV = P^T dO (2, 3) ----
      if (it.n > 0) {
        ok = mbar_wait(b_fin, (uint32_t)((ac - 1) & 1), abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      g += it.n;
      const bool is_k = wg < 2;
      const int half = (wg & 1) * (D / 2);  // this warpgroup's half of the columns
      const int col_acc = (is_k ? L::COL_DK : L::COL_DV) + half;
      const float mul = is_k ? a.scale : 1.0f;
      float* part = (is_k ? a.dk_w : a.dv_w) + grow * D + half;
      bf16* out = (is_k ? a.dk : a.dv) + grow * D + half;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t y[32];
        if (it.n > 0) {
          tmem_ld32(tl + col_acc + 32 * c, y);
          tmem_ld_wait(y);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = 0u;
        }
        if constexpr (GROUP) {  // list part into the key's slot
          if (row_ok) {
            float* sl = (is_k ? a.dk_s : a.dv_s) + (int64_t)__popc(m_low) * a.B * a.N * a.H_kv * D +
                        grow * D + half;
            emit32<false>(y, mul, sl + 32 * c, nullptr);
          }
        } else if (row_ok) {
          emit32<LONG>(y, mul, part + 32 * c, out + 32 * c);
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------- preparation kernels --
// D[b, h, i] = dO[b, i, h, :] . O[b, i, h, :] (fp32 sums of bf16 products); one
// thread per (b, i, h).
template <int D>
__global__ void __launch_bounds__(256)
bwd_rowdot(int64_t rows, int N, int H, const uint4* __restrict__ o, const uint4* __restrict__ d_o,
           float* __restrict__ dvec) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= rows) return;
  const uint4* a = o + x * (D / 8);
  const uint4* b = d_o + x * (D / 8);
  float acc = 0.0f;
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 va = __ldg(a + c), vb = __ldg(b + c);
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[i]));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[i]));
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
  const int h = (int)(x % H);
  const int64_t bn = x / H;
  dvec[((bn / N) * H + h) * N + bn % N] = acc;
}

// Permuted, head-major copy of dO: dOp[b][h][n'][:] = dO[b][perm[n']][h][:] for the
// heads of routing head rho.  One CTA per permuted row.
__global__ void __launch_bounds__(256)
permute_rows(int N, int NR, int H, int R, int d, const int* __restrict__ perm,
             const uint4* __restrict__ src, uint4* __restrict__ dst) {
  const int64_t row = blockIdx.x;  // (b * R + rho) * NR + n'
  const int br = (int)(row / NR), np = (int)(row % NR);
  const int b = br / R, rho = br % R;
  const int n = perm[row];
  const int hq = H / R, vec = d / 8;
  for (int i = threadIdx.x; i < hq * vec; i += blockDim.x) {
    const int hh = rho * hq + i / vec, c = i % vec;
    dst[(((int64_t)b * H + hh) * NR + np) * vec + c] = src[(((int64_t)b * N + n) * H + hh) * vec + c];
  }
}

// Group lists, last step: gradient = window part + the top_k list parts, in bf16.
// One thread per four values of a row.
__global__ void __launch_bounds__(256)
bwd_sum_slots(int64_t n4, int top_k, const float4* __restrict__ win, const float4* __restrict__ slots,
              uint2* __restrict__ out) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n4) return;
  float4 acc = __ldg(win + x);
  for (int s = 0; s < top_k; ++s) {
    const float4 v = __ldg(slots + s * n4 + x);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  uint2 o;
  o.x = pack_bf16(acc.x, acc.y);
  o.y = pack_bf16(acc.z, acc.w);
  out[x] = o;
}

// ------------------------------------------------------------- host side --
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// Tensor map over rows of D bf16 values, box 64 columns x box_rows rows (x 1 head
// when heads > 0: 3-D d, head, token), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int64_t rows, int heads, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r;
  if (heads > 0) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;
  return n;
}

template <typename Kernel, typename... Maps>
cudaError_t launch_persistent(Kernel kernel, int smem, const BwdArgs& a, int n_items, cudaStream_t s,
                              const Maps&... maps) {
  smem = smem < kMinSmem ? kMinSmem : smem;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  const int grid = n_items < sms ? n_items : sms;
  if (grid < 1) return cudaSuccess;
  kernel<<<grid, NTHREADS, smem, s>>>(maps..., a, n_items);
  return cudaGetLastError();
}

template <int D, int MODE>
cudaError_t launch_mode(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                        const CUtensorMap& mdo, const BwdArgs& a, int nq_items, int nk_items,
                        bool dq_kernel, cudaStream_t s) {
  return dq_kernel
             ? launch_persistent(bwd_dq<D, MODE>, DqLayout<D>::SMEM, a, nq_items, s, mk, mv, mq, mdo)
             : launch_persistent(bwd_dkdv<D, MODE>, DkvLayout<D>::SMEM, a, nk_items, s, mk, mv, mq, mdo);
}

template <int D>
cudaError_t launch_pass(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                        const CUtensorMap& mdo, const BwdArgs& a, int nq_items, int nk_items,
                        bool long_pass, bool group, bool dq_kernel, cudaStream_t s) {
  if (!long_pass) return launch_mode<D, kWin>(mk, mv, mq, mdo, a, nq_items, nk_items, dq_kernel, s);
  if (group) return launch_mode<D, kGrp>(mk, mv, mq, mdo, a, nq_items, nk_items, dq_kernel, s);
  return launch_mode<D, kSeg>(mk, mv, mq, mdo, a, nq_items, nk_items, dq_kernel, s);
}

}  // namespace

cudaError_t launch_bwd_rowdot(const focus_params& p, const bf16* o, const bf16* d_o, float* dvec,
                              cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.N * p.H;
  const unsigned grid = (unsigned)((rows + 255) / 256);
  if (p.d_head == 64)
    bwd_rowdot<64><<<grid, 256, 0, s>>>(rows, p.N, p.H, reinterpret_cast<const uint4*>(o),
                                        reinterpret_cast<const uint4*>(d_o), dvec);
  else
    bwd_rowdot<128><<<grid, 256, 0, s>>>(rows, p.N, p.H, reinterpret_cast<const uint4*>(o),
                                         reinterpret_cast<const uint4*>(d_o), dvec);
  return cudaGetLastError();
}

cudaError_t launch_permute_rows(const focus_params& p, const WsLayout& L, const bf16* src, bf16* dst,
                                const char* ws, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.R * L.NR;
  permute_rows<<<(unsigned)rows, 256, 0, s>>>(p.N, L.NR, p.H, p.R, p.d_head,
                                              reinterpret_cast<const int*>(ws + L.perm),
                                              reinterpret_cast<const uint4*>(src),
                                              reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const focus_params& p, const BwdPlan& bp, const bf16* q, const bf16* k,
                            const bf16* v, const bf16* d_o, const float* lse, bf16* dq, bf16* dk,
                            bf16* dv, char* ws, float scale, bool long_pass, bool dq_kernel,
                            cudaStream_t s) {
  const WsLayout& L = bp.L;
  BwdArgs a{};
  a.B = p.B;
  a.N = p.N;
  a.H = p.H;
  a.H_kv = p.H_kv;
  a.R = p.R;
  a.w = p.w;
  a.nseg = L.nseg;
  a.qtab_cap = L.qtab_cap;
  a.NR = L.NR;
  a.sl2 = scale * kLog2e;
  a.scale = scale;
  a.perm = reinterpret_cast<const int*>(ws + L.perm);
  a.qtab = reinterpret_cast<const QBlock*>(ws + L.qtab);
  a.qtab_count = &reinterpret_cast<const WsHeader*>(ws)->qtab_count;
  a.qhead = reinterpret_cast<const PlanHead*>(ws + bp.qhead);
  a.qent = reinterpret_cast<const PlanEnt*>(ws + bp.qent);
  a.rhead = reinterpret_cast<const PlanHead*>(ws + bp.rhead);
  a.rent = reinterpret_cast<const PlanEnt*>(ws + bp.rent);
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = d_o;
  a.lse = lse;
  a.dvec = reinterpret_cast<const float*>(ws + bp.dvec);
  a.dq_w = reinterpret_cast<float*>(ws + bp.dqw);
  a.dk_w = reinterpret_cast<float*>(ws + bp.dkw);
  a.dv_w = reinterpret_cast<float*>(ws + bp.dvw);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.pmask = reinterpret_cast<const uint32_t*>(ws + L.pmask);
  a.dq_s = reinterpret_cast<float*>(ws + bp.dqs);
  a.dk_s = reinterpret_cast<float*>(ws + bp.dks);
  a.dv_s = reinterpret_cast<float*>(ws + bp.dvs);
  a.status = &reinterpret_cast<WsHeader*>(ws)->status;
  // one counter per launch of the call: window dQ, window dK/dV, long dQ, long dK/dV
  a.item_counter = &reinterpret_cast<WsHeader*>(ws)->item_counter[(long_pass ? 2 : 0) + (dq_kernel ? 0 : 1)];
  a.timeout_cycles = kTimeoutCycles;
  const int D = p.d_head;
  CUtensorMap mk, mv, mq, mdo;
  int nq_items, nk_items;
  if (!long_pass) {
    // window: token-order maps over K, V, Q, dO
    if (!make_map(&mk, k, D, (int64_t)p.B * p.N, p.H_kv, NK) ||
        !make_map(&mv, v, D, (int64_t)p.B * p.N, p.H_kv, NK) ||
        !make_map(&mq, q, D, (int64_t)p.B * p.N, p.H, NQ) ||
        !make_map(&mdo, d_o, D, (int64_t)p.B * p.N, p.H, NQ))
      return cudaErrorInvalidValue;
    const int nb = (p.N + BM - 1) / BM;
    nq_items = p.B * p.H * nb;
    nk_items = p.B * p.H_kv * nb;
  } else {
    // long range: maps over the permuted head-major copies
    if (!make_map(&mk, ws + L.kp, D, (int64_t)p.B * p.H_kv * L.NR, 0, NK) ||
        !make_map(&mv, ws + L.vp, D, (int64_t)p.B * p.H_kv * L.NR, 0, NK) ||
        !make_map(&mq, ws + L.qp, D, (int64_t)p.B * p.H * L.NR, 0, NQ) ||
        !make_map(&mdo, ws + bp.dop, D, (int64_t)p.B * p.H * L.NR, 0, NQ))
      return cudaErrorInvalidValue;
    nq_items = L.qtab_cap * (p.H / p.R);
    nk_items = L.qtab_cap * (p.H_kv / p.R);
  }
  const bool group = L.group != 0;
  return D == 64 ? launch_pass<64>(mk, mv, mq, mdo, a, nq_items, nk_items, long_pass, group, dq_kernel, s)
                 : launch_pass<128>(mk, mv, mq, mdo, a, nq_items, nk_items, long_pass, group, dq_kernel, s);
}

cudaError_t launch_bwd_merge_slots(const focus_params& p, const BwdPlan& bp, const char* ws, bf16* dq,
                                   bf16* dk, bf16* dv, cudaStream_t s) {
  const int64_t nq4 = (int64_t)p.B * p.N * p.H * p.d_head / 4;
  const int64_t nk4 = (int64_t)p.B * p.N * p.H_kv * p.d_head / 4;
  auto run = [&](int64_t n4, size_t win, size_t slots, bf16* out) {
    bwd_sum_slots<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(
        n4, p.top_k, reinterpret_cast<const float4*>(ws + win), reinterpret_cast<const float4*>(ws + slots),
        reinterpret_cast<uint2*>(out));
    return cudaGetLastError();
  };
  cudaError_t e;
  if ((e = run(nq4, bp.dqw, bp.dqs, dq))) return e;
  if ((e = run(nk4, bp.dkw, bp.dks, dk))) return e;
  return run(nk4, bp.dvw, bp.dvs, dv);
}

}  // namespace focus
