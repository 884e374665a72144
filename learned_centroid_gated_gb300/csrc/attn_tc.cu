// Focus attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// "Why Attend to Everything? Focus is the Key", gist.science technical summary,
// section 2 "Core Architecture": a local window of w tokens attends with exact
// softmax, distant tokens only within a shared group ("Inference Efficiency
// (Top-k)": at least one shared group); jindou-blog deep read, method bullets:
// exact softmax inside the groups too.  The two key sets are disjoint
// (long-range keys have i - j >= w, window keys i - j < w), so the union
// softmax is the log-sum-exp merge of two partial softmaxes; every key is
// visited once because tokens are bucketed by their exact group set.
//
// Persistent kernel: one CTA per SM; the producer warp takes the next work item
// (query block of 256 rows of one head) from a global counter and hands it to the
// MMA issuer and the softmax warps through a small shared-memory ring, so the CTAs
// share the items dynamically in the schedule's order (heaviest first within a head):
// a static round-robin share left the average SM idle ~10% of the launch while the
// most loaded one finished.  Each item is two 128-row query tiles A and B that
// ping-pong on the tensor core:
//   warp 8      TMA producer: Q tiles of each item, then K and V tiles through a
//               4-slot ring; runs ahead across item boundaries
//   warp 9      MMA issuer (one thread): S = Q K^T into TMEM, O += P V into TMEM
//   warps 0-3   softmax of tile A (thread = row = TMEM lane), warps 4-7 of tile B;
//               each warpgroup also writes its tile's output rows
//   warps 10-11 idle (they complete the third warpgroup for the register split)
// TMEM (512 columns): S_A | S_B | O_A | O_B.  P (bf16) is written over the first
// 64 columns of its S tile once S is in registers and is the TMEM A operand of
// O += P V, so neither P nor its reads touch shared memory (the S and PV operand
// traffic through shared memory is what bounds this kernel).  Issue order on the tensor
// core: S_A(0) S_B(0) | PV_A(t) S_A(t+1) PV_B(t) S_B(t+1) | ..., so the softmax of
// one tile runs while the tensor core works on the other.  The running max is
// rescaled lazily (only when it grows by more than 2^8), in place in TMEM.
// Barrier phases run on across items; a tile's P barrier also orders the previous
// item's reads of O before the next item's first P V.
//
//   attn_tc<D, kWin>   window part (runs first), token order, keys (i - w, i];
//                      writes the normalised partial O_w (fp32) and LSE_w.
//   attn_tc<D, kSeg>   long-range part: query block of one segment x the key
//                      tiles of every compatible segment (permuted copies),
//                      keys with pos_j <= pos_i - w; merges with (O_w, LSE_w)
//                      and writes O (bf16) and LSE.  Long items run ~100 key
//                      tiles, so the merge's loads cost little there.
//   attn_tc<D, kGrp>   long-range part over group lists: query block of list g x
//                      the keys of list g with pos_j <= pos_i - w, a key counted
//                      only when g is the lowest group it shares with the query
//                      (mask_i & mask_j & (2^g - 1) == 0).  The four warps of a
//                      softmax warpgroup turn the tile's key masks into one
//                      128-bit column set per group bit (warp ballots, shared
//                      memory), and each row ORs the sets of its groups below g.
//                      Writes the normalised part of list g into the token's slot
//                      popc(mask_i & (2^g - 1)); a separate pass merges the slots.
#include <math.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace focus {
namespace {

using namespace ptx;

constexpr int QT = 128;        // rows per query tile (MMA M)
constexpr int BMQ = 2 * QT;    // query rows per work item
constexpr int BNK = kKeyTile;  // keys per tile (MMA N of S, K of P V)
constexpr int NSTAGE = 4;      // K/V ring slots
constexpr int NRING = 4;       // work items handed from the producer to the other roles
constexpr int RING_CONSUMERS = 9;  // MMA issuer + the 8 softmax warps
constexpr int NTHREADS = 384;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kSumCap = 1.8446744e19f;  // 2^64: a tile's exponentials above this retake the max
// Register split after launch (384 threads x 168): warpgroup 2 (producer, MMA,
// idle) drops to 104, the two softmax warpgroups rise to 192:
// 128 * 104 + 256 * 192 = 62464 <= 384 * 168 = 64512.
constexpr int kRegsLow = 104;
constexpr int kRegsHigh = 192;

// Kernel modes: window part, long-range part over exact-set segments, over group lists.
enum : int { kWin = 0, kSeg = 1, kGrp = 2 };

template <int D, int MODE>
struct Layout {
  static constexpr int BOX = QT * 128;        // one TMA box: 128 rows x 128 bytes
  static constexpr int BOXES = D / 64;        // boxes per 128 x D tile
  static constexpr int TILE = BOXES * BOX;    // a 128-row Q/K/V tile, bf16
  static constexpr int Q = 0;
  static constexpr int RING = Q + 2 * TILE;
  static constexpr int BAR = RING + NSTAGE * TILE;
  // barrier block: q, q_empty, full[NSTAGE], empty[NSTAGE], s[2], p[2], o[2], drain,
  // key-set[2], item ring full[NRING] / empty[NRING] (8 bytes each), then the TMEM
  // address word, the abort flag and the ring's item indices
  static constexpr int BAR_Q = 0, BAR_QE = 8, BAR_FULL = 16, BAR_EMPTY = BAR_FULL + 8 * NSTAGE;
  static constexpr int BAR_S = BAR_EMPTY + 8 * NSTAGE, BAR_P = BAR_S + 16, BAR_O = BAR_P + 16;
  static constexpr int BAR_DRAIN = BAR_O + 16, BAR_KS = BAR_DRAIN + 8;
  static constexpr int BAR_RF = BAR_KS + 16, BAR_RE = BAR_RF + 8 * NRING;  // item ring full / empty
  static constexpr int TMEM_SLOT = BAR_RE + 8 * NRING, ABORT = TMEM_SLOT + 4, RING_X = ABORT + 4;
  static constexpr int BAR_BYTES = 256;
  static_assert(RING_X + 4 * NRING <= BAR_BYTES, "barrier block overflow");
  // group lists: per query tile, two buffers of [32 group bits][4 words] key sets
  static constexpr int KSET = BAR + BAR_BYTES;
  static constexpr int KSET_BYTES = MODE == kGrp ? 2 * 2 * 32 * 4 * 4 : 0;
  // window pass: per softmax warp a 32 x 32 fp32 block that turns its rows of O_w
  // into coalesced stores
  static constexpr int STAGE = KSET + KSET_BYTES;
  static constexpr int STAGE_BYTES = MODE == kWin ? 8 * 32 * 32 * 4 : 0;
  static constexpr int SMEM = STAGE + STAGE_BYTES + 1024;  // + 1 KB alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct TcArgs {
  int B, N, H, H_kv, R, w, nseg, qtab_cap;
  int NR;     // permuted rows per (b, rho): N, or N * top_k with group lists
  float sl2;  // softmax scale * log2(e)
  const int* perm;
  const uint32_t* pmask;  // group lists: mask of each permuted row
  float* o_slot;          // group lists: [top_k][B, N, H, d] fp32 list parts
  float* lse_slot;        // group lists: [top_k][B, H, N]
  const QBlock* qtab;
  const int* qtab_count;
  const PlanHead* plan_head;
  const PlanEnt* plan_ent;
  float* o_part;   // window pass output, [B, N, H, d] fp32, normalised
  float* lse_part; // window pass LSE, [B, H, N]
  bf16* o;
  float* lse;
  int* status;
  int* item_counter;         // next work item (zero before the launch)
  long long timeout_cycles;  // limit of every bounded wait
  int stall_producer;        // diagnostic: the producer issues nothing (waits run out)
};

// First index in [lo, hi) with P[index] > x (P ascending), or hi.
__device__ __forceinline__ int upper_bound_g(const int* __restrict__ P, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
}
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
}

// One work item: a 256-row query block of one head.
struct Item {
  bool valid;
  int b, h, kvh, rows, row0;  // row0: first permuted row (long) or first token (window)
  int n;                      // key tiles
  int u;                      // long: schedule entry
  int br;                     // long: b * R + rho
  int seg;                    // long: segment (group list g)
  int j_lo, j_hi;             // window key range
  int skew;                   // window: tile B's key tiles start one tile after tile A's
};

template <bool LONG>
__device__ __forceinline__ Item decode(const TcArgs& a, int x) {
  Item it{};
  if constexpr (LONG) {
    // Heads sharing a KV head are adjacent, then the schedule entries (heaviest
    // first), then the KV heads of a routing head: co-resident CTAs share K/V in L2.
    const int gq = a.H / a.H_kv, nkv = a.H_kv / a.R;
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
    const int rho = e.br % a.R;
    it.kvh = rho * nkv + kvl;
    it.h = it.kvh * gq + jq;
    it.rows = e.rows;
    it.row0 = e.row0;
    it.n = a.plan_head[u].n_tiles;
  } else {
    const int nqb = (a.N + BMQ - 1) / BMQ;
    const int qb = x % nqb;
    const int bh = x / nqb;
    it.valid = true;
    it.h = bh % a.H;
    it.b = bh / a.H;
    it.kvh = it.h / (a.H / a.H_kv);
    it.row0 = qb * BMQ;
    it.rows = min(BMQ, a.N - it.row0);
    it.j_lo = max(0, it.row0 - a.w + 1);
    it.j_hi = it.row0 + it.rows;
    it.n = (it.j_hi - it.j_lo + BNK - 1) / BNK;
    // A full block past the first w - 1 tokens: query tile A (rows row0 ..
    // row0 + 127) needs key tiles 0 .. n - 2 and tile B (row0 + 128 .. row0 + 255)
    // needs 1 .. n - 1 (the band of tile A ends w - 1 + 127 keys after j_lo, tile
    // B's starts 128 keys after it), so each runs n - 1 tiles.
    it.skew = (it.row0 >= a.w - 1 && it.rows == BMQ && it.n >= 2) ? 1 : 0;
  }
  return it;
}

template <int D, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
        const __grid_constant__ CUtensorMap mv, const TcArgs a, const int n_items) {
  constexpr bool LONG = MODE != kWin;
  constexpr bool GROUP = MODE == kGrp;
  using L = Layout<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint8_t* bar = sm + L::BAR;
  const uint32_t b_q = smem_u32(bar) + L::BAR_Q;     // Q tiles landed
  const uint32_t b_qe = smem_u32(bar) + L::BAR_QE;   // Q buffer free (last S of an item done)
  const uint32_t b_full = smem_u32(bar) + L::BAR_FULL, b_empty = smem_u32(bar) + L::BAR_EMPTY;  // + 8 * stage
  const uint32_t b_s = smem_u32(bar) + L::BAR_S, b_p = smem_u32(bar) + L::BAR_P;  // + 8 * query tile
  const uint32_t b_o = smem_u32(bar) + L::BAR_O;
  const uint32_t b_drain = smem_u32(bar) + L::BAR_DRAIN;
  const uint32_t b_ks = smem_u32(bar) + L::BAR_KS;  // + 8 * query tile
  const uint32_t b_rf = smem_u32(bar) + L::BAR_RF, b_re = smem_u32(bar) + L::BAR_RE;  // + 8 * slot
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar + L::TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + L::ABORT);
  volatile int* ring_x = reinterpret_cast<volatile int*>(bar + L::RING_X);

  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(bar + L::TMEM_SLOT), TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qe, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b_s + 8 * t, 1);
      mbar_init(b_p + 8 * t, 4);  // one arrival per softmax warp
      mbar_init(b_o + 8 * t, 1);
    }
    mbar_init(b_drain, 1);
    for (int t = 0; t < 2; ++t) mbar_init(b_ks + 8 * t, 4);
    for (int r = 0; r < NRING; ++r) {
      mbar_init(b_rf + 8 * r, 1);
      mbar_init(b_re + 8 * r, RING_CONSUMERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* status = a.status;
  const long long tlim = a.timeout_cycles;

  if (warp >= 8) {
    setmaxnreg_dec();
    if (warp == PRODUCER_WARP && lane == 0) {
      // ----------------------------------------------------------- producer --
      tma_prefetch(&mq);
      tma_prefetch(&mk);
      tma_prefetch(&mv);
      int last_par[NSTAGE];
      for (int s = 0; s < NSTAGE; ++s) last_par[s] = -1;
      int stage = 0, qcnt = 0, q_par = -1;
      uint32_t phase = 0;
      bool ok = true;
      for (int kr = 0; !a.stall_producer; ++kr) {  // diagnostic: a stalled producer hands out nothing
        const int rs = kr % NRING;
        if (!(ok = mbar_wait(b_re + 8 * rs, ((kr / NRING) & 1) ^ 1, abort_flag, status, tlim))) break;
        const int x = atomicAdd(a.item_counter, 1);
        ring_x[rs] = x;
        mbar_arrive(b_rf + 8 * rs);
        if (x >= n_items) break;
        const Item it = decode<LONG>(a, x);
        if (!it.valid || it.n == 0) continue;
        if (!(ok = mbar_wait(b_qe, (qcnt & 1) ^ 1, abort_flag, status, tlim))) break;
        mbar_expect_tx(b_q, 2 * L::TILE);
        for (int qt = 0; qt < 2; ++qt)
          for (int bx = 0; bx < L::BOXES; ++bx) {
            const uint32_t dst = smem_u32(sm + L::Q + qt * L::TILE + bx * L::BOX);
            if constexpr (LONG)
              tma_load_2d(dst, &mq, 64 * bx, (it.b * a.H + it.h) * a.NR + it.row0 + qt * QT, b_q);
            else
              tma_load_3d(dst, &mq, 64 * bx, it.h, it.b * a.N + it.row0 + qt * QT, b_q);
          }
        q_par = qcnt & 1;
        ++qcnt;
        // key tiles: long = each plan entry's tiles in order; window = consecutive
        int e = 0, t_in = 0;
        PlanEnt pe{};
        if constexpr (LONG) pe = a.plan_ent[(int64_t)it.u * a.nseg];
        for (int t = 0; t < it.n && ok; ++t) {
          int row;
          if constexpr (LONG) {
            row = (it.b * a.H_kv + it.kvh) * a.NR + pe.start + t_in * BNK;
            if (++t_in * BNK >= pe.cnt && ++e < a.nseg) {
              t_in = 0;
              pe = a.plan_ent[(int64_t)it.u * a.nseg + e];
            }
          } else {
            row = it.b * a.N + it.j_lo + t * BNK;
          }
          for (int kv = 0; kv < 2; ++kv) {
            if (!(ok = mbar_wait(b_empty + 8 * stage, phase ^ 1, abort_flag, status, tlim))) break;
            const uint32_t full = b_full + 8 * stage;
            mbar_expect_tx(full, L::TILE);
            for (int bx = 0; bx < L::BOXES; ++bx) {
              const uint32_t dst = smem_u32(sm + L::RING + stage * L::TILE + bx * L::BOX);
              const CUtensorMap* m = kv ? &mv : &mk;
              if constexpr (LONG) tma_load_2d(dst, m, 64 * bx, row, full);
              else tma_load_3d(dst, m, 64 * bx, it.kvh, row, full);
            }
            last_par[stage] = (int)phase;
            if (++stage == NSTAGE) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        if (q_par >= 0) mbar_drain(b_q, (uint32_t)q_par);
        for (int s = 0; s < NSTAGE; ++s)
          if (last_par[s] >= 0) mbar_drain(b_full + 8 * s, (uint32_t)last_par[s]);
      }
    } else if (warp == MMA_WARP && lane == 0) {
      // ---------------------------------------------------------- MMA issue --
      constexpr uint32_t IS = idesc_bf16(QT, BNK, 0);  // S = Q K^T, both K-major
      constexpr uint32_t IPV = idesc_bf16(QT, D, 1);   // O += P V, V MN-major
      const uint32_t q_base = smem_u32(sm + L::Q);
      const uint32_t r_base = smem_u32(sm + L::RING);
      auto slot = [&](int item) { return r_base + (item % NSTAGE) * L::TILE; };
      auto ring_wait = [&](int item) {
        return mbar_wait(b_full + 8 * (item % NSTAGE), (item / NSTAGE) & 1, abort_flag, status, tlim);
      };
      // Descriptors are built once per tile; a K step only moves the start address
      // (bits 0-13, in 16-byte units, no carry out of the field inside shared
      // memory), so each MMA costs the issuing thread one add.
      auto issue_S = [&](int qt, uint32_t kaddr) {
        const uint64_t da = sw128_desc(q_base + qt * L::TILE, 16, 1024);
        const uint64_t db = sw128_desc(kaddr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * L::BOX + (kk % 4) * 32) >> 4;
          umma_ss(tmem + qt * BNK, da + off, db + off, IS, kk > 0);
        }
      };
      auto issue_PV = [&](int qt, uint32_t vaddr, bool acc) {
        // A = P in TMEM (written over the first 64 columns of S_qt), 8 columns per K step
        const uint64_t dv = sw128_desc(vaddr, L::BOX, 1024);
#pragma unroll
        for (int kk = 0; kk < BNK / 16; ++kk)
          umma_ts(tmem + 2 * BNK + qt * D, tmem + qt * BNK + 8 * kk, dv + ((kk * 2048) >> 4), IPV,
                  (acc || kk > 0) ? 1u : 0u);
      };
      int ri = 0, gt = 0, qcnt = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        const int rs = kr % NRING;
        if (!(ok = mbar_wait(b_rf + 8 * rs, (kr / NRING) & 1, abort_flag, status, tlim))) break;
        const int x = ring_x[rs];
        mbar_arrive(b_re + 8 * rs);
        if (x >= n_items) break;
        const Item it = decode<LONG>(a, x);
        if (!it.valid || it.n == 0) continue;
        // sk: the window pass's skew (0 in the long-range passes, at compile time, so
        // their issue stream carries no extra waits: every instruction of this thread
        // between MMA groups delays the tensor core)
        const int n = it.n, sk = LONG ? 0 : it.skew, ns = n - sk;  // ns key steps of each tile
        if (!(ok = mbar_wait(b_q, qcnt & 1, abort_flag, status, tlim) && ring_wait(ri))) break;
        if (sk && !(ok = ring_wait(ri + 2))) break;
        ++qcnt;
        tc_fence_after();
        issue_S(0, slot(ri));
        umma_commit(b_s);
        issue_S(1, slot(ri + 2 * sk));
        umma_commit(b_s + 8);
        umma_commit(b_empty + 8 * (ri % NSTAGE));
        if (ns == 1) umma_commit(b_qe);
        // A commit makes the tensor core finish everything issued before it, so
        // the commits are gathered at two points per key step (after S_A and
        // after S_B; measured: six commits at four points cost ~10% of the
        // tensor core's rate).  O is signalled once per item, after its last P V;
        // V(t) is released together with K(t+1), after S_B(t+1).
        // Tile A's step t uses V(t) and K(t + 1), tile B's V(t + sk) and K(t + 1 + sk)
        // (ring items V(u) = ri + 2u + 1, K(u) = ri + 2u).  At the end of step t,
        // V(t) and K(t + 1) have had their last use; with the skew V(n - 1) too.
        for (int t = 0; t < ns; ++t) {
          const int iva = ri + 2 * t + 1, ika = ri + 2 * t + 2;
          const int ivb = iva + 2 * sk, ikb = ika + 2 * sk;
          const uint32_t par = (uint32_t)((gt + t) & 1);
          const bool last = t + 1 == ns;
          if (!(ok = ring_wait(iva) && mbar_wait(b_p, par, abort_flag, status, tlim))) break;
          tc_fence_after();
          issue_PV(0, slot(iva), t > 0);
          if (last) umma_commit(b_o);
          if (!last) {
            if (!(ok = ring_wait(ika))) break;
            tc_fence_after();
            issue_S(0, slot(ika));
            umma_commit(b_s);
          }
          if (sk && !(ok = ring_wait(ivb))) break;
          if (!(ok = mbar_wait(b_p + 8, par, abort_flag, status, tlim))) break;
          tc_fence_after();
          issue_PV(1, slot(ivb), t > 0);
          if (last) umma_commit(b_o + 8);
          if (!last) {
            if (sk) {
              if (!(ok = ring_wait(ikb))) break;
              tc_fence_after();
            }
            issue_S(1, slot(ikb));
            umma_commit(b_s + 8);
            if (t + 2 == ns) umma_commit(b_qe);  // last S of this item issued
          }
          if (!last) umma_commit(b_empty + 8 * (ika % NSTAGE));  // t + 1 < n
          else if (sk) umma_commit(b_empty + 8 * (ika % NSTAGE));
          umma_commit(b_empty + 8 * (iva % NSTAGE));
          if (sk && last) umma_commit(b_empty + 8 * (ivb % NSTAGE));
        }
        ri += 2 * n;
        gt += ns;
        if (!ok) break;
      }
      umma_commit(b_drain);  // every MMA issued above completes before TMEM is released
      mbar_drain(b_drain, 0);
    }
    __syncwarp();
  } else {
    setmaxnreg_inc();
    // -------------------------------------------------------------- softmax --
    const int qt = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + qt * BNK;
    const uint32_t tO = tmem + lane_off + 2 * BNK + qt * D;
    const float sl2 = a.sl2;
    int gt = 0;
    int o_items = 0;  // items with key tiles so far: b_o completes once per such item
    int ks_cnt = 0;  // key-set barrier uses (group lists)
    bool ok = true;
    for (int kr = 0;; ++kr) {
      const int rs = kr % NRING;
      ok = mbar_wait(b_rf + 8 * rs, (kr / NRING) & 1, abort_flag, status, tlim);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int x = ring_x[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_re + 8 * rs);
      if (x >= n_items) break;
      const Item it = decode<LONG>(a, x);
      if (!it.valid) continue;
      const int n = it.n - it.skew;  // key steps of this tile
      const int rg = qt * QT + r;  // row in the item
      const bool row_ok = rg < it.rows;
      const int* P = LONG ? a.perm + (int64_t)it.br * a.NR : nullptr;
      int qp;
      if constexpr (LONG) qp = __ldg(P + it.row0 + min(rg, it.rows - 1));
      else qp = it.row0 + min(rg, it.rows - 1);
      float m_use = -INFINITY, l = 0.0f;
      int e = 0, t_in = 0;
      PlanEnt pe{};
      if constexpr (LONG) {
        if (n > 0) pe = a.plan_ent[(int64_t)it.u * a.nseg];
      }
      // group lists: this row's groups below g (keys sharing one of them are counted
      // in a lower list), its slot, and the next key tile's masks (one per thread)
      const int g = GROUP ? it.seg : 0;
      const uint32_t* PM = GROUP ? a.pmask + (int64_t)it.br * a.NR : nullptr;
      uint32_t m_low = 0u, mj_next = 0u;
      const int kc = (warp & 3) * 32 + lane;  // key column this thread fetches
      if constexpr (GROUP) {
        m_low = __ldg(PM + it.row0 + min(rg, it.rows - 1)) & ((1u << g) - 1u);
        if (g > 0 && n > 0 && kc < pe.cnt) mj_next = __ldg(PM + pe.start + kc);
      }
      for (int t = 0; t < n; ++t) {
        int c_lo = 0, c_hi = BNK;
        bool need_mask;
        uint32_t mj = 0u;
        if constexpr (GROUP) mj = mj_next;
        if constexpr (LONG) {
          const int valid = min(BNK, pe.cnt - t_in * BNK);
          need_mask = t_in >= pe.nfull;
          if (need_mask) c_hi = upper_bound_g(P + pe.start + t_in * BNK, 0, valid, qp - a.w);
          if (++t_in * BNK >= pe.cnt && ++e < a.nseg) {
            t_in = 0;
            pe = a.plan_ent[(int64_t)it.u * a.nseg + e];
          }
          if constexpr (GROUP) {  // (pe, t_in) now describe tile t + 1
            if (g > 0 && t + 1 < n) {
              const int c = t_in * BNK + kc;
              mj_next = c < pe.cnt ? __ldg(PM + pe.start + c) : 0u;
            }
          }
        } else {
          const int j0 = it.j_lo + (t + (qt ? it.skew : 0)) * BNK;
          c_lo = max(0, qp - a.w + 1 - j0);
          c_hi = min(min(BNK, it.j_hi - j0), qp - j0 + 1);
          need_mask = c_lo > 0 || c_hi < BNK;
        }
        // key columns whose key shares a group below g with this row
        uint32_t dk0 = 0u, dk1 = 0u, dk2 = 0u, dk3 = 0u;
        if constexpr (GROUP) {
          if (g > 0) {
            uint32_t* ks = reinterpret_cast<uint32_t*>(sm + L::KSET) + (qt * 2 + (ks_cnt & 1)) * 128;
            for (int bit = 0; bit < g; ++bit) {
              const unsigned bal = __ballot_sync(0xffffffffu, (mj >> bit) & 1u);
              if (lane == 0) ks[bit * 4 + (warp & 3)] = bal;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(b_ks + 8 * qt);
            ok = mbar_wait(b_ks + 8 * qt, (uint32_t)(ks_cnt & 1), abort_flag, status, tlim);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            ++ks_cnt;
            uint32_t mm = m_low;
            while (mm) {
              const int bit = __ffs(mm) - 1;
              mm &= mm - 1u;
              const uint4 v = *reinterpret_cast<const uint4*>(ks + bit * 4);
              dk0 |= v.x;
              dk1 |= v.y;
              dk2 |= v.z;
              dk3 |= v.w;
            }
          }
        }
        ok = mbar_wait(b_s + 8 * qt, (uint32_t)((gt + t) & 1), abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t x0[32], x1[32], x2[32], x3[32];
        tmem_ld32(tS + 0, x0);
        tmem_ld32(tS + 32, x1);
        tmem_ld32(tS + 64, x2);
        tmem_ld32(tS + 96, x3);
        tmem_ld_wait(x0);
        tie32(x1);
        tie32(x2);
        tie32(x3);
        // mask (raw logits; the scale is positive, so the max commutes with it)
        if (need_mask) {
          const uint32_t width = (uint32_t)max(c_hi - c_lo, 0);
          auto mask32 = [&](uint32_t(&xx)[32], int cb) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if ((uint32_t)(cb + i - c_lo) >= width) xx[i] = 0xff800000u;  // -inf
          };
          mask32(x0, 0);
          mask32(x1, 32);
          mask32(x2, 64);
          mask32(x3, 96);
        }
        if constexpr (GROUP) {
          if (__any_sync(0xffffffffu, (dk0 | dk1 | dk2 | dk3) != 0u)) {
            auto drop32 = [&](uint32_t(&xx)[32], uint32_t ex) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if ((ex >> i) & 1u) xx[i] = 0xff800000u;  // -inf
            };
            drop32(x0, dk0);
            drop32(x1, dk1);
            drop32(x2, dk2);
            drop32(x3, dk3);
          }
        }
        // Row max, taken lazily: the exponentials use the running estimate m_use and
        // the tile's max is computed only while a row has none yet (m_use = -inf) or
        // when the tile's exponentials sum past kSumCap (then the tile is redone with
        // its max).  P keeps its relative precision at any magnitude (bf16 has fp32's
        // exponent range) and O and l have headroom far above kSumCap * keys * |v|,
        // so this equals the exact online softmax up to rounding, without 64 max
        // operations per row on every tile.
        float f = 1.0f;
        bool rescale = false;
        auto take_max = [&]() {
          float mm[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) mm[j] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            mm[i & 7] = max3(mm[i & 7], __uint_as_float(x0[i]), __uint_as_float(x1[i]));
#pragma unroll
          for (int i = 0; i < 32; ++i)
            mm[i & 7] = max3(mm[i & 7], __uint_as_float(x2[i]), __uint_as_float(x3[i]));
          const float mx = max3(max3(mm[0], mm[1], mm[2]), max3(mm[3], mm[4], mm[5]),
                                fmaxf(mm[6], mm[7])) * sl2;
          rescale = mx > m_use + kRescale;
          if (rescale) {
            f = ex2(m_use - mx);  // 0 when m_use is -inf
            l *= f;
            m_use = mx;
          }
        };
        if (__any_sync(0xffffffffu, m_use == -INFINITY)) take_max();
        float la, lb;
        // P (bf16 pairs) goes over the first 64 TMEM columns of this tile's S, which
        // are already in registers: column 16k + i holds keys 32k + 2i and 32k + 2i + 1.
        auto emit_all = [&]() {
          const float nms = (m_use == -INFINITY) ? 0.0f : -m_use;
          la = 0.0f;
          lb = 0.0f;
          auto emit = [&](uint32_t(&xx)[32], int k) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              ffma2(y0, y1, __uint_as_float(xx[2 * i]), __uint_as_float(xx[2 * i + 1]), sl2, sl2, nms, nms);
              const float p0 = ex2(y0), p1 = ex2(y1);
              fadd2(la, lb, la, lb, p0, p1);
              pk[i] = pack_bf16(p0, p1);
            }
            tmem_st16(tS + 16 * k, pk);
          };
          emit(x0, 0);
          emit(x1, 1);
          emit(x2, 2);
          emit(x3, 3);
        };
        emit_all();
        if (__any_sync(0xffffffffu, !(la + lb <= kSumCap))) {  // rare: the max grew a lot
          take_max();
          emit_all();
        }
        l += la + lb;
        // O (from P V of earlier tiles, all complete once S of this tile is) follows
        // the new maximum; skipped while this row has seen no key (O is still zero).
        if (__any_sync(0xffffffffu, rescale && t > 0 && f != 0.0f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t y[32];
            tmem_ld32(tO + 32 * c, y);
            tmem_ld_wait(y);
            const float g = (rescale && t > 0) ? f : 1.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = __float_as_uint(__uint_as_float(y[i]) * g);
            tmem_st32(tO + 32 * c, y);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p + 8 * qt);
      }
      if (!ok) break;
      // ---- epilogue of this item ----
      if (n > 0) {
        ok = mbar_wait(b_o + 8 * qt, (uint32_t)(o_items & 1), abort_flag, status, tlim);
        ++o_items;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      gt += n;
      const int64_t orow = (((int64_t)it.b * a.N + qp) * a.H + it.h) * D;
      const int64_t lrow = ((int64_t)it.b * a.H + it.h) * a.N + qp;
      if constexpr (!LONG) {
        // window pass (runs first): normalised partial output and its LSE.  A thread
        // holds its row; rows are stored 32 columns at a time through this warp's
        // 32 x 32 block in shared memory (XOR-swizzled: both the row writes and the
        // column reads are free of bank conflicts), one 128-byte row segment per
        // store instead of 32 scattered 16-byte pieces.  A warp's 32 rows are
        // consecutive tokens, so row j is `H * D` floats after row 0.
        const float inv = 1.0f / l;  // the diagonal key is always in the window
        const float lse = (m_use + log2f(l)) * kLn2;
        float* st = reinterpret_cast<float*>(sm + L::STAGE) + (warp & 7) * 32 * 32;
        const int rg0 = qt * QT + (warp & 3) * 32;  // the warp's first row in the item
        const int64_t orow0 = (((int64_t)it.b * a.N + it.row0 + rg0) * a.H + it.h) * D;
        const int64_t rstride = (int64_t)a.H * D;
        const int nrows = min(32, it.rows - rg0);  // rows of this warp inside the item
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t y[32];
          tmem_ld32(tO + 32 * c, y);
          tmem_ld_wait(y);
#pragma unroll
          for (int i = 0; i < 32; ++i) st[lane * 32 + (i ^ lane)] = __uint_as_float(y[i]) * inv;
          __syncwarp();
          for (int j = 0; j < nrows; ++j)
            a.o_part[orow0 + j * rstride + 32 * c + lane] = st[j * 32 + (lane ^ j)];
          __syncwarp();
        }
        if (row_ok) a.lse_part[lrow] = lse;
      } else if constexpr (GROUP) {
        // list g's normalised part into the token's slot; a row that met no key
        // leaves weight 0 (LSE -inf) for the merge
        const int slot = __popc(m_low);
        const bool any = l > 0.0f;
        const float inv = any ? 1.0f / l : 0.0f;
        const float lse = any ? (m_use + log2f(l)) * kLn2 : -INFINITY;
        float* os = a.o_slot + (int64_t)slot * a.B * a.N * a.H * D + orow;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t y[32];
          if (n > 0) {
            tmem_ld32(tO + 32 * c, y);
            tmem_ld_wait(y);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = 0u;
          }
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(os + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(y[4 * i]) * inv, __uint_as_float(y[4 * i + 1]) * inv,
                                   __uint_as_float(y[4 * i + 2]) * inv, __uint_as_float(y[4 * i + 3]) * inv);
          }
        }
        if (row_ok) a.lse_slot[(int64_t)slot * a.B * a.H * a.N + lrow] = lse;
      } else {
        // long-range pass: one softmax over the union = LSE merge of this pass with
        // the window pass (disjoint key sets); writes the final O and LSE
        float wo = 0.0f, ww = 1.0f, lse = 0.0f;
        if (row_ok) {
          const float lse_w = a.lse_part[lrow];
          lse = lse_w;
          if (l > 0.0f) {
            const float lse_o = (m_use + log2f(l)) * kLn2;
            const float M = fmaxf(lse_w, lse_o);
            const float ew = expf(lse_w - M), eo = expf(lse_o - M);
            const float tot = ew + eo;
            lse = M + logf(tot);
            wo = eo / tot / l;
            ww = ew / tot;
          }
        }
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t y[32];
          if (n > 0) {
            tmem_ld32(tO + 32 * c, y);
            tmem_ld_wait(y);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = 0u;
          }
          if (row_ok) {
            const float4* src = reinterpret_cast<const float4*>(a.o_part + orow + 32 * c);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 ow = src[i];
              pk[2 * i] = pack_bf16(__uint_as_float(y[4 * i]) * wo + ow.x * ww,
                                    __uint_as_float(y[4 * i + 1]) * wo + ow.y * ww);
              pk[2 * i + 1] = pack_bf16(__uint_as_float(y[4 * i + 2]) * wo + ow.z * ww,
                                        __uint_as_float(y[4 * i + 3]) * wo + ow.w * ww);
            }
            uint4* dst = reinterpret_cast<uint4*>(a.o + orow + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (row_ok && a.lse) a.lse[lrow] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side --
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

// Tensor map over rows of D bf16 values: `heads` rows per token when heads > 0
// (3-D: d, head, token), else plain rows (2-D: d, row).  Box: 64 columns x 128 rows
// (x 1 head), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int64_t rows, int heads) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r;
  if (heads > 0) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, 128};
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

TcArgs make_args(const focus_params& p, const WsLayout& L, char* ws, float scale) {
  TcArgs a{};
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
  a.perm = reinterpret_cast<const int*>(ws + L.perm);
  a.pmask = reinterpret_cast<const uint32_t*>(ws + L.pmask);
  a.o_slot = reinterpret_cast<float*>(ws + L.oslot);
  a.lse_slot = reinterpret_cast<float*>(ws + L.lseslot);
  a.qtab = reinterpret_cast<const QBlock*>(ws + L.qtab);
  a.qtab_count = &reinterpret_cast<const WsHeader*>(ws)->qtab_count;
  a.plan_head = reinterpret_cast<const PlanHead*>(ws + L.plan_head);
  a.plan_ent = reinterpret_cast<const PlanEnt*>(ws + L.plan_ent);
  a.o_part = reinterpret_cast<float*>(ws + L.olr);
  a.lse_part = reinterpret_cast<float*>(ws + L.lselr);
  a.status = &reinterpret_cast<WsHeader*>(ws)->status;
  a.item_counter = &reinterpret_cast<WsHeader*>(ws)->item_counter[0];
  a.timeout_cycles = kTimeoutCycles;
  a.stall_producer = 0;
  return a;
}

template <int D, int MODE>
cudaError_t launch_tc(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const TcArgs& a, int n_items, cudaStream_t s) {
  const int smem = Layout<D, MODE>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(attn_tc<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  const int grid = n_items < sms ? n_items : sms;
  if (grid < 1) return cudaSuccess;
  attn_tc<D, MODE><<<grid, NTHREADS, smem, s>>>(mq, mk, mv, a, n_items);
  return cudaGetLastError();
}

}  // namespace

int tc_block_rows() { return BMQ; }

// Diagnostic launch: the window kernel on a tiny problem with its producer held back
// and ~10 ms waits, so the MMA issuer's first wait runs out, the CTA aborts (nothing
// is in flight), frees its tensor memory and exits with FOCUS_ERR_TIMEOUT raised.
cudaError_t launch_timeout_selftest(char* ws, size_t ws_bytes, cudaStream_t s) {
  focus_params p{};
  p.B = 1;
  p.N = 256;
  p.H = p.H_kv = 1;
  p.d_head = 64;
  p.R = 1;
  p.K = 1;
  p.top_k = 1;
  p.w = 64;
  WsLayout L{};
  L.nseg = 1;
  L.olr = 4096;
  L.lselr = 4096 + 256 * 64 * 4;
  if (ws_bytes < L.lselr + 256 * 4) return cudaErrorInvalidValue;
  TcArgs a = make_args(p, L, ws, 0.125f);
  a.timeout_cycles = 20000000LL;
  a.stall_producer = 1;
  CUtensorMap mq, mk, mv;  // valid maps over the workspace; nothing is loaded
  if (!make_map(&mq, ws, 64, 256, 1) || !make_map(&mk, ws, 64, 256, 1) ||
      !make_map(&mv, ws, 64, 256, 1))
    return cudaErrorInvalidValue;
  return launch_tc<64, kWin>(mq, mk, mv, a, 1, s);
}

// FOCUS_LONG_ENGINE=pair runs the long-range pass on CTA pairs where that engine
// applies (d = 128, exact-set segments); otherwise this kernel runs it.  Both give
// the same result up to rounding order.
bool use_pair_engine(const focus_params& p, const WsLayout& L) {
  const char* e = std::getenv("FOCUS_LONG_ENGINE");
  return e && std::strcmp(e, "pair") == 0 && pair_engine_supported(p, L);
}

cudaError_t launch_attn_long_tc(const focus_params& p, const WsLayout& L, char* ws, bf16* o,
                                float* lse, float scale, cudaStream_t s) {
  if (use_pair_engine(p, L)) return launch_attn_long_pair(p, L, ws, o, lse, scale, s);
  TcArgs a = make_args(p, L, ws, scale);
  a.o = o;
  a.lse = lse;
  a.item_counter = &reinterpret_cast<WsHeader*>(ws)->item_counter[1];
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, ws + L.qp, p.d_head, (int64_t)p.B * p.H * L.NR, 0) ||
      !make_map(&mk, ws + L.kp, p.d_head, (int64_t)p.B * p.H_kv * L.NR, 0) ||
      !make_map(&mv, ws + L.vp, p.d_head, (int64_t)p.B * p.H_kv * L.NR, 0))
    return cudaErrorInvalidValue;
  const int n_items = a.qtab_cap * (p.H / p.R);
  if (L.group)
    return p.d_head == 64 ? launch_tc<64, kGrp>(mq, mk, mv, a, n_items, s)
                          : launch_tc<128, kGrp>(mq, mk, mv, a, n_items, s);
  return p.d_head == 64 ? launch_tc<64, kSeg>(mq, mk, mv, a, n_items, s)
                        : launch_tc<128, kSeg>(mq, mk, mv, a, n_items, s);
}

cudaError_t launch_attn_window_tc(const focus_params& p, const WsLayout& L, const bf16* q,
                                  const bf16* k, const bf16* v, char* ws, float scale,
                                  cudaStream_t s) {
  TcArgs a = make_args(p, L, ws, scale);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, p.d_head, (int64_t)p.B * p.N, p.H) ||
      !make_map(&mk, k, p.d_head, (int64_t)p.B * p.N, p.H_kv) ||
      !make_map(&mv, v, p.d_head, (int64_t)p.B * p.N, p.H_kv))
    return cudaErrorInvalidValue;
  const int n_items = p.B * p.H * ((p.N + BMQ - 1) / BMQ);
  return p.d_head == 64 ? launch_tc<64, kWin>(mq, mk, mv, a, n_items, s)
                        : launch_tc<128, kWin>(mq, mk, mv, a, n_items, s);
}

}  // namespace focus
