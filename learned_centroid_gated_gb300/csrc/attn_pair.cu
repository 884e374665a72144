// Long-range Focus attention on CTA pairs (tcgen05 cta_group::2), d = 128.
//
// "Why Attend to Everything? Focus is the Key", gist.science technical summary,
// section 2 "Core Architecture" and "Inference Efficiency (Top-k)": distant keys are
// attended only within a shared group, with exact softmax; the long-range keys
// (pos_j <= pos_i - w) and the window keys are disjoint, so this pass merges with the
// window pass's normalised partial (O_w, LSE_w) by log-sum-exp.  Same work items,
// plans, tile order and result as attn_tc<128, kSeg> (exact-set segments), on an
// engine built to take the next S off the softmax's critical path.  On the workloads
// measured it is slower than attn_tc (7.1 against 5.5 ms at 32K tokens: a thread's
// fixed costs per tile, not the tensor core, bound it), so it runs only when
// FOCUS_LONG_ENGINE=pair asks for it:
//
// A cluster of two CTAs (the two SMs of a TPC) runs each 256-row query block; CTA r
// holds rows 128 r .. 128 r + 127.  One thread of CTA 0 issues every MMA with
// cta_group::2 (M = 256): S = Q K^T with each CTA's Q from its own shared memory and
// the K tile split by keys (CTA r holds keys 64 r .. 64 r + 63), O += P V with P from
// each CTA's tensor memory and the V tile split by columns (CTA r holds d columns
// 64 r .. 64 r + 63).  Each SM loads half of every K/V tile and keeps only its 128
// rows of S and O, so its 512 TMEM columns hold two S buffers and two O buffers:
// S(t + 1) is computed while the softmax of tile t runs, and the softmax of
// consecutive tiles runs back to back instead of waiting for P V(t) and S(t + 1).
//   warps 0-3   softmax: thread = row = TMEM lane, the whole 128-key row of each
//               tile; the item's epilogue (merge with the window pass) as well
//   warps 4-7   no role (complete the warpgroup for the register split)
//   warp 8      TMA producer of this CTA's halves; in CTA 0 it also takes the work
//               items from the global counter and hands them to both CTAs
//   warp 9      MMA issuer (CTA 0); warp 9 of both CTAs allocates the tensor memory
//   warp 10     CTA 1: forwards the completion of its loads to CTA 0's barriers
//   warp 11     idle (completes the third warpgroup for the register split)
// TMEM: S0 | S1 | O0 | O1 (128 columns each).  P (bf16 pairs: keys 2i, 2i + 1 in
// column i) is written over the first 64 columns of its S buffer by the thread that
// has just read that row.  O alternates between items, so the next item's first
// P V need not wait for the previous epilogue.  Every wait is bounded; a CTA that
// gives up raises FOCUS_ERR_TIMEOUT, and its peer's waits then run out as well.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace focus {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int QT = 128;        // query rows per CTA
constexpr int BNK = kKeyTile;  // keys per tile
constexpr int NST = 8;         // K/V half slots per CTA
constexpr int NRING = 4;       // work items in flight between the roles
constexpr int NTHREADS = 384;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int FWD_WARP = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 2 * 128;  // O0, O1 (S0, S1 before them)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
// Arrivals on CTA 0's item-ring "empty" barrier: its MMA issuer and 4 softmax warps,
// CTA 1's producer, 4 softmax warps and forwarder.
constexpr int RING_CONSUMERS = 11;
constexpr int PAIR_WARPS = 8;  // softmax warps of both CTAs (P ready, O read)
constexpr float kSumCap = 1.8446744e19f;  // 2^64: a tile's exponentials above this retake the max
// Register split after launch (384 threads x 168): warpgroup 2 drops to 104, the two
// softmax warpgroups rise to 192: 128 * 104 + 256 * 192 = 62464 <= 64512.
constexpr int kRegsLow = 104;
constexpr int kRegsHigh = 192;
static_assert(BNK == 128, "the key tile is split 64 + 64 between the pair");

struct PairLayout {
  static constexpr int QBOX = QT * 128;    // Q box: 128 rows x 64 bf16 (128 B)
  static constexpr int QTILE = 2 * QBOX;   // this CTA's 128 x 128 Q tile
  static constexpr int KBOX = 64 * 128;    // K half box: 64 keys x 64 bf16
  static constexpr int SLOT = 16384;       // K half (2 boxes) or V half (128 keys x 64 bf16)
  static constexpr int Q = 0;              // two Q buffers
  static constexpr int RING = Q + 2 * QTILE;
  static constexpr int BAR = RING + NST * SLOT;
  // barriers (8 bytes each): q_full[2], q_free[2], full[NST], empty[NST], s_full[2],
  // p_ready[2], o_full[2], o_free[2], pv_last, ring_full[NRING], ring_empty[NRING],
  // drain; then the TMEM address word, the abort flag and the ring's item indices
  static constexpr int B_QFULL = 0, B_QFREE = 16, B_FULL = 32, B_EMPTY = B_FULL + 8 * NST;
  static constexpr int B_SFULL = B_EMPTY + 8 * NST, B_PREADY = B_SFULL + 16;
  static constexpr int B_OFULL = B_PREADY + 16, B_OFREE = B_OFULL + 16, B_PVLAST = B_OFREE + 16;
  static constexpr int B_RF = B_PVLAST + 8, B_RE = B_RF + 8 * NRING, B_DRAIN = B_RE + 8 * NRING;
  static constexpr int TMEM_SLOT = B_DRAIN + 8, ABORT = TMEM_SLOT + 4, RING_X = ABORT + 4;
  static constexpr int BAR_BYTES = 512;
  static_assert(RING_X + 4 * NRING <= BAR_BYTES, "barrier block overflow");
  static constexpr int SMEM = BAR + BAR_BYTES + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct PairArgs {
  int B, N, H, H_kv, R, w, nseg, qtab_cap;
  int NR;     // permuted rows per (b, rho)
  float sl2;  // softmax scale * log2(e)
  const int* perm;
  const QBlock* qtab;
  const int* qtab_count;
  const PlanHead* plan_head;
  const PlanEnt* plan_ent;
  const float* o_part;    // window pass output, [B, N, H, d] fp32, normalised
  const float* lse_part;  // window pass LSE, [B, H, N]
  bf16* o;
  float* lse;
  int* status;
  int* item_counter;  // next work item (zero before the launch)
  long long timeout_cycles;
};

// One work item: a 256-row query block of one head (rows of one exact-set segment).
struct Item {
  bool valid;
  int b, h, kvh, rows, row0, n, u, br;
};

// The long-range work list of attn_tc<D, kSeg>: query heads sharing a KV head are
// adjacent, then the schedule entries (heaviest first), then the KV heads of a
// routing head, so co-resident pairs share K/V tiles in L2.
__device__ __forceinline__ Item decode(const PairArgs& a, int x) {
  Item it{};
  const int gq = a.H / a.H_kv, nkv = a.H_kv / a.R;
  const int jq = x % gq;
  const int rest = x / gq;
  const int u = rest % a.qtab_cap, kvl = rest / a.qtab_cap;
  it.valid = u < *a.qtab_count;
  if (!it.valid) return it;
  const QBlock e = a.qtab[u];
  it.u = u;
  it.br = e.br;
  it.b = e.br / a.R;
  const int rho = e.br % a.R;
  it.kvh = rho * nkv + kvl;
  it.h = it.kvh * gq + jq;
  it.rows = e.rows;
  it.row0 = e.row0;
  it.n = a.plan_head[u].n_tiles;
  return it;
}

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

__global__ void __launch_bounds__(NTHREADS, 1)
attn_pair(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
          const __grid_constant__ CUtensorMap mv, const PairArgs a, const int n_items) {
  using L = PairLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool lead = rank == 0;

  const uint32_t bar = smem_u32(sm + L::BAR);
  auto q_full = [&](int i) { return bar + L::B_QFULL + 8 * i; };
  auto q_free = [&](int i) { return bar + L::B_QFREE + 8 * i; };
  auto full = [&](int i) { return bar + L::B_FULL + 8 * (i % NST); };    // ring item i
  auto empty = [&](int i) { return bar + L::B_EMPTY + 8 * (i % NST); };
  auto s_full = [&](int b) { return bar + L::B_SFULL + 8 * b; };
  auto p_ready = [&](int b) { return bar + L::B_PREADY + 8 * b; };
  auto o_full = [&](int b) { return bar + L::B_OFULL + 8 * b; };
  auto o_free = [&](int b) { return bar + L::B_OFREE + 8 * b; };
  const uint32_t pv_last = bar + L::B_PVLAST, drain = bar + L::B_DRAIN;
  auto ring_full = [&](int r) { return bar + L::B_RF + 8 * r; };
  auto ring_empty = [&](int r) { return bar + L::B_RE + 8 * r; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + L::BAR + L::TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::BAR + L::ABORT);
  volatile int* ring_x = reinterpret_cast<volatile int*>(sm + L::BAR + L::RING_X);
  // arrive on CTA 0's copy of a barrier (local in CTA 0, remote from CTA 1); used
  // where the data is in tensor memory (completed and fenced) or already read
  auto arrive_lead = [&](uint32_t b) {
    if (lead) mbar_arrive(b); else mbar_arrive_remote(mapa_shared(b, 0));
  };

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), lead ? 2 : 1);  // CTA 0: its own load + CTA 1's forwarded one
      mbar_init(q_free(i), 1);
      mbar_init(s_full(i), 1);
      mbar_init(p_ready(i), PAIR_WARPS);
      mbar_init(o_full(i), 1);
      mbar_init(o_free(i), PAIR_WARPS);
    }
    for (int s = 0; s < NST; ++s) {
      mbar_init(full(s), lead ? 2 : 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(pv_last, 1);
    for (int r = 0; r < NRING; ++r) {
      mbar_init(ring_full(r), 1);
      mbar_init(ring_empty(r), RING_CONSUMERS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc2(smem_u32(sm + L::BAR + L::TMEM_SLOT), TMEM_COLS);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
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
      int last_par[NST], q_last[2] = {-1, -1};
      for (int s = 0; s < NST; ++s) last_par[s] = -1;
      int ri = 0, qcnt = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        const int rs = kr % NRING, rpar = (kr / NRING) & 1;
        int x;
        if (lead) {
          if (!(ok = mbar_wait_cl(ring_empty(rs), rpar ^ 1, abort_flag, status, tlim))) break;
          x = atomicAdd(a.item_counter, 1);
          ring_x[rs] = x;
          const uint32_t xa = smem_u32((const void*)(ring_x + rs));
          st_cluster_u32(mapa_shared(xa, 1), (uint32_t)x);
          mbar_arrive(ring_full(rs));
          mbar_arrive_cluster(mapa_shared(ring_full(rs), 1));  // releases the store above
        } else {
          if (!(ok = mbar_wait_cl(ring_full(rs), rpar, abort_flag, status, tlim))) break;
          x = ring_x[rs];
          mbar_arrive_remote(mapa_shared(ring_empty(rs), 0));
        }
        if (x >= n_items) break;
        const Item it = decode(a, x);
        if (!it.valid || it.n == 0) continue;
        const int qb = qcnt & 1;
        if (!(ok = mbar_wait_cl(q_free(qb), ((qcnt >> 1) & 1) ^ 1, abort_flag, status, tlim))) break;
        mbar_expect_tx(q_full(qb), L::QTILE);
        const int qrow = (it.b * a.H + it.h) * a.NR + it.row0 + (int)rank * QT;
        for (int bx = 0; bx < 2; ++bx)
          tma_load_2d(smem_u32(sm + L::Q + qb * L::QTILE + bx * L::QBOX), &mq, 64 * bx, qrow, q_full(qb));
        q_last[qb] = (qcnt >> 1) & 1;
        ++qcnt;
        // key tiles: each plan entry's tiles in order; ring item 2t = K half, 2t + 1 = V half
        int e = 0, t_in = 0;
        PlanEnt pe = a.plan_ent[(int64_t)it.u * a.nseg];
        for (int t = 0; t < it.n && ok; ++t) {
          const int krow = (it.b * a.H_kv + it.kvh) * a.NR + pe.start + t_in * BNK;
          if (++t_in * BNK >= pe.cnt && ++e < a.nseg) {
            t_in = 0;
            pe = a.plan_ent[(int64_t)it.u * a.nseg + e];
          }
          for (int kv = 0; kv < 2; ++kv, ++ri) {
            const int par = (ri / NST) & 1;
            if (!(ok = mbar_wait_cl(empty(ri), par ^ 1, abort_flag, status, tlim))) break;
            mbar_expect_tx(full(ri), L::SLOT);
            const uint32_t dst = smem_u32(sm + L::RING + (ri % NST) * L::SLOT);
            if (kv == 0) {
              for (int bx = 0; bx < 2; ++bx)
                tma_load_2d(dst + bx * L::KBOX, &mk, 64 * bx, krow + (int)rank * 64, full(ri));
            } else {
              tma_load_2d(dst, &mv, 64 * (int)rank, krow, full(ri));
            }
            last_par[ri % NST] = par;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        for (int i = 0; i < 2; ++i)
          if (q_last[i] >= 0) mbar_drain_cl(q_full(i), (uint32_t)q_last[i]);
        for (int s = 0; s < NST; ++s)
          if (last_par[s] >= 0) mbar_drain_cl(full(s), (uint32_t)last_par[s]);
      }
    } else if (warp == FWD_WARP && lane == 0 && !lead) {
      // --------------------------------------------------------- forwarder --
      // CTA 0's MMA issuer waits on its own barriers; the completion of each of this
      // CTA's loads is passed on to CTA 0's copy of the barrier, in load order.
      int ri = 0, qcnt = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        const int rs = kr % NRING, rpar = (kr / NRING) & 1;
        if (!(ok = mbar_wait_cl(ring_full(rs), rpar, abort_flag, status, tlim))) break;
        const int x = ring_x[rs];
        mbar_arrive_remote(mapa_shared(ring_empty(rs), 0));
        if (x >= n_items) break;
        const Item it = decode(a, x);
        if (!it.valid || it.n == 0) continue;
        const int qb = qcnt & 1;
        if (!(ok = mbar_wait_cl(q_full(qb), (qcnt >> 1) & 1, abort_flag, status, tlim))) break;
        mbar_arrive_remote(mapa_shared(q_full(qb), 0));
        ++qcnt;
        for (int i = 0; i < 2 * it.n; ++i, ++ri) {
          if (!(ok = mbar_wait_cl(full(ri), (ri / NST) & 1, abort_flag, status, tlim))) break;
          mbar_arrive_remote(mapa_shared(full(ri), 0));
        }
        if (!ok) break;
      }
    } else if (warp == MMA_WARP && lane == 0 && lead) {
      // ---------------------------------------------------------- MMA issue --
      constexpr uint32_t IS = idesc_bf16(2 * QT, BNK, 0);  // S = Q K^T, M = 256, both K-major
      constexpr uint32_t IPV = idesc_bf16(2 * QT, D, 1);   // O += P V, M = 256, V MN-major
      constexpr uint16_t BOTH = 3;                          // commit to both CTAs' barrier
      const uint32_t q_base = smem_u32(sm + L::Q);
      const uint32_t r_base = smem_u32(sm + L::RING);
      auto slot = [&](int i) { return r_base + (i % NST) * L::SLOT; };
      auto ring_wait = [&](int i) {
        return mbar_wait_cl(full(i), (i / NST) & 1, abort_flag, status, tlim);
      };
      // S(buffer sb) = Q(qb) K^T: A = this CTA's 128 Q rows (two 64-column boxes of 128
      // rows), B = its 64 keys of the tile (two 64-column boxes of 64 rows); each K step
      // of 16 columns moves 32 bytes inside a box, then to the next box.
      auto issue_S = [&](int sb, int qb, uint32_t kaddr) {
        const uint64_t da = sw128_desc(q_base + qb * L::QTILE, 16, 1024);
        const uint64_t db = sw128_desc(kaddr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = ((kk / 4) * L::QBOX + (kk % 4) * 32) >> 4;
          const uint32_t offb = ((kk / 4) * L::KBOX + (kk % 4) * 32) >> 4;
          umma2_ss(tmem + sb * BNK, da + offa, db + offb, IS, kk > 0);
        }
      };
      // O(ob) += P(sb) V: A = P in TMEM (over S(sb), 8 columns per K step of 16 keys),
      // B = this CTA's 64 d columns of the V tile (one box of 128 keys).
      auto issue_PV = [&](int ob, int sb, uint32_t vaddr, bool acc) {
        const uint64_t dv = sw128_desc(vaddr, L::SLOT, 1024);
#pragma unroll
        for (int kk = 0; kk < BNK / 16; ++kk)
          umma2_ts(tmem + TM_O + ob * D, tmem + sb * BNK + 8 * kk, dv + ((kk * 2048) >> 4), IPV,
                   (acc || kk > 0) ? 1u : 0u);
      };
      // Per key step t: P V(t), then S(t + 2) into the buffer S(t) and P(t) used.  One
      // commit point per step (after S(t + 2)): S(t + 2) ready, K(t + 2) and V(t)
      // free; the last two steps commit after P V (pv_last after the second-to-last,
      // O done after the last).  S(t + 1) done implies P V(t - 1) done, which the
      // softmax uses before it rescales O.
      int ri = 0, gs = 0, qcnt = 0, ocnt = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        const int rs = kr % NRING;
        if (!(ok = mbar_wait_cl(ring_full(rs), (kr / NRING) & 1, abort_flag, status, tlim))) break;
        const int x = ring_x[rs];
        mbar_arrive(ring_empty(rs));
        if (x >= n_items) break;
        const Item it = decode(a, x);
        if (!it.valid || it.n == 0) continue;
        const int n = it.n, qb = qcnt & 1, ob = ocnt & 1;
        if (!(ok = mbar_wait_cl(q_full(qb), (qcnt >> 1) & 1, abort_flag, status, tlim) && ring_wait(ri)))
          break;
        tc_fence_after();
        issue_S(gs & 1, qb, slot(ri));
        umma2_commit_mc(s_full(gs & 1), BOTH);
        umma2_commit_mc(empty(ri), BOTH);
        if (n >= 2) {
          if (!(ok = ring_wait(ri + 2))) break;
          tc_fence_after();
          issue_S((gs + 1) & 1, qb, slot(ri + 2));
          umma2_commit_mc(s_full((gs + 1) & 1), BOTH);
          umma2_commit_mc(empty(ri + 2), BOTH);
        }
        if (n <= 2) umma2_commit_mc(q_free(qb), BOTH);
        // the epilogue of this O buffer's previous item has read it
        if (!(ok = mbar_wait_cl(o_free(ob), ((ocnt >> 1) & 1) ^ 1, abort_flag, status, tlim))) break;
        for (int t = 0; t < n; ++t) {
          const int g = gs + t, sb = g & 1, iv = ri + 2 * t + 1;
          if (!(ok = ring_wait(iv) && mbar_wait_cl(p_ready(sb), (g >> 1) & 1, abort_flag, status, tlim)))
            break;
          tc_fence_after();
          issue_PV(ob, sb, slot(iv), t > 0);
          if (t + 2 < n) {
            const int ik = ri + 2 * (t + 2);
            if (!(ok = ring_wait(ik))) break;
            tc_fence_after();
            issue_S(sb, qb, slot(ik));
            umma2_commit_mc(s_full(sb), BOTH);
            umma2_commit_mc(empty(ik), BOTH);
            umma2_commit_mc(empty(iv), BOTH);
            if (t + 3 == n) umma2_commit_mc(q_free(qb), BOTH);
          } else {
            umma2_commit_mc(t + 1 == n ? o_full(ob) : pv_last, BOTH);
            umma2_commit_mc(empty(iv), BOTH);
          }
        }
        if (!ok) break;
        ri += 2 * n;
        gs += n;
        ++qcnt;
        ++ocnt;
      }
      umma2_commit_mc(drain, BOTH);  // every MMA issued above completes before TMEM is released
      mbar_drain_cl(drain, 0);
    } else if (warp == MMA_WARP && lane == 0) {
      mbar_drain_cl(drain, 0);  // CTA 1: CTA 0's MMAs into this tensor memory are done
    }
    __syncwarp();
  } else {
    setmaxnreg_inc();
    // -------------------------------------------------------------- softmax --
    // Warps 0-3: thread = row = TMEM lane, the whole 128-column row of each tile.
    // Warps 4-7 have no role (they complete the warpgroup for the register split).
    if (warp < 4) {
      const int r = warp * 32 + lane;  // row in this CTA's tile
      const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
      const float sl2 = a.sl2;
      int gs = 0, ocnt = 0, n2 = 0;
      bool ok = true;
      for (int kr = 0;; ++kr) {
        const int rs = kr % NRING;
        ok = mbar_wait_cl(ring_full(rs), (kr / NRING) & 1, abort_flag, status, tlim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const int x = ring_x[rs];
        __syncwarp();
        if (lane == 0) arrive_lead(ring_empty(rs));
        if (x >= n_items) break;
        const Item it = decode(a, x);
        if (!it.valid) continue;
        const int n = it.n, ob = ocnt & 1;
        const int rg = (int)rank * QT + r;  // row in the item
        const bool row_ok = rg < it.rows;
        const int* P = a.perm + (int64_t)it.br * a.NR;
        const int qp = __ldg(P + it.row0 + min(rg, it.rows - 1));
        const uint32_t tO = tmem + lane_off + TM_O + ob * D;
        float m_use = -INFINITY, l = 0.0f;
        int e = 0, t_in = 0;
        PlanEnt pe{};
        if (n > 0) pe = a.plan_ent[(int64_t)it.u * a.nseg];
        for (int t = 0; t < n; ++t) {
          const int g = gs + t, sb = g & 1;
          const uint32_t tS = tmem + lane_off + sb * BNK;
          // this row's keys in the tile: columns below c_hi (positions <= qp - w)
          int c_hi = BNK;
          const int valid = min(BNK, pe.cnt - t_in * BNK);
          const bool need_mask = t_in >= pe.nfull;
          if (need_mask) c_hi = upper_bound_g(P + pe.start + t_in * BNK, 0, valid, qp - a.w);
          if (++t_in * BNK >= pe.cnt && ++e < a.nseg) {
            t_in = 0;
            pe = a.plan_ent[(int64_t)it.u * a.nseg + e];
          }
          ok = mbar_wait_cl(s_full(sb), (uint32_t)((g >> 1) & 1), abort_flag, status, tlim);
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
          if (need_mask) {  // raw logits; the scale is positive, so the max commutes with it
            auto mask32 = [&](uint32_t(&xx)[32], int cb) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (cb + i >= c_hi) xx[i] = 0xff800000u;  // -inf
            };
            mask32(x0, 0);
            mask32(x1, 32);
            mask32(x2, 64);
            mask32(x3, 96);
          }
          // Row max, taken lazily: the exponentials use the running estimate m_use and
          // the tile's max is computed only while a row has none yet or when the
          // tile's exponentials sum past kSumCap (the tile is then redone with its
          // max).  P keeps its relative precision at any magnitude (bf16 has fp32's
          // exponent range), and O and l have headroom far above kSumCap * keys * |v|.
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
          // P (bf16 pairs) over the first 64 columns of this row's S, already in
          // registers: column 16k + i holds keys 32k + 2i and 32k + 2i + 1
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
          // O follows the new maximum once it holds every earlier P V: S(t + 1) done
          // implies P V(t - 1) done; at the last tile the pv_last commit says so.
          if (__any_sync(0xffffffffu, rescale && t > 0 && f != 0.0f)) {
            if (t + 1 < n)
              ok = mbar_wait_cl(s_full((g + 1) & 1), (uint32_t)(((g + 1) >> 1) & 1), abort_flag, status, tlim);
            else
              ok = mbar_wait_cl(pv_last, (uint32_t)(n2 & 1), abort_flag, status, tlim);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float gsc = (rescale && t > 0) ? f : 1.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t y[32];
              tmem_ld32(tO + 32 * c, y);
              tmem_ld_wait(y);
#pragma unroll
              for (int i = 0; i < 32; ++i) y[i] = __float_as_uint(__uint_as_float(y[i]) * gsc);
              tmem_st32(tO + 32 * c, y);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_lead(p_ready(sb));
        }
        if (!ok) break;
        if (n >= 2) ++n2;
        gs += n;
        // ---- epilogue: one softmax over the union = LSE merge with the window pass ----
        if (n > 0) {
          ok = mbar_wait_cl(o_full(ob), (uint32_t)((ocnt >> 1) & 1), abort_flag, status, tlim);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const int64_t orow = (((int64_t)it.b * a.N + qp) * a.H + it.h) * D;
        const int64_t lrow = ((int64_t)it.b * a.H + it.h) * a.N + qp;
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
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (n > 0) {  // this O buffer may take the item after next
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_lead(o_free(ob));
          ++ocnt;
        }
        if (row_ok && a.lse) a.lse[lrow] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA releases the pair's tensor memory while the other uses it
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc2(tmem, TMEM_COLS);
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

// Tensor map over `rows` rows of D bf16 values; box 64 columns x box_rows rows,
// 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool pair_engine_supported(const focus_params& p, const WsLayout& L) {
  return p.d_head == D && !L.group;
}

cudaError_t launch_attn_long_pair(const focus_params& p, const WsLayout& L, char* ws, bf16* o,
                                  float* lse, float scale, cudaStream_t s) {
  PairArgs a{};
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
  a.qtab = reinterpret_cast<const QBlock*>(ws + L.qtab);
  a.qtab_count = &reinterpret_cast<const WsHeader*>(ws)->qtab_count;
  a.plan_head = reinterpret_cast<const PlanHead*>(ws + L.plan_head);
  a.plan_ent = reinterpret_cast<const PlanEnt*>(ws + L.plan_ent);
  a.o_part = reinterpret_cast<const float*>(ws + L.olr);
  a.lse_part = reinterpret_cast<const float*>(ws + L.lselr);
  a.o = o;
  a.lse = lse;
  a.status = &reinterpret_cast<WsHeader*>(ws)->status;
  a.item_counter = &reinterpret_cast<WsHeader*>(ws)->item_counter[1];
  a.timeout_cycles = ptx::kTimeoutCycles;
  CUtensorMap mq, mk, mv;
  if (!make_rows_map(&mq, ws + L.qp, (int64_t)p.B * p.H * L.NR, QT) ||
      !make_rows_map(&mk, ws + L.kp, (int64_t)p.B * p.H_kv * L.NR, 64) ||
      !make_rows_map(&mv, ws + L.vp, (int64_t)p.B * p.H_kv * L.NR, BNK))
    return cudaErrorInvalidValue;
  const int n_items = a.qtab_cap * (p.H / p.R);
  if (n_items < 1) return cudaSuccess;
  const int smem = PairLayout::SMEM;
  cudaError_t e = cudaFuncSetAttribute(attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one pair per TPC that can hold one (persistent: the pairs draw the items)
  int clusters = 0;
  cfg.gridDim = dim3(2);
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, attn_pair, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorLaunchOutOfResources;
  if (clusters > n_items) clusters = n_items;
  cfg.gridDim = dim3(2 * clusters);
  return cudaLaunchKernelEx(&cfg, attn_pair, mq, mk, mv, a, n_items);
}

}  // namespace focus
