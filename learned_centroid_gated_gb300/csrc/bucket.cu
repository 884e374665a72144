// Bucketing of tokens by group bitmask, the long-range query-block schedule, and
// the permuted Q/K/V copies.
//
// Distant tokens attend only when their groups intersect ("Why Attend to
// Everything? Focus is the Key", gist.science technical summary, section 2,
// "Inference Efficiency (Top-k)"). Tokens are sorted stably by their mask
// VALUE (the exact k-subset of groups, ranked in colex order), so every segment
// holds tokens with one mask and ascending positions. A query segment S then
// attends to whole key segments T with mask(S) & mask(T) != 0: every key appears
// once in a query's candidate list, so the union softmax needs no deduplication,
// and the tiles inside a segment are dense.
//
// When C(K, top_k) is large (e.g. K = 32, top_k = 4 gives 35960 sets) the
// segments are too many and too small for dense tiles, so a second schedule keeps
// one position-ordered list per GROUP instead (a token appears in its top_k
// lists; rows per (b, rho) are N * top_k).  The attention kernel then counts a
// key only in the list of the lowest group it shares with the query, which keeps
// "each key once" without a per-set split.
#include "common.cuh"

namespace focus {
namespace {

// Colex rank of a k-subset given as a bitmask: sum_m C(c_m, m + 1) over the set
// bits c_0 < c_1 < ...  Returns -1 unless exactly top_k of the low K bits are set.
__device__ __forceinline__ int seg_of(uint32_t m, int K, int top_k) {
  if (K < 32 && (m >> K) != 0u) return -1;
  if (__popc(m) != top_k) return -1;
  int rank = 0, idx = 0;
  while (m) {
    const int c = __ffs(m) - 1;
    m &= m - 1;
    ++idx;
    rank += (int)binom(c, idx);
  }
  return rank;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

// Histogram of segment ids over one chunk of kChunk tokens. One warp per chunk,
// grid = (nchunk, B*R).  Invalid masks raise FOCUS_ERR_BOUNDS and count in segment 0.
__global__ void __launch_bounds__(32)
bucket_hist(int N, int K, int top_k, int nseg, const uint32_t* __restrict__ mask,
            int* __restrict__ hist, int* status) {
  extern __shared__ int cnt[];
  const int br = blockIdx.y, chunk = blockIdx.x, lane = threadIdx.x;
  for (int s = lane; s < nseg; s += 32) cnt[s] = 0;
  __syncwarp();
  const uint32_t* m = mask + (int64_t)br * N;
  const int n0 = chunk * kChunk;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int n = n0 + it * 32 + lane;
    int sg = -2;
    if (n < N) {
      sg = seg_of(m[n], K, top_k);
      if (sg < 0) {
        raise_status(status, FOCUS_ERR_BOUNDS);
        sg = 0;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, sg);
    if (sg >= 0 && (peers & lanemask_lt()) == 0u) cnt[sg] += __popc(peers);
    __syncwarp();
  }
  int* h = hist + ((int64_t)br * gridDim.x + chunk) * nseg;
  for (int s = lane; s < nseg; s += 32) h[s] = cnt[s];
}

// Segment offsets and per-chunk scatter bases. grid = B*R, 1024 threads (>= nseg).
__global__ void __launch_bounds__(1024)
bucket_scan(int nseg, int nchunk, const int* __restrict__ hist, int* __restrict__ seg_off,
            int* __restrict__ cbase) {
  __shared__ int wsum[32];
  const int br = blockIdx.x, s = threadIdx.x;
  const int* h = hist + (int64_t)br * nchunk * nseg;
  int t = 0;
  if (s < nseg)
    for (int c = 0; c < nchunk; ++c) t += h[(int64_t)c * nseg + s];
  // exclusive block scan of t over s
  const int lane = s & 31, wid = s >> 5;
  int x = t;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int v = wsum[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  const int excl = x - t + (wid > 0 ? wsum[wid - 1] : 0);
  if (s < nseg) {
    seg_off[(int64_t)br * (nseg + 1) + s] = excl;
    if (s == nseg - 1) seg_off[(int64_t)br * (nseg + 1) + nseg] = excl + t;
    int run = excl;
    int* cb = cbase + (int64_t)br * nchunk * nseg;
    for (int c = 0; c < nchunk; ++c) {
      cb[(int64_t)c * nseg + s] = run;
      run += h[(int64_t)c * nseg + s];
    }
  }
}

// Stable scatter: perm[seg_base + rank] = n. Same chunking as bucket_hist.
__global__ void __launch_bounds__(32)
bucket_scatter(int N, int K, int top_k, int nseg, const uint32_t* __restrict__ mask,
               const int* __restrict__ cbase, int* __restrict__ perm, int* status) {
  extern __shared__ int cur[];
  const int br = blockIdx.y, chunk = blockIdx.x, lane = threadIdx.x;
  const int* cb = cbase + ((int64_t)br * gridDim.x + chunk) * nseg;
  for (int s = lane; s < nseg; s += 32) cur[s] = cb[s];
  __syncwarp();
  const uint32_t* m = mask + (int64_t)br * N;
  int* P = perm + (int64_t)br * N;
  const int n0 = chunk * kChunk;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int n = n0 + it * 32 + lane;
    int sg = -2;
    if (n < N) {
      sg = seg_of(m[n], K, top_k);
      if (sg < 0) sg = 0;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, sg);
    if (sg >= 0) {
      const int dst = cur[sg] + __popc(peers & lanemask_lt());
      if (FOCUS_IN_BOUNDS(dst >= 0 && dst < N, status)) P[dst] = n;
    }
    __syncwarp();
    if (sg >= 0 && (peers & lanemask_lt()) == 0u) cur[sg] += __popc(peers);
    __syncwarp();
  }
}

// Group-list schedule.  A mask with the wrong number of bits (or bits >= K) is
// filed under groups 0..top_k-1 so that every token still fills top_k rows.
__device__ __forceinline__ uint32_t group_bits(uint32_t m, int K, int top_k, int* status) {
  if ((K < 32 && (m >> K) != 0u) || __popc(m) != top_k) {
    if (status) raise_status(status, FOCUS_ERR_BOUNDS);
    return top_k >= 32 ? 0xffffffffu : (1u << top_k) - 1u;
  }
  return m;
}

// List sizes over one chunk of kChunk tokens; one warp per chunk, lane g counts
// group g.  grid = (nchunk, B*R); hist layout as bucket_hist with nseg = K.
__global__ void __launch_bounds__(32)
group_hist(int N, int K, int top_k, const uint32_t* __restrict__ mask, int* __restrict__ hist,
           int* status) {
  const int br = blockIdx.y, chunk = blockIdx.x, lane = threadIdx.x;
  const uint32_t* m = mask + (int64_t)br * N;
  const int n0 = chunk * kChunk;
  int cnt = 0;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int n = n0 + it * 32 + lane;
    const uint32_t mm = n < N ? group_bits(m[n], K, top_k, status) : 0u;
    for (int g = 0; g < K; ++g) {
      const unsigned bal = __ballot_sync(0xffffffffu, (mm >> g) & 1u);
      if (lane == g) cnt += __popc(bal);
    }
  }
  if (lane < K) hist[((int64_t)br * gridDim.x + chunk) * K + lane] = cnt;
}

// Stable scatter into the K lists: perm[list base + rank] = n, and the token's
// mask beside it (pmask), which the attention kernel reads for the lowest-group
// test.  Same chunking as group_hist; lane g carries list g's cursor.
__global__ void __launch_bounds__(32)
group_scatter(int N, int NR, int K, int top_k, const uint32_t* __restrict__ mask,
              const int* __restrict__ cbase, int* __restrict__ perm, uint32_t* __restrict__ pmask) {
  const int br = blockIdx.y, chunk = blockIdx.x, lane = threadIdx.x;
  int cur = lane < K ? cbase[((int64_t)br * gridDim.x + chunk) * K + lane] : 0;
  const uint32_t* m = mask + (int64_t)br * N;
  int* P = perm + (int64_t)br * NR;
  uint32_t* PM = pmask + (int64_t)br * NR;
  const int n0 = chunk * kChunk;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int n = n0 + it * 32 + lane;
    const uint32_t mm = n < N ? group_bits(m[n], K, top_k, nullptr) : 0u;
    for (int g = 0; g < K; ++g) {
      const bool in = (mm >> g) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      const int base = __shfl_sync(0xffffffffu, cur, g);
      if (in) {
        const int dst = base + __popc(bal & lanemask_lt());
        P[dst] = n;
        PM[dst] = mm;
      }
      if (lane == g) cur += __popc(bal);
    }
  }
}

// Long-range schedule: one entry per query block of bm rows inside a segment,
// ordered by descending position of the block's last row (the blocks with the most
// candidate keys start first).  Single CTA.
constexpr int kTabThreads = 1024;
constexpr int kTabBuckets = 4096;

__global__ void __launch_bounds__(kTabThreads)
build_qtab(int N, int NR, int nseg, int BR, int bm, const int* __restrict__ seg_off, const int* __restrict__ perm,
           int* __restrict__ entoff, QBlock* __restrict__ qtab, int* __restrict__ qtab_count) {
  __shared__ int bucket[kTabBuckets];
  __shared__ int wsum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nitems = BR * nseg;
  // exclusive scan of block counts over (br, seg)
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nitems; base += kTabThreads) {
    const int it = base + tid;
    int c = 0;
    if (it < nitems) {
      const int br = it / nseg, s = it % nseg;
      const int* so = seg_off + (int64_t)br * (nseg + 1);
      const int cnt = so[s + 1] - so[s];
      c = (cnt + bm - 1) / bm;
    }
    int x = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int v = wsum[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      wsum[lane] = v;
    }
    __syncthreads();
    const int excl = carry + x - c + (wid > 0 ? wsum[wid - 1] : 0);
    if (it < nitems) entoff[it] = excl;
    __syncthreads();
    if (tid == kTabThreads - 1) carry = excl + c;
    __syncthreads();
  }
  const int E = carry;
  if (tid == 0) {
    entoff[nitems] = E;
    *qtab_count = E;
  }
  int shift = 0;
  while (((N - 1) >> shift) >= kTabBuckets) ++shift;
  for (int i = tid; i < kTabBuckets; i += kTabThreads) bucket[i] = 0;
  __syncthreads();
  // pass 1: histogram of sort keys; pass 2: scatter
  for (int pass = 0; pass < 2; ++pass) {
    for (int e = tid; e < E; e += kTabThreads) {
      int lo = 0, hi = nitems - 1;  // last item with entoff <= e
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (entoff[mid] <= e) lo = mid; else hi = mid - 1;
      }
      const int br = lo / nseg, s = lo % nseg;
      const int t = e - entoff[lo];
      const int* so = seg_off + (int64_t)br * (nseg + 1);
      const int cnt = so[s + 1] - so[s];
      const int row0 = so[s] + t * bm;
      const int rows = min(bm, cnt - t * bm);
      const int last = perm[(int64_t)br * NR + row0 + rows - 1];
      const int key = (N - 1 - last) >> shift;
      if (pass == 0) {
        atomicAdd(&bucket[key], 1);
      } else {
        const int dst = atomicAdd(&bucket[key], 1);
        qtab[dst] = QBlock{br, s, row0, rows};
      }
    }
    __syncthreads();
    if (pass == 0) {  // exclusive scan of the buckets, in place (single thread chunks)
      constexpr int per = kTabBuckets / kTabThreads;
      int loc[per], sum = 0;
      for (int j = 0; j < per; ++j) {
        loc[j] = bucket[tid * per + j];
        sum += loc[j];
      }
      int x = sum;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[wid] = x;
      __syncthreads();
      if (wid == 0) {
        int v = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += y;
        }
        wsum[lane] = v;
      }
      __syncthreads();
      int run = x - sum + (wid > 0 ? wsum[wid - 1] : 0);
      for (int j = 0; j < per; ++j) {
        bucket[tid * per + j] = run;
        run += loc[j];
      }
      __syncthreads();
    }
  }
}

// First index in P[lo, hi) whose value exceeds x (P ascending).
__device__ __forceinline__ int upper_bound_pos(const int* __restrict__ P, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Long-range plan: for query block u (segment S, positions p_lo..p_hi), every
// segment T with mask(S) & mask(T) != 0 and keys at pos <= p_hi - w, in segment
// order; with group lists, the block's own list only.  One warp per block; lanes
// take segments in parallel.
__global__ void __launch_bounds__(32)
build_plan(int N, int NR, int w, int nseg, int group, const int* __restrict__ seg_off,
           const int* __restrict__ perm, const uint32_t* __restrict__ mask,
           const QBlock* __restrict__ qtab, const int* __restrict__ qtab_count,
           PlanHead* __restrict__ heads, PlanEnt* __restrict__ ents) {
  const int u = blockIdx.x, lane = threadIdx.x;
  if (u >= *qtab_count) return;
  const QBlock e = qtab[u];
  const int* P = perm + (int64_t)e.br * NR;
  const int* SO = seg_off + (int64_t)e.br * (nseg + 1);
  const uint32_t* M = mask + (int64_t)e.br * N;
  const int p_lo = __ldg(P + e.row0), p_hi = __ldg(P + e.row0 + e.rows - 1);
  const uint32_t mS = group ? 0u : __ldg(M + p_lo);
  PlanEnt* out = ents + (int64_t)u * nseg;
  int n_ent = 0, n_tiles = 0;
  for (int T0 = 0; T0 < nseg; T0 += 32) {
    const int T = T0 + lane;
    bool ok = false;
    PlanEnt pe{0, 0, 0, 0};
    if (T < nseg) {
      const int s0 = __ldg(SO + T), s1 = __ldg(SO + T + 1);
      const bool compatible = group ? T == e.seg : (s1 > s0 && (__ldg(M + __ldg(P + s0)) & mS));
      if (s1 > s0 && compatible) {
        const int hi = upper_bound_pos(P, s0, s1, p_hi - w) - s0;
        if (hi > 0) {
          ok = true;
          pe.start = s0;
          pe.cnt = hi;
          pe.nfull = (upper_bound_pos(P, s0, s1, p_lo - w) - s0) / kKeyTile;
        }
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (ok) out[n_ent + __popc(bal & lanemask_lt())] = pe;
    n_ent += __popc(bal);
    int tiles = ok ? (pe.cnt + kKeyTile - 1) / kKeyTile : 0;
    for (int o = 16; o > 0; o >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
    n_tiles += tiles;
  }
  if (lane == 0) heads[u] = PlanHead{n_ent, n_tiles, 0, 0};
}

// Backward plans of 128-row block u (segment S, positions p_lo..p_hi), over the
// compatible segments T in segment order (exact-set schedule; with group lists the
// block's own list only):
//   query-major (dQ):  keys of T with pos <= p_hi - w, in tiles of kBwdKeyTile;
//                      PlanEnt.nfull = keys with pos <= p_lo - w (need no mask);
//   key-major (dK, dV): queries of T with pos >= p_lo + w, in tiles of kBwdQryTile.
// One warp per block; lanes take segments in parallel.
__global__ void __launch_bounds__(32)
build_plan_bwd(int N, int NR, int w, int nseg, int group, const int* __restrict__ seg_off,
               const int* __restrict__ perm, const uint32_t* __restrict__ mask,
               const QBlock* __restrict__ qtab, const int* __restrict__ qtab_count,
               PlanHead* __restrict__ qheads, PlanEnt* __restrict__ qents,
               PlanHead* __restrict__ rheads, PlanEnt* __restrict__ rents) {
  const int u = blockIdx.x, lane = threadIdx.x;
  if (u >= *qtab_count) return;
  const QBlock e = qtab[u];
  const int* P = perm + (int64_t)e.br * NR;
  const int* SO = seg_off + (int64_t)e.br * (nseg + 1);
  const uint32_t* M = mask + (int64_t)e.br * N;
  const int p_lo = __ldg(P + e.row0), p_hi = __ldg(P + e.row0 + e.rows - 1);
  const uint32_t mS = group ? 0u : __ldg(M + p_lo);
  PlanEnt* qo = qents + (int64_t)u * nseg;
  PlanEnt* ro = rents + (int64_t)u * nseg;
  int nq = 0, nr = 0, tq = 0, tr = 0;
  for (int T0 = 0; T0 < nseg; T0 += 32) {
    const int T = T0 + lane;
    PlanEnt qe{0, 0, 0, 0}, re{0, 0, 0, 0};
    bool qok = false, rok = false;
    if (T < nseg) {
      const int s0 = __ldg(SO + T), s1 = __ldg(SO + T + 1);
      const bool compatible = group ? T == e.seg : (s1 > s0 && (__ldg(M + __ldg(P + s0)) & mS));
      if (s1 > s0 && compatible) {
        const int hi = upper_bound_pos(P, s0, s1, p_hi - w) - s0;
        if (hi > 0) {
          qok = true;
          qe.start = s0;
          qe.cnt = hi;
          qe.nfull = upper_bound_pos(P, s0, s1, p_lo - w) - s0;
        }
        const int lo = upper_bound_pos(P, s0, s1, p_lo + w - 1);
        if (lo < s1) {
          rok = true;
          re.start = lo;
          re.cnt = s1 - lo;
        }
      }
    }
    unsigned bal = __ballot_sync(0xffffffffu, qok);
    if (qok) qo[nq + __popc(bal & lanemask_lt())] = qe;
    nq += __popc(bal);
    bal = __ballot_sync(0xffffffffu, rok);
    if (rok) ro[nr + __popc(bal & lanemask_lt())] = re;
    nr += __popc(bal);
    int a = qok ? (qe.cnt + kBwdKeyTile - 1) / kBwdKeyTile : 0;
    int c = rok ? (re.cnt + kBwdQryTile - 1) / kBwdQryTile : 0;
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    tq += a;
    tr += c;
  }
  if (lane == 0) {
    qheads[u] = PlanHead{nq, tq, 0, 0};
    rheads[u] = PlanHead{nr, tr, 0, 0};
  }
}

// Permuted, head-major copies: Qp[b][h][n'][:] = q[b][perm[n']][h][:] for the heads
// of routing head rho, and likewise K/V for its KV heads; NR permuted rows per
// (b, rho).  One CTA per permuted row.
__global__ void __launch_bounds__(256)
permute_qkv(int N, int NR, int H, int H_kv, int R, int d, const int* __restrict__ perm,
            const uint4* __restrict__ q, const uint4* __restrict__ k, const uint4* __restrict__ v,
            uint4* __restrict__ qp, uint4* __restrict__ kp, uint4* __restrict__ vp, int* status) {
  const int64_t row = blockIdx.x;  // (b * R + rho) * NR + n'
  const int br = (int)(row / NR), np = (int)(row % NR);
  const int b = br / R, rho = br % R;
  const int n = perm[row];
  if (!FOCUS_IN_BOUNDS(n >= 0 && n < N, status)) return;
  const int hq = H / R, hkv = H_kv / R;
  const int vec = d / 8;  // uint4 per head row
  const int nq = hq * vec, nk = hkv * vec, total = nq + 2 * nk;
  // Up to four 16-byte loads in flight per thread before their stores.
  constexpr int U = 4;
  for (int base = threadIdx.x; base < total; base += U * blockDim.x) {
    uint4 val[U];
    int64_t dst[U];
    int which[U];  // 0 = Q, 1 = K, 2 = V, -1 = past the end
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * blockDim.x;
      which[u] = -1;
      if (i >= total) continue;
      if (i < nq) {
        const int hh = rho * hq + i / vec, c = i % vec;
        which[u] = 0;
        dst[u] = (((int64_t)b * H + hh) * NR + np) * vec + c;
        val[u] = q[(((int64_t)b * N + n) * H + hh) * vec + c];
      } else {
        const int j = (i - nq) % nk;
        const int hh = rho * hkv + j / vec, c = j % vec;
        const int64_t src = (((int64_t)b * N + n) * H_kv + hh) * vec + c;
        which[u] = i < nq + nk ? 1 : 2;
        dst[u] = (((int64_t)b * H_kv + hh) * NR + np) * vec + c;
        val[u] = which[u] == 1 ? k[src] : v[src];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (which[u] == 0) qp[dst[u]] = val[u];
      else if (which[u] == 1) kp[dst[u]] = val[u];
      else if (which[u] == 2) vp[dst[u]] = val[u];
    }
  }
}

}  // namespace

cudaError_t launch_bucket(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                          cudaStream_t s) {
  const int BR = p.B * p.R;
  int* status = &reinterpret_cast<WsHeader*>(ws)->status;
  int* hist = reinterpret_cast<int*>(ws + L.hist);
  int* segoff = reinterpret_cast<int*>(ws + L.segoff);
  int* cbase = reinterpret_cast<int*>(ws + L.cbase);
  int* perm = reinterpret_cast<int*>(ws + L.perm);
  dim3 grid(L.nchunk, BR);
  if (L.group) {
    uint32_t* pmask = reinterpret_cast<uint32_t*>(ws + L.pmask);
    group_hist<<<grid, 32, 0, s>>>(p.N, p.K, p.top_k, mask, hist, status);
    bucket_scan<<<BR, 1024, 0, s>>>(L.nseg, L.nchunk, hist, segoff, cbase);
    group_scatter<<<grid, 32, 0, s>>>(p.N, L.NR, p.K, p.top_k, mask, cbase, perm, pmask);
    return cudaGetLastError();
  }
  const size_t shm = sizeof(int) * L.nseg;
  bucket_hist<<<grid, 32, shm, s>>>(p.N, p.K, p.top_k, L.nseg, mask, hist, status);
  bucket_scan<<<BR, 1024, 0, s>>>(L.nseg, L.nchunk, hist, segoff, cbase);
  bucket_scatter<<<grid, 32, shm, s>>>(p.N, p.K, p.top_k, L.nseg, mask, cbase, perm, status);
  return cudaGetLastError();
}

cudaError_t launch_qtab(const focus_params& p, const WsLayout& L, char* ws, int block_rows,
                        cudaStream_t s) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  build_qtab<<<1, kTabThreads, 0, s>>>(p.N, L.NR, L.nseg, p.B * p.R, block_rows,
                                       reinterpret_cast<int*>(ws + L.segoff),
                                       reinterpret_cast<int*>(ws + L.perm),
                                       reinterpret_cast<int*>(ws + L.entoff),
                                       reinterpret_cast<QBlock*>(ws + L.qtab), &hdr->qtab_count);
  return cudaGetLastError();
}

cudaError_t launch_plan(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                        int block_rows, cudaStream_t s) {
  const int cap = p.B * p.R * ((L.NR + block_rows - 1) / block_rows + L.nseg);
  build_plan<<<cap, 32, 0, s>>>(p.N, L.NR, p.w, L.nseg, L.group,
                                reinterpret_cast<const int*>(ws + L.segoff),
                                reinterpret_cast<const int*>(ws + L.perm), mask,
                                reinterpret_cast<const QBlock*>(ws + L.qtab),
                                &reinterpret_cast<const WsHeader*>(ws)->qtab_count,
                                reinterpret_cast<PlanHead*>(ws + L.plan_head),
                                reinterpret_cast<PlanEnt*>(ws + L.plan_ent));
  return cudaGetLastError();
}

cudaError_t launch_permute(const focus_params& p, const WsLayout& L, const bf16* q, const bf16* k,
                           const bf16* v, char* ws, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.R * L.NR;
  permute_qkv<<<(unsigned)rows, 256, 0, s>>>(
      p.N, L.NR, p.H, p.H_kv, p.R, p.d_head, reinterpret_cast<const int*>(ws + L.perm),
      reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k),
      reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(ws + L.qp),
      reinterpret_cast<uint4*>(ws + L.kp), reinterpret_cast<uint4*>(ws + L.vp),
      &reinterpret_cast<WsHeader*>(ws)->status);
  return cudaGetLastError();
}

cudaError_t launch_plan_bwd(const focus_params& p, const WsLayout& L, const uint32_t* mask, char* ws,
                            PlanHead* qheads, PlanEnt* qents, PlanHead* rheads, PlanEnt* rents,
                            cudaStream_t s) {
  build_plan_bwd<<<L.qtab_cap, 32, 0, s>>>(p.N, L.NR, p.w, L.nseg, L.group,
                                           reinterpret_cast<const int*>(ws + L.segoff),
                                           reinterpret_cast<const int*>(ws + L.perm), mask,
                                           reinterpret_cast<const QBlock*>(ws + L.qtab),
                                           &reinterpret_cast<const WsHeader*>(ws)->qtab_count,
                                           qheads, qents, rheads, rents);
  return cudaGetLastError();
}

}  // namespace focus
