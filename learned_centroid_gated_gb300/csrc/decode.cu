// Decode: attention of the newest token of each sequence (position N - 1) over its
// cache, on the same union set as the forward pass ("Why Attend to Everything?
// Focus is the Key", gist.science technical summary, section 2, "Core Architecture"
// and "Inference Efficiency (Top-k)": window keys with exact softmax plus distant
// keys that share a group).
//
// The decode step is memory-bound (each allowed key's K and V rows are read once per
// KV head).  It runs as independent warps, each streaming the allowed keys of one
// slice of the cache through shared memory:
//   decode_split    one warp (a CTA of its own) per (slice of the cache, KV head, up
//                   to kDecHeads of that KV head's query heads), one wave of warps in
//                   all.  It compacts the slice's allowed keys (window, or mask
//                   overlap) block by block, the next block's mask words loading while
//                   the current one is compacted; streams tiles of kDecTile keys' K and
//                   V rows into a kDecStages-deep shared-memory ring with 16-byte
//                   asynchronous copies (a warp instruction moves whole rows; one bulk
//                   copy per 256-byte row measured a third slower, bound by the copy
//                   engine's per-copy cost); and keeps an online softmax over the
//                   tiles.  A tile's two products (scores of the warp's query heads,
//                   then P V) are register-fragment MMAs (m16n8k16, bf16 in, fp32 sums,
//                   P rounded to bf16 as in the forward pass): one warp instruction per
//                   16 x 8 x 16 block keeps the instruction count per byte low enough
//                   for the loads to stay the bound (with scalar fp32 FMAs the warps
//                   were issue-bound at about a third of the memory bandwidth).  It
//                   writes the slice's (max, sum, acc) per query head.  No CTA-wide
//                   barrier: each warp's loads stay in flight while it computes.
//                   (Interleaving the slices' blocks to spread the dense window over
//                   the warps measured slower: the contiguous slices keep the KV heads'
//                   warps on the same tokens at the same time.)
//   decode_combine  merges the slices of one (batch, head) by their maxima: O, LSE.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace focus {
namespace {

using namespace ptx;

constexpr int kDecTile = 16;           // keys per pipeline tile (one MMA reduction step)
constexpr int kDecStages = 3;          // tiles in the shared-memory ring
constexpr int kDecHeads = 8;           // most query heads per warp (rows of the MMA tile)
constexpr int kDecBlock = 256;         // raw keys per compaction block (8 mask words per lane)
constexpr int kDecMinSlice = 256;      // fewest raw keys per slice
constexpr int kDecTargetWarps = 1216;  // warps per launch: one wave of 8 per SM on 152 SMs
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Per-warp shared memory (bytes): kDecStages tiles of kDecTile K rows then kDecTile V
// rows, each row padded by 16 bytes so that the eight rows one ldmatrix phase reads
// start in different banks; the compacted key list; the keys per stage.
template <int D>
struct DecLayout {
  static constexpr int ROW = 2 * D + 16;
  static constexpr int STAGE = 2 * kDecTile * ROW;
  static constexpr int OFF_IDX = kDecStages * STAGE;
  static constexpr int OFF_CNT = OFF_IDX + kDecBlock * 4;
  static constexpr int BYTES = (OFF_CNT + kDecStages * 4 + 15) / 16 * 16;
  static_assert(ROW % 16 == 0 && STAGE % 16 == 0, "16-byte aligned rows");
};

__device__ __forceinline__ unsigned lanemask_lt_dec() {
  unsigned r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

// Four 8x8 bf16 matrices from shared memory (lane L gives the row address of
// matrix L / 8); .trans delivers them transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col), one warp.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int P>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(P) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&t);
}

// Lane (g, t) = (lane / 4, lane % 4) of the MMA fragments.  Scores S^T = q K^T: rows =
// query heads (g < nh; rows g + 8 are zero), columns = the tile's keys (two 8-key
// halves), reduction over d; the lane holds head g's scores of keys 2t, 2t + 1,
// 8 + 2t, 9 + 2t, which are exactly its B operand of O^T = V^T P^T (rows = d,
// columns = heads, reduction over the keys), so P never leaves the registers.
template <int D>
__global__ void __launch_bounds__(32)
decode_split(int N, int H, int H_kv, int R, int w, int B, int nsl, int nsl1, int s1, int s2,
             float sl2,
             const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
             const uint32_t* __restrict__ mask, float2* __restrict__ part_ml,
             float* __restrict__ part_acc) {
  using L = DecLayout<D>;
  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x, g = lane >> 2, t4 = lane & 3;
  const int gq = H / H_kv, nhg = (gq + kDecHeads - 1) / kDecHeads;
  int item = blockIdx.x;  // ((slice index * B + b) * H_kv + kvh) * nhg + hg
  const int hg = item % nhg;
  item /= nhg;
  const int kvh = item % H_kv;
  item /= H_kv;
  const int b = item % B, sl = item / B;
  const int h0 = kvh * gq + hg * kDecHeads, nh = min(kDecHeads, gq - hg * kDecHeads);
  const int rho = kvh / (H_kv / R);
  const int i = N - 1;
  const uint32_t* M = mask + ((int64_t)b * R + rho) * N;
  const uint32_t mq = __ldg(M + i);

  int* idx = reinterpret_cast<int*>(smem + L::OFF_IDX);
  int* cnt = reinterpret_cast<int*>(smem + L::OFF_CNT);
  const uint32_t stage0 = smem_u32(smem);

  // Rows of a partial tile beyond its keys keep older rows; zero them once so that
  // they are finite (their probabilities are exactly zero).
  for (int o = 16 * lane; o < kDecStages * L::STAGE; o += 512)
    *reinterpret_cast<uint4*>(smem + o) = make_uint4(0u, 0u, 0u, 0u);
  // q fragments (A of the scores): head g, k-step c: columns 16c + 2t (+1), 16c + 2t + 8 (+9)
  uint32_t qa[D / 16][2];
  {
    const int hq = g < nh ? h0 + g : h0;
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(q + ((int64_t)b * H + hq) * D);
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      qa[c][0] = g < nh ? __ldg(qr + 8 * c + t4) : 0u;
      qa[c][1] = g < nh ? __ldg(qr + 8 * c + 4 + t4) : 0u;
    }
  }

  // PDL: the combine kernel may be scheduled now; it waits for this grid's results.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- compaction of the allowed keys of keys [js, je), one block of kDecBlock raw
  // keys at a time; tiles of kDecTile keys are issued from a block's list.  Slices
  // 0 .. nsl1-1 cover the keys before the window (s1 keys each), the rest cover the
  // window (s2 keys each, all of them allowed).
  const int nw = max(0, N - w);
  const int js = sl < nsl1 ? sl * s1 : nw + (sl - nsl1) * s2;
  const int je = sl < nsl1 ? min(nw, js + s1) : min(N, js + s2);
  int jb = js, ncomp = 0, pos = 0;  // next block; keys in the list; keys issued
  constexpr int MW = kDecBlock / 32;
  uint32_t mw[MW];  // mask words of block jb, loaded one block ahead
#pragma unroll
  for (int t = 0; t < MW; ++t) {
    const int j = jb + 32 * t + lane;
    mw[t] = j < je ? __ldg(M + j) : 0u;
  }
  const int64_t rs = (int64_t)H_kv * D;  // elements per token in the caches
  const bf16* kb = k + (int64_t)b * N * rs + (int64_t)kvh * D;
  const bf16* vb = v + (int64_t)b * N * rs + (int64_t)kvh * D;

  // Fills stage s with the next tile of allowed keys; false when the slice is done.
  auto issue = [&](int s) -> bool {
    while (pos >= ncomp) {
      if (jb >= je) return false;
      ncomp = 0;
#pragma unroll
      for (int t = 0; t < MW; ++t) {
        const int j = jb + 32 * t + lane;
        const bool ok = j < je && (i - j < w || (mw[t] & mq) != 0u);
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) idx[ncomp + __popc(bal & lanemask_lt_dec())] = j;
        ncomp += __popc(bal);
      }
      jb += kDecBlock;
#pragma unroll
      for (int t = 0; t < MW; ++t) {  // the next block's words, in flight meanwhile
        const int j = jb + 32 * t + lane;
        mw[t] = j < je ? __ldg(M + j) : 0u;
      }
      pos = 0;
      __syncwarp();
    }
    const int n = min(kDecTile, ncomp - pos);
    if (lane == 0) cnt[s] = n;
    // 16-byte asynchronous copies, one row segment per lane: CH lanes cover a row, so
    // one warp instruction moves 32 / CH whole rows
    constexpr int CH = D / 8, RPI = 32 / CH;
    const int ch = lane % CH;
    const uint32_t st = stage0 + s * L::STAGE + 16 * ch;
    for (int rr = lane / CH; rr < n; rr += RPI) {
      const int64_t j = idx[pos + rr];
      cp_async16(st + rr * L::ROW, kb + j * rs + 8 * ch);
      cp_async16(st + (kDecTile + rr) * L::ROW, vb + j * rs + 8 * ch);
    }
    cp_async_commit();
    pos += n;
    return true;
  };

  float m = -INFINITY, l = 0.0f;  // head g's running maximum (log2 domain) and sum
  float acc[D / 16][4];           // O^T: d = 16 mt + g (+8), heads 2t, 2t + 1
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;
  __syncwarp();  // zeroed stages before the first copy
  int issued = 0;  // one copy group per stage and per refill, empty or not
  for (int s = 0; s < kDecStages; ++s) {
    if (issue(s)) ++issued;
    else cp_async_commit();
  }
  // ldmatrix row address of this lane: matrices (keys 0-7 | 8-15) x (columns +0 | +8)
  const uint32_t loff = ((lane & 7) + ((lane >> 4) << 3)) * L::ROW + ((lane >> 3) & 1) * 16;
  for (int t = 0; t < issued; ++t) {
    const int s = t % kDecStages;
    cp_async_wait<kDecStages - 1>();  // tile t's group has landed (this lane's copies)
    __syncwarp();                     // ... and every lane's
    const int n = cnt[s];
    const uint32_t kst = stage0 + s * L::STAGE + loff, vst = kst + kDecTile * L::ROW;
    float c0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4(kst + 32 * c, r0, r1, r2, r3);
      mma_bf16(c0, qa[c][0], 0u, qa[c][1], 0u, r0, r1);
      mma_bf16(c1, qa[c][0], 0u, qa[c][1], 0u, r2, r3);
    }
    // online softmax of head g over keys 2t, 2t+1, 8+2t, 9+2t (log2 domain)
    float sv[4] = {c0[0] * sl2, c0[1] * sl2, c1[0] * sl2, c1[1] * sl2};
    sv[0] = 2 * t4 < n ? sv[0] : -INFINITY;
    sv[1] = 2 * t4 + 1 < n ? sv[1] : -INFINITY;
    sv[2] = 2 * t4 + 8 < n ? sv[2] : -INFINITY;
    sv[3] = 2 * t4 + 9 < n ? sv[3] : -INFINITY;
    float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float mn = fmaxf(m, mt);
    const float corr = ex2(m - mn);
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = ex2(sv[e] - mn);
    l = l * corr + ((p[0] + p[1]) + (p[2] + p[3]));
    m = mn;
    // rescale the accumulator columns (heads 2t, 2t + 1: their statistics sit in lanes 8t, 8t + 4)
    const float ca = __shfl_sync(0xffffffffu, corr, 8 * t4);
    const float cb = __shfl_sync(0xffffffffu, corr, 8 * t4 + 4);
    const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
#pragma unroll
    for (int mi = 0; mi < D / 16; ++mi) {
      acc[mi][0] *= ca;
      acc[mi][1] *= cb;
      acc[mi][2] *= ca;
      acc[mi][3] *= cb;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vst + 32 * mi, a0, a1, a2, a3);
      mma_bf16(acc[mi], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();  // every lane is done with the stage
    if (issue(s)) ++issued;
    else cp_async_commit();
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  if (t4 == 0 && g < nh) {
    const int64_t slot = ((int64_t)b * H + h0 + g) * nsl + sl;
    part_ml[slot] = make_float2(m, l);
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int hh = 2 * t4 + e;
    if (hh < nh) {
      float* dst = part_acc + (((int64_t)b * H + h0 + hh) * nsl + sl) * D;
#pragma unroll
      for (int mi = 0; mi < D / 16; ++mi) {
        dst[16 * mi + g] = acc[mi][e];
        dst[16 * mi + g + 8] = acc[mi][2 + e];
      }
    }
  }
}

// Merge the slices of one (batch, head): grid = B * H, 32 warps; warp g folds the
// slices c = g (mod 32) into a running (max, sum, acc) (lane: D / 32 columns; the
// loads of 8 slices in flight together), then warp 0 folds the 32 warps' results in
// order.  Launched as a programmatic dependent
// of decode_split: it waits for that grid's results before reading them.
constexpr int kCombWarps = 32;
template <int D>
__global__ void __launch_bounds__(32 * kCombWarps)
decode_combine(int nch, const float2* __restrict__ part_ml, const float* __restrict__ part_acc,
               bf16* __restrict__ o, float* __restrict__ lse) {
  constexpr int CPL = D / 32;
  __shared__ float wm[kCombWarps], wl[kCombWarps];
  __shared__ __align__(16) float wacc[kCombWarps][D];
  const int bh = blockIdx.x, g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float m = -INFINITY, l = 0.0f, a[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) a[e] = 0.0f;
  constexpr int U = 8;  // slices whose loads are issued together
  for (int c0 = g; c0 < nch; c0 += U * kCombWarps) {
    float2 x[U];
    float v[U][CPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * kCombWarps;
      const int64_t slot = (int64_t)bh * nch + min(c, nch - 1);
      x[u] = c < nch ? part_ml[slot] : make_float2(-INFINITY, 0.0f);
      if constexpr (CPL == 4) {
        const float4 t = *reinterpret_cast<const float4*>(part_acc + slot * D + 4 * lane);
        v[u][0] = t.x, v[u][1] = t.y, v[u][2] = t.z, v[u][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(part_acc + slot * D + 2 * lane);
        v[u][0] = t.x, v[u][1] = t.y;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (x[u].y > 0.0f) {  // a slice without allowed keys holds (-inf, 0)
        const float mn = fmaxf(m, x[u].x), f0 = ex2(m - mn), f1 = ex2(x[u].x - mn);
        l = l * f0 + x[u].y * f1;
#pragma unroll
        for (int e = 0; e < CPL; ++e) a[e] = a[e] * f0 + v[u][e] * f1;
        m = mn;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < CPL; ++e) wacc[g][CPL * lane + e] = a[e];
  if (lane == 0) {
    wm[g] = m;
    wl[g] = l;
  }
  __syncthreads();
  if (g == 0) {
    float M = -INFINITY;
    for (int gg = 0; gg < kCombWarps; ++gg) M = fmaxf(M, wm[gg]);
    float L = 0.0f, A[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) A[e] = 0.0f;
    for (int gg = 0; gg < kCombWarps; ++gg) {
      if (wl[gg] > 0.0f) {
        const float f = ex2(wm[gg] - M);
        L += wl[gg] * f;
#pragma unroll
        for (int e = 0; e < CPL; ++e) A[e] += wacc[gg][CPL * lane + e] * f;
      }
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) o[(int64_t)bh * D + CPL * lane + e] = __float2bfloat16_rn(A[e] / L);
    if (lane == 0 && lse) lse[bh] = (M + log2f(L)) * kLn2;
  }
}

// Work split: head groups per KV head (nhg) and slices of the cache per (batch, KV
// head, head group): nsl1 slices of s1 keys before the window, nsl - nsl1 slices of
// s2 keys over it.  The window is fully allowed, the rest only where the masks meet,
// so the slices are sized for equal expected work: the density outside the window is
// estimated as the chance that two uniformly drawn top_k-sets of the K groups share
// one, 1 - C(K - k, k) / C(K, k) (load balance only; every key is still visited).
struct DecPlan {
  int nhg, nsl, nsl1, s1, s2;
};

DecPlan dec_plan(const focus_params& p) {
  DecPlan d;
  const int gq = p.H / p.H_kv;
  d.nhg = (gq + kDecHeads - 1) / kDecHeads;
  const int64_t base = (int64_t)p.B * p.H_kv * d.nhg;
  int64_t nsl = std::max<int64_t>(1, (kDecTargetWarps + base - 1) / base);
  nsl = std::min<int64_t>(nsl, (p.N + kDecMinSlice - 1) / kDecMinSlice);
  const int64_t nwin = std::min<int64_t>(p.w, p.N), nrest = p.N - nwin;
  double miss = 1.0;  // C(K - k, k) / C(K, k)
  for (int t = 0; t < p.top_k; ++t) miss *= std::max(0.0, (double)(p.K - p.top_k - t)) / (p.K - t);
  const double work = (1.0 - miss) * nrest + nwin;
  int64_t n2 = nrest == 0 ? nsl : std::llround(nwin * nsl / std::max(work, 1.0));
  n2 = std::min<int64_t>(std::max<int64_t>(n2, 1), nrest == 0 ? nsl : std::max<int64_t>(nsl - 1, 1));
  const int64_t n1 = nrest == 0 ? 0 : std::max<int64_t>(nsl - n2, 1);
  d.s1 = n1 ? (int)(((nrest + n1 - 1) / n1 + 31) / 32 * 32) : 32;
  d.s2 = (int)(((nwin + n2 - 1) / n2 + 31) / 32 * 32);
  d.nsl1 = n1 ? (int)((nrest + d.s1 - 1) / d.s1) : 0;
  d.nsl = d.nsl1 + (int)((nwin + d.s2 - 1) / d.s2);
  return d;
}

size_t dec_ml_bytes(const focus_params& p, const DecPlan& d) {
  return align_up(sizeof(float2) * (size_t)p.B * p.H * d.nsl, 256);
}

template <int D>
cudaError_t launch_split(const focus_params& p, const DecPlan& d, float sl2, const bf16* q,
                         const bf16* k, const bf16* v, const uint32_t* mask, float2* part_ml,
                         float* part_acc, cudaStream_t s) {
  using L = DecLayout<D>;
  static bool configured = false;  // host-side attribute, set once before the first launch
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_split<D>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t items = (int64_t)p.B * p.H_kv * d.nhg * d.nsl;
  decode_split<D><<<(unsigned)items, 32, L::BYTES, s>>>(p.N, p.H, p.H_kv, p.R, p.w, p.B, d.nsl,
                                                        d.nsl1, d.s1, d.s2, sl2, q, k, v, mask,
                                                        part_ml, part_acc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const focus_params& p, const bf16* q, const bf16* k, const bf16* v,
                          const uint32_t* mask, bf16* o, float* lse, char* ws, float scale,
                          cudaStream_t s) {
  const DecPlan d = dec_plan(p);
  float2* part_ml = reinterpret_cast<float2*>(ws);
  float* part_acc = reinterpret_cast<float*>(ws + dec_ml_bytes(p, d));
  const float sl2 = scale * kLog2e;
  cudaError_t e = p.d_head == 64
                      ? launch_split<64>(p, d, sl2, q, k, v, mask, part_ml, part_acc, s)
                      : launch_split<128>(p, d, sl2, q, k, v, mask, part_ml, part_acc, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.H));
  cfg.blockDim = dim3(32 * kCombWarps);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float2* ml = part_ml;
  const float* pa = part_acc;
  e = p.d_head == 64 ? cudaLaunchKernelEx(&cfg, decode_combine<64>, d.nsl, ml, pa, o, lse)
                     : cudaLaunchKernelEx(&cfg, decode_combine<128>, d.nsl, ml, pa, o, lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t decode_workspace_bytes(const focus_params& p) {
  const DecPlan d = dec_plan(p);
  return dec_ml_bytes(p, d) +
         align_up(sizeof(float) * (size_t)p.B * p.H * d.nsl * p.d_head, 256);
}

}  // namespace focus
