// Decode: attention of the newest token of each sequence (position N - 1) over its
// cache, on the same union set as the forward pass ("Why Attend to Everything?
// Focus is the Key", gist.science technical summary, section 2, "Core Architecture"
// and "Inference Efficiency (Top-k)": window keys with exact softmax plus distant
// keys that share a group).
//
// One query row per head is memory-bound work (each allowed key's K and V rows are
// read once per KV head), so this runs on the CUDA cores, split over the keys:
//   decode_chunk    one CTA per (chunk of CHUNK keys, KV head, batch row) and up
//                   to NH query heads of that KV head (NH, a template parameter, is the
//                   GQA ratio rounded down to 1, 2, 4 or 8, so the per-thread arrays fit
//                   the heads there are): compacts the allowed keys of the chunk
//                   (window, or mask overlap), scores them (one thread per key, its K
//                   row as independent 16-byte loads), and accumulates P V (16-byte V
//                   loads, kDecUnroll batches of keys in flight); writes (max, sum, acc).
//   decode_combine  merges the chunks of one (batch, head) by their maxima: O, LSE.
// CHUNK is 1024 keys, or 2048 when that still leaves at least 2048 CTAs (long
// caches: fewer, longer CTAs amortise the chunk's dependent memory round trips).
#include <math.h>

#include "common.cuh"

namespace focus {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecHeads = 8;     // most query heads per CTA (of one KV head)
constexpr int kDecUnroll = 8;    // P V: batches of keys whose V loads are in flight together
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ unsigned lanemask_lt_dec() {
  unsigned r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

template <int D, int NH, int CHUNK>
__global__ void __launch_bounds__(kDecThreads)
decode_chunk(int N, int H, int H_kv, int R, int w, float sl2, const bf16* __restrict__ q,
             const bf16* __restrict__ k, const bf16* __restrict__ v,
             const uint32_t* __restrict__ mask, float2* __restrict__ part_ml,
             float* __restrict__ part_acc, int nch) {
  __shared__ float qs[NH][D];
  __shared__ int idx[CHUNK];
  __shared__ float sc[NH][CHUNK];
  __shared__ int wsum[kDecThreads / 32];
  __shared__ float red[NH][kDecThreads / 32];
  __shared__ float stat[NH];
  __shared__ float accx[kDecThreads / (D / 8)][D];

  const int c = blockIdx.x, b = blockIdx.z;
  const int gq = H / H_kv;
  const int nhg = (gq + NH - 1) / NH;
  const int kvh = blockIdx.y / nhg, hg = blockIdx.y % nhg;
  const int h0 = kvh * gq + hg * NH;
  const int nh = min(NH, gq - hg * NH);
  const int rho = kvh / (H_kv / R);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = N - 1;
  const uint32_t* M = mask + ((int64_t)b * R + rho) * N;
  const uint32_t mq = __ldg(M + i);

  for (int t = tid; t < nh * D; t += kDecThreads) {
    const int hh = t / D, e = t % D;
    qs[hh][e] = __bfloat162float(q[((int64_t)b * H + h0 + hh) * D + e]);
  }
  // compaction of the chunk's allowed keys (every key of the cache is j <= i)
  const int j0 = c * CHUNK, j1 = min(N, j0 + CHUNK);
  int na = 0;
  for (int jb = j0; jb < j1; jb += kDecThreads) {
    const int j = jb + tid;
    bool ok = false;
    if (j < j1) ok = (i - j < w) || ((__ldg(M + j) & mq) != 0u);
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    int off = na, tot = 0;
    for (int w2 = 0; w2 < kDecThreads / 32; ++w2) {
      if (w2 < warp) off += wsum[w2];
      tot += wsum[w2];
    }
    if (ok) idx[off + __popc(bal & lanemask_lt_dec())] = j;
    __syncthreads();
    na += tot;
  }
  // scores: one thread per key; a key's row is read as D/8 independent 16-byte loads
  for (int a = tid; a < na; a += kDecThreads) {
    const uint4* kr = reinterpret_cast<const uint4*>(k + (((int64_t)b * N + idx[a]) * H_kv + kvh) * D);
    uint4 raw[D / 8];
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) raw[c8] = __ldg(kr + c8);
    float s[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) s[hh] = 0.0f;
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[c8]);
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const float2 f = __bfloat1622float2(p2[e2]);
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          if (hh < nh) {
            s[hh] = fmaf(f.x, qs[hh][c8 * 8 + 2 * e2], s[hh]);
            s[hh] = fmaf(f.y, qs[hh][c8 * 8 + 2 * e2 + 1], s[hh]);
          }
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
      if (hh < nh) sc[hh][a] = s[hh] * sl2;
  }
  __syncthreads();
  // chunk max and exponentials (log2 domain), chunk sums
  for (int hh = 0; hh < nh; ++hh) {
    float m = -INFINITY;
    for (int a = tid; a < na; a += kDecThreads) m = fmaxf(m, sc[hh][a]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[hh][warp] = m;
  }
  __syncthreads();
  if (tid < nh) {
    float m = -INFINITY;
    for (int w2 = 0; w2 < kDecThreads / 32; ++w2) m = fmaxf(m, red[tid][w2]);
    stat[tid] = m;
  }
  __syncthreads();
  for (int hh = 0; hh < nh; ++hh) {
    const float m = stat[hh];
    float l = 0.0f;
    for (int a = tid; a < na; a += kDecThreads) {
      const float p = exp2f(sc[hh][a] - m);
      sc[hh][a] = p;
      l += p;
    }
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) red[hh][warp] = l;
  }
  __syncthreads();
  // P V: D/8 threads cover a V row with 16-byte loads, kDecThreads/(D/8) keys at once
  constexpr int TPR = D / 8;                // threads per row
  constexpr int KPAR = kDecThreads / TPR;   // keys in flight per iteration
  const int seg = tid % TPR, kg = tid / TPR;
  float acc[NH][8];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh)
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[hh][u] = 0.0f;
  const uint4* vbase = reinterpret_cast<const uint4*>(v + ((int64_t)b * N * H_kv + kvh) * D) + seg;
  const int64_t vstride = (int64_t)H_kv * D / 8;  // uint4 per token
  for (int a0 = kg; a0 < na; a0 += KPAR * kDecUnroll) {
    uint4 raw[kDecUnroll];  // the batch's V loads are issued before any is used
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int a = a0 + u * KPAR;
      raw[u] = a < na ? __ldg(vbase + idx[a] * vstride) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int a = a0 + u * KPAR;
      if (a >= na) break;
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
      float vv[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(p2[e]);
        vv[2 * e] = f.x;
        vv[2 * e + 1] = f.y;
      }
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        if (hh < nh) {
          const float pa = sc[hh][a];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(pa, vv[e], acc[hh][e]);
        }
      }
    }
  }
  // reduce the KPAR key groups: group kg writes its partial row, then the sums
  for (int hh = 0; hh < nh; ++hh) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) accx[kg][seg * 8 + u] = acc[hh][u];
    __syncthreads();
    for (int ee = tid; ee < D; ee += kDecThreads) {
      float t = 0.0f;
      for (int g = 0; g < KPAR; ++g) t += accx[g][ee];
      const int64_t slot = ((int64_t)b * H + h0 + hh) * nch + c;
      part_acc[slot * D + ee] = t;
      if (ee == 0) {
        float l = 0.0f;
        for (int w2 = 0; w2 < kDecThreads / 32; ++w2) l += red[hh][w2];
        part_ml[slot] = make_float2(stat[hh], l);
      }
    }
  }
}

// Merge the chunks of one (batch, head): grid = B * H, kCombThreads threads: thread
// (g, e) sums element e over the chunks c = g (mod kCombThreads / D).
constexpr int kCombThreads = 1024;
template <int D>
__global__ void __launch_bounds__(kCombThreads)
decode_combine(int H, int nch, const float2* __restrict__ part_ml, const float* __restrict__ part_acc,
               bf16* __restrict__ o, float* __restrict__ lse) {
  constexpr int G = kCombThreads / D;
  __shared__ float red[kCombThreads / 32];
  __shared__ float partial[G][D];
  __shared__ float lpart[G];
  __shared__ float Ms;
  const int bh = blockIdx.x, tid = threadIdx.x, e = tid % D, g = tid / D;
  const float2* ml = part_ml + (int64_t)bh * nch;
  float M = -INFINITY;
  for (int c = tid; c < nch; c += kCombThreads) M = fmaxf(M, ml[c].x);
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((tid & 31) == 0) red[tid >> 5] = M;
  __syncthreads();
  if (tid == 0) {
    float m = -INFINITY;
    for (int w2 = 0; w2 < kCombThreads / 32; ++w2) m = fmaxf(m, red[w2]);
    Ms = m;
  }
  __syncthreads();
  M = Ms;
  float L = 0.0f, acc = 0.0f;
#pragma unroll 4
  for (int c = g; c < nch; c += G) {
    const float2 x = ml[c];
    const float f = x.y > 0.0f ? exp2f(x.x - M) : 0.0f;
    L += x.y * f;
    acc += part_acc[((int64_t)bh * nch + c) * D + e] * f;
  }
  partial[g][e] = acc;
  if (e == 0) lpart[g] = L;
  __syncthreads();
  if (g == 0) {
    float tot = 0.0f, Lt = 0.0f;
    for (int gg = 0; gg < G; ++gg) {
      tot += partial[gg][e];
      Lt += lpart[gg];
    }
    o[(int64_t)bh * D + e] = __float2bfloat16_rn(tot / Lt);
    if (e == 0 && lse) lse[bh] = (M + log2f(Lt)) * kLn2;
  }
}

}  // namespace

int heads_per_cta(const focus_params& p) {
  const int gq = p.H / p.H_kv;
  return gq >= 8 ? 8 : gq >= 4 ? 4 : gq >= 2 ? 2 : 1;
}

int chunk_keys(const focus_params& p) {
  const int gq = p.H / p.H_kv, nh = heads_per_cta(p);
  const int64_t ctas = (int64_t)((p.N + 1023) / 1024) * p.H_kv * ((gq + nh - 1) / nh) * p.B;
  return (nh <= 4 && ctas >= 2048) ? 2048 : 1024;
}

int decode_chunks(const focus_params& p) { return (p.N + chunk_keys(p) - 1) / chunk_keys(p); }

cudaError_t launch_decode(const focus_params& p, const bf16* q, const bf16* k, const bf16* v,
                          const uint32_t* mask, bf16* o, float* lse, char* ws, float scale,
                          cudaStream_t s) {
  const int nch = decode_chunks(p);
  const int gq = p.H / p.H_kv;
  const int nh = heads_per_cta(p);  // query heads per CTA
  const int nhg = (gq + nh - 1) / nh;
  const bool wide = chunk_keys(p) == 2048;
  float2* part_ml = reinterpret_cast<float2*>(ws);
  float* part_acc = reinterpret_cast<float*>(ws + align_up(sizeof(float2) * (size_t)p.B * p.H * nch, 256));
  dim3 grid(nch, p.H_kv * nhg, p.B);
  const float sl2 = scale * kLog2e;
  auto chunk = [&](auto kernel) {
    kernel<<<grid, kDecThreads, 0, s>>>(p.N, p.H, p.H_kv, p.R, p.w, sl2, q, k, v, mask, part_ml,
                                        part_acc, nch);
  };
  if (p.d_head == 64) {
    if (nh == 8) chunk(decode_chunk<64, 8, 1024>);
    else if (nh == 4) wide ? chunk(decode_chunk<64, 4, 2048>) : chunk(decode_chunk<64, 4, 1024>);
    else if (nh == 2) wide ? chunk(decode_chunk<64, 2, 2048>) : chunk(decode_chunk<64, 2, 1024>);
    else wide ? chunk(decode_chunk<64, 1, 2048>) : chunk(decode_chunk<64, 1, 1024>);
    decode_combine<64><<<p.B * p.H, kCombThreads, 0, s>>>(p.H, nch, part_ml, part_acc, o, lse);
  } else {
    if (nh == 8) chunk(decode_chunk<128, 8, 1024>);
    else if (nh == 4) wide ? chunk(decode_chunk<128, 4, 2048>) : chunk(decode_chunk<128, 4, 1024>);
    else if (nh == 2) wide ? chunk(decode_chunk<128, 2, 2048>) : chunk(decode_chunk<128, 2, 1024>);
    else wide ? chunk(decode_chunk<128, 1, 2048>) : chunk(decode_chunk<128, 1, 1024>);
    decode_combine<128><<<p.B * p.H, kCombThreads, 0, s>>>(p.H, nch, part_ml, part_acc, o, lse);
  }
  return cudaGetLastError();
}

size_t decode_workspace_bytes(const focus_params& p) {
  const size_t nch = (size_t)decode_chunks(p);
  return align_up(sizeof(float2) * (size_t)p.B * p.H * nch, 256) +
         align_up(sizeof(float) * (size_t)p.B * p.H * nch * p.d_head, 256);
}

}  // namespace focus
