// Routing kernels: centroid scores, optional Sinkhorn balancing, hard top-k.
//
// "Why Attend to Everything? Focus is the Key":
//   gist.science technical summary, section 2 "Core Architecture" (K learnable
//   centroids C in R^{K x d_g}, tokens projected into centroid space) and
//   "Inference Efficiency (Top-k)" (each token joins its top-k groups);
//   "Key Technical Innovation: Sinkhorn Normalization" (balanced assignment);
//   jindou-blog deep read, method bullets (d_g = 16, dot-product scores).
//
// Memory-bound: each token reads its 64-byte routing vector once per pass and
// writes a 4-byte bitmask; centroids sit in shared memory.
#include <math.h>

#include "common.cuh"

namespace focus {
namespace {

constexpr int kRouteThreads = 256;

__device__ __forceinline__ void load_r(const float* __restrict__ r, int64_t idx, float (&rv)[16]) {
  const float4* rp = reinterpret_cast<const float4*>(r + idx * 16);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float4 x = __ldg(rp + c);
    rv[4 * c + 0] = x.x;
    rv[4 * c + 1] = x.y;
    rv[4 * c + 2] = x.z;
    rv[4 * c + 3] = x.w;
  }
}

// s_g = r . c_g as a fused multiply-add chain over t = 0..15 (fixed order), then
// divided by eps when Sinkhorn is on.
__device__ __forceinline__ void scores(const float (&rv)[16], const float* Cs, int K, bool scaled,
                                       float eps, float (&s)[FOCUS_MAX_K]) {
#pragma unroll
  for (int g = 0; g < FOCUS_MAX_K; ++g) {
    float a = 0.0f;
    if (g < K) {
#pragma unroll
      for (int t = 0; t < 16; ++t) a = fmaf(rv[t], Cs[g * 16 + t], a);
      if (scaled) a = a / eps;
    }
    s[g] = a;
  }
}

// Row potential alpha_i = -LSE_g(L_ig + beta_g) of the previous Sinkhorn iteration.
__device__ __forceinline__ float row_potential(const float (&L)[FOCUS_MAX_K], const float* beta,
                                               int K) {
  float m = -INFINITY;
#pragma unroll
  for (int g = 0; g < FOCUS_MAX_K; ++g)
    if (g < K) m = fmaxf(m, L[g] + beta[g]);
  float acc = 0.0f;
#pragma unroll
  for (int g = 0; g < FOCUS_MAX_K; ++g)
    if (g < K) acc += expf(L[g] + beta[g] - m);
  return -(m + logf(acc));
}

// Column step, part 1: per block of tokens and group g, the pair (max, sum exp(x - max))
// of x_i = L_ig + alpha_i.  grid = (blocks, B*R); one thread per token.
__global__ void __launch_bounds__(kRouteThreads)
sinkhorn_col_partial(int N, int R, int K, float eps, const float* __restrict__ r,
                     const float* __restrict__ C, const float* __restrict__ beta_prev,
                     int first_iter, float2* __restrict__ part) {
  __shared__ float Cs[FOCUS_MAX_K * 16];
  __shared__ float bs[FOCUS_MAX_K];
  __shared__ float red[kRouteThreads / 32][FOCUS_MAX_K];
  __shared__ float colmax[FOCUS_MAX_K];
  const int br = blockIdx.y;
  const int b = br / R, rho = br % R;
  for (int t = threadIdx.x; t < K * 16; t += blockDim.x) Cs[t] = C[t];
  for (int t = threadIdx.x; t < K; t += blockDim.x) bs[t] = first_iter ? 0.0f : beta_prev[br * K + t];
  __syncthreads();

  const int n = blockIdx.x * kRouteThreads + threadIdx.x;
  const bool valid = n < N;
  float x[FOCUS_MAX_K];
  if (valid) {
    float rv[16];
    load_r(r, ((int64_t)b * N + n) * R + rho, rv);
    scores(rv, Cs, K, true, eps, x);
    const float alpha = first_iter ? 0.0f : row_potential(x, bs, K);
#pragma unroll
    for (int g = 0; g < FOCUS_MAX_K; ++g) x[g] += alpha;
  } else {
#pragma unroll
    for (int g = 0; g < FOCUS_MAX_K; ++g) x[g] = -INFINITY;
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // block max per group
#pragma unroll
  for (int g = 0; g < FOCUS_MAX_K; ++g) {
    if (g >= K) break;
    float v = x[g];
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[wid][g] = v;
  }
  __syncthreads();
  if (threadIdx.x < K) {
    float v = -INFINITY;
    for (int w = 0; w < kRouteThreads / 32; ++w) v = fmaxf(v, red[w][threadIdx.x]);
    colmax[threadIdx.x] = v;
  }
  __syncthreads();
  // block sum of exp(x - max) per group
#pragma unroll
  for (int g = 0; g < FOCUS_MAX_K; ++g) {
    if (g >= K) break;
    const float m = colmax[g];
    float v = (valid && m > -INFINITY) ? expf(x[g] - m) : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[wid][g] = v;
  }
  __syncthreads();
  if (threadIdx.x < K) {
    float v = 0.0f;
    for (int w = 0; w < kRouteThreads / 32; ++w) v += red[w][threadIdx.x];
    part[((int64_t)br * gridDim.x + blockIdx.x) * K + threadIdx.x] = make_float2(colmax[threadIdx.x], v);
  }
}

// Column step, part 2: merge the partials in a fixed order (deterministic) and set
// beta_g = log(N/K) - LSE_i(x_ig).  grid = B*R, one thread per group.
__global__ void sinkhorn_col_final(int N, int K, int nblk, const float2* __restrict__ part,
                                   float* __restrict__ beta) {
  const int br = blockIdx.x, g = threadIdx.x;
  if (g >= K) return;
  float m = -INFINITY, s = 0.0f;
  for (int j = 0; j < nblk; ++j) {
    const float2 pj = part[((int64_t)br * nblk + j) * K + g];
    if (pj.y <= 0.0f) continue;
    const float mm = fmaxf(m, pj.x);
    s = s * expf(m - mm) + pj.y * expf(pj.x - mm);
    m = mm;
  }
  const float lse = m + logf(s);
  beta[br * K + g] = (float)log((double)N / (double)K) - lse;
}

// Top-k membership.  One thread per (b, n, rho) in r's memory order.  A ranking
// key that is not finite (NaN or +-inf, from non-finite r or C or an overflow)
// raises FOCUS_ERR_NONFINITE when `status` is given; a NaN key ranks as -inf, so
// the token's membership is still well defined (ties go to the lower group).
__global__ void __launch_bounds__(kRouteThreads)
route_topk(int B, int N, int R, int K, int top_k, int use_beta, float eps,
           const float* __restrict__ r, const float* __restrict__ C, const float* __restrict__ beta,
           uint32_t* __restrict__ mask, float* __restrict__ margin, int* status) {
  __shared__ float Cs[FOCUS_MAX_K * 16];
  for (int t = threadIdx.x; t < K * 16; t += blockDim.x) Cs[t] = C[t];
  __syncthreads();
  const int64_t total = (int64_t)B * N * R;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int rho = (int)(idx % R);
    const int64_t bn = idx / R;
    const int n = (int)(bn % N);
    const int b = (int)(bn / N);
    const int br = b * R + rho;
    float rv[16];
    load_r(r, idx, rv);
    float key[FOCUS_MAX_K];
    scores(rv, Cs, K, use_beta != 0, eps, key);
    if (use_beta) {
#pragma unroll
      for (int g = 0; g < FOCUS_MAX_K; ++g)
        if (g < K) key[g] += __ldg(beta + br * K + g);
    }
    bool finite = true;
#pragma unroll
    for (int g = 0; g < FOCUS_MAX_K; ++g) {
      if (g < K && !isfinite(key[g])) {
        finite = false;
        if (isnan(key[g])) key[g] = -INFINITY;
      }
    }
    if (!finite && status) raise_status(status, FOCUS_ERR_NONFINITE);
    uint32_t bits = 0;
    float kth = 0.0f;
    for (int sel = 0; sel < top_k; ++sel) {
      int best = -1;
      float bv = 0.0f;
#pragma unroll
      for (int g = 0; g < FOCUS_MAX_K; ++g) {
        if (g < K && !((bits >> g) & 1u) && (best < 0 || key[g] > bv)) {
          best = g;
          bv = key[g];
        }
      }
      bits |= 1u << best;
      kth = bv;
    }
    const int64_t o = (int64_t)br * N + n;
    mask[o] = bits;
    if (margin) {
      float nxt = -INFINITY;
      bool any = false;
#pragma unroll
      for (int g = 0; g < FOCUS_MAX_K; ++g)
        if (g < K && !((bits >> g) & 1u)) {
          nxt = any ? fmaxf(nxt, key[g]) : key[g];
          any = true;
        }
      margin[o] = any ? kth - nxt : INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_route(const focus_params& p, const WsLayout& L, const float* r, const float* C,
                         char* ws, uint32_t* mask_out, float* margin_out, int* status,
                         cudaStream_t s) {
  const int BR = p.B * p.R;
  float* beta = reinterpret_cast<float*>(ws + L.beta);
  float2* part = reinterpret_cast<float2*>(ws + L.skpart);
  for (int it = 0; it < p.sinkhorn_iters; ++it) {
    dim3 grid(L.nblk_sk, BR);
    sinkhorn_col_partial<<<grid, kRouteThreads, 0, s>>>(p.N, p.R, p.K, p.sinkhorn_eps, r, C, beta,
                                                        it == 0, part);
    sinkhorn_col_final<<<BR, 32, 0, s>>>(p.N, p.K, L.nblk_sk, part, beta);
  }
  const int64_t total = (int64_t)p.B * p.N * p.R;
  int64_t blocks = (total + kRouteThreads - 1) / kRouteThreads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  route_topk<<<(unsigned)blocks, kRouteThreads, 0, s>>>(p.B, p.N, p.R, p.K, p.top_k,
                                                        p.sinkhorn_iters > 0, p.sinkhorn_eps, r, C,
                                                        beta, mask_out, margin_out, status);
  return cudaGetLastError();
}

}  // namespace focus

// ------------------------------------------------------ allocation-free entry --
// focus_route_static: focus_route without a caller workspace.  Its only scratch
// (the Sinkhorn column partials and potentials) lives in the file-scope device
// array below, which every GPU that loads this library holds until the process
// exits.  Without Sinkhorn iterations the routing needs no scratch at all.
#include <mutex>

namespace focus {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

using CtxGetCurrent = int (*)(void**);  // cuCtxGetCurrent(CUcontext*)

CtxGetCurrent ctx_get_current() {
  static CtxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrent>(p);
  });
  return fn;
}

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

// Device address of g_route_scratch on the current device.  Host code cannot use
// the symbol itself as a device pointer, so the address is looked up with
// cudaGetSymbolAddress once per device and kept with the CUDA context it belongs
// to; a call under another context of that device (after cudaDeviceReset, say)
// looks it up again.
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrent get = ctx_get_current();
  if (!get) return cudaErrorNotSupported;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  void* ctx = nullptr;
  if (get(&ctx) != 0) return cudaErrorDeviceUninitialized;
  if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
    // cudaGetSymbolAddress also makes the device's primary context current on a
    // thread that has none yet; the context is read after it
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// Scratch bytes of a Sinkhorn routing problem: beta [B*R, K] fp32, 256-byte
// aligned, then the column partials [B*R, ceil(N/256), K] (max, sum) pairs.
size_t static_scratch_need(const focus_params& p, size_t* skpart_off, int* nblk) {
  const size_t BR = (size_t)p.B * p.R;
  *nblk = (p.N + kSinkBlock - 1) / kSinkBlock;
  *skpart_off = align_up(sizeof(float) * BR * p.K, 256);
  return *skpart_off + sizeof(float2) * BR * (size_t)*nblk * p.K;
}

}  // namespace
}  // namespace focus

extern "C" size_t focus_route_static_limit(void) { return focus::kStaticScratchBytes; }

extern "C" int focus_route_static(const focus_params* p, const float* r, const float* C,
                                  uint32_t* mask_out, float* margin_out, void* stream) {
  using namespace focus;
  int rc = check_params(p);  // the same shape checks and codes as focus_route
  if (rc) return rc;
  // The size limit comes before anything else about the call, so that an
  // oversized problem is rejected whatever its pointers are.
  WsLayout L{};
  L.beta = 0;
  if (p->sinkhorn_iters > 0 &&
      static_scratch_need(*p, &L.skpart, &L.nblk_sk) > kStaticScratchBytes)
    return FOCUS_ERR_WORKSPACE;
  if (!r || !C || !mask_out) return FOCUS_ERR_INVALID_ARG;
  if ((uintptr_t)r % 16 || (uintptr_t)C % 4 || (uintptr_t)mask_out % 4 ||
      (uintptr_t)margin_out % 4)
    return FOCUS_ERR_ALIGNMENT;
  // Every partial is written before it is read and beta is not read before the
  // first column step writes it, so nothing in the array needs clearing between
  // calls.  Without Sinkhorn no kernel touches the array.
  void* scratch = nullptr;
  if (p->sinkhorn_iters > 0 && static_scratch(&scratch) != cudaSuccess) return FOCUS_ERR_CUDA;
  const cudaError_t e = launch_route(*p, L, r, C, static_cast<char*>(scratch), mask_out,
                                     margin_out, nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? FOCUS_OK : FOCUS_ERR_CUDA;
}
