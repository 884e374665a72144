// Last step of the group-list schedule: union softmax of one (token, head) from
// its disjoint parts.
//
// "Why Attend to Everything? Focus is the Key", gist.science technical summary,
// section 2 "Core Architecture": one exact softmax over the window keys and the
// distant keys of shared groups.  With group lists a token's distant keys are
// split over its top_k lists (a key counted only in the list of the lowest group
// it shares with the query), so the window part (O_w, LSE_w) and the top_k list
// parts (O_s, LSE_s) cover disjoint key sets whose union is the allowed set, and
//   LSE = log(exp(LSE_w) + sum_s exp(LSE_s)),
//   O   = (exp(LSE_w - LSE) O_w + sum_s exp(LSE_s - LSE) O_s).
// A list part with no key has LSE_s = -inf and weight 0.  HBM-bound: reads
// (1 + top_k) fp32 rows and writes one bf16 row per (token, head).
#include <math.h>

#include "common.cuh"

namespace focus {
namespace {

// D/4 threads per (b, n, h) row, four consecutive columns each.
template <int D>
__global__ void __launch_bounds__(256)
merge_slots(int64_t rows, int N, int H, int top_k, const float* __restrict__ o_part,
            const float* __restrict__ lse_part, const float* __restrict__ o_slot,
            const float* __restrict__ lse_slot, bf16* __restrict__ o, float* __restrict__ lse) {
  constexpr int TPR = D / 4;
  const int64_t x = (int64_t)blockIdx.x * (blockDim.x / TPR) + threadIdx.x / TPR;
  if (x >= rows) return;
  const int c = (threadIdx.x % TPR) * 4;
  const int h = (int)(x % H);
  const int64_t bn = x / H;  // b * N + n
  const int n = (int)(bn % N);
  const int64_t b = bn / N;
  const int64_t li = (b * H + h) * N + n;  // [B, H, N]
  const int64_t BHN = rows;                // B * N * H == B * H * N
  const int64_t oi = x * D + c;            // [B, N, H, D]
  const int64_t BNHD = rows * D;
  const float lw = __ldg(lse_part + li);   // finite: the window holds the diagonal key
  float M = lw;
  for (int s = 0; s < top_k; ++s) M = fmaxf(M, __ldg(lse_slot + s * BHN + li));
  float ew = expf(lw - M);
  float tot = ew;
  const float4 w4 = __ldg(reinterpret_cast<const float4*>(o_part + oi));
  float a0 = ew * w4.x, a1 = ew * w4.y, a2 = ew * w4.z, a3 = ew * w4.w;
  for (int s = 0; s < top_k; ++s) {
    const float ls = __ldg(lse_slot + s * BHN + li);
    if (ls == -INFINITY) continue;
    const float es = expf(ls - M);
    const float4 v = __ldg(reinterpret_cast<const float4*>(o_slot + s * BNHD + oi));
    tot += es;
    a0 += es * v.x;
    a1 += es * v.y;
    a2 += es * v.z;
    a3 += es * v.w;
  }
  const float inv = 1.0f / tot;
  __nv_bfloat162 p01 = __floats2bfloat162_rn(a0 * inv, a1 * inv);
  __nv_bfloat162 p23 = __floats2bfloat162_rn(a2 * inv, a3 * inv);
  uint2 out;
  out.x = *reinterpret_cast<uint32_t*>(&p01);
  out.y = *reinterpret_cast<uint32_t*>(&p23);
  *reinterpret_cast<uint2*>(o + oi) = out;
  if (lse && c == 0) lse[li] = M + logf(tot);
}

}  // namespace

cudaError_t launch_merge_slots(const focus_params& p, const WsLayout& L, const char* ws, bf16* o,
                               float* lse, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.N * p.H;
  const float* o_part = reinterpret_cast<const float*>(ws + L.olr);
  const float* lse_part = reinterpret_cast<const float*>(ws + L.lselr);
  const float* o_slot = reinterpret_cast<const float*>(ws + L.oslot);
  const float* lse_slot = reinterpret_cast<const float*>(ws + L.lseslot);
  const int per_block = 256 / (p.d_head / 4);
  const unsigned grid = (unsigned)((rows + per_block - 1) / per_block);
  if (p.d_head == 64)
    merge_slots<64><<<grid, 256, 0, s>>>(rows, p.N, p.H, p.top_k, o_part, lse_part, o_slot,
                                         lse_slot, o, lse);
  else
    merge_slots<128><<<grid, 256, 0, s>>>(rows, p.N, p.H, p.top_k, o_part, lse_part, o_slot,
                                          lse_slot, o, lse);
  return cudaGetLastError();
}

}  // namespace focus
