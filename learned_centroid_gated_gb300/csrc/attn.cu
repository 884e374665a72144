// Focus attention: long-range part over compatible segments and window part with
// the union merge (warp-level mma.sync tensor-core path).
//
// "Why Attend to Everything? Focus is the Key", gist.science technical summary,
// section 2 "Core Architecture": the local window of w tokens attends with exact
// softmax; distant tokens attend only within a shared group; jindou-blog deep read,
// method bullets: exact softmax inside groups as well.  One softmax runs over the
// union of the two sets.  The two sets are disjoint by construction (long-range
// keys satisfy i - j >= w, window keys i - j < w), so the union softmax is the
// log-sum-exp merge of the two partial softmaxes, each key counted once.
//
//   attn_long   query block (128 rows of one segment S, one head) x the key tiles
//               of every segment T with mask(S) & mask(T) != 0, positions
//               pos_j <= pos_i - w.  Writes O_lr (fp32, normalised) and LSE_lr
//               scattered back to natural token order.
//   attn_window query tile (128 consecutive tokens, one head) x keys (i-w, i];
//               merges (O_lr, LSE_lr) and writes O (bf16) and LSE.
#include <math.h>

#include "common.cuh"

namespace focus {
namespace {

constexpr int BM = kAttnBM;  // 128 query rows, 16 per warp
constexpr int BN = 64;       // keys per tile
constexpr int NW = 8;
constexpr int NT = NW * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct TileEnt {
  int start;   // first permuted row of the key segment
  int cnt;     // keys of the segment with pos <= p_hi - w
  int nfull;   // leading tiles whose keys all satisfy pos <= p_lo - w
};

template <int D>
struct Smem {
  alignas(128) bf16 q[BM * D];
  alignas(128) bf16 k[2][BN * D];
  alignas(128) bf16 v[2][BN * D];
  int kpos[2][BN];
  int qpos[BM];
  int tmask[2];
  int n_ent;
  TileEnt ent[1];  // n_ent entries follow (dynamic shared memory)
};

// 16-byte chunk c of row `row` in a tile whose rows hold D bf16: XOR swizzle on
// the low three chunk bits, so that ldmatrix rows hit distinct bank groups.
template <int D>
__device__ __forceinline__ int swz(int row, int c) {
  return row * (D / 8) + (c ^ (row & 7));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(unsigned addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(unsigned addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// First index in P[lo, hi) whose value exceeds x (P ascending).
__device__ __forceinline__ int upper_bound(const int* __restrict__ P, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

struct AttnArgs {
  const bf16* q;  // long: Qp [B, H, N, d]; window: q [B, N, H, d]
  const bf16* k;  // long: Kp [B, H_kv, N, d]; window: k [B, N, H_kv, d]
  const bf16* v;
  int B, N, H, H_kv, R, w, nseg;
  float sl2;  // softmax scale * log2(e)
  const int* perm;
  const int* seg_off;
  const uint32_t* mask;
  const QBlock* qtab;
  const int* qtab_count;
  float* o_lr;   // [B, N, H, d] fp32
  float* lse_lr; // [B, H, N] fp32
  bf16* o;       // [B, N, H, d]
  float* lse;    // [B, H, N] or null
};

// One CTA: 128 query rows of one head; 8 warps, each owns 16 rows.
template <int D, bool LONG>
__global__ void __launch_bounds__(NT, 1) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem<D>& s = *reinterpret_cast<Smem<D>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int b, h, kvh, rows;
  const bf16* qbase;      // first query row
  int64_t q_stride;       // elements between query rows
  const bf16 *kbase, *vbase;
  int64_t kv_stride;
  int total_tiles;
  // window geometry
  int i0 = 0, j_lo = 0, j_hi = 0;
  // long geometry
  const int* P = nullptr;
  int64_t kv_head_row0 = 0;

  if constexpr (LONG) {
    const int hpg = a.H / a.R;
    const int u = blockIdx.x / hpg;
    if (u >= *a.qtab_count) return;
    const QBlock e = a.qtab[u];
    const int rho = e.br % a.R;
    b = e.br / a.R;
    h = rho * hpg + (int)(blockIdx.x % hpg);
    kvh = h / (a.H / a.H_kv);
    rows = e.rows;
    P = a.perm + (int64_t)e.br * a.N;
    const int* SO = a.seg_off + (int64_t)e.br * (a.nseg + 1);
    qbase = a.q + (((int64_t)b * a.H + h) * a.N + e.row0) * D;
    q_stride = D;
    kv_head_row0 = ((int64_t)b * a.H_kv + kvh) * a.N;
    kbase = a.k;
    vbase = a.v;
    kv_stride = D;
    for (int r = tid; r < BM; r += NT) s.qpos[r] = __ldg(P + e.row0 + min(r, rows - 1));
    if (warp == 0) {
      const int p_lo = __ldg(P + e.row0), p_hi = __ldg(P + e.row0 + rows - 1);
      const uint32_t mS = __ldg(a.mask + (int64_t)e.br * a.N + p_lo);
      int n_ent = 0;
      for (int T0 = 0; T0 < a.nseg; T0 += 32) {
        const int T = T0 + lane;
        bool ok = false;
        TileEnt te{0, 0, 0};
        if (T < a.nseg) {
          const int st = __ldg(SO + T), en = __ldg(SO + T + 1);
          if (en > st) {
            const uint32_t mT = __ldg(a.mask + (int64_t)e.br * a.N + __ldg(P + st));
            if (mT & mS) {
              const int hi = upper_bound(P, st, en, p_hi - a.w) - st;
              if (hi > 0) {
                ok = true;
                te.start = st;
                te.cnt = hi;
                te.nfull = (upper_bound(P, st, en, p_lo - a.w) - st) / BN;
              }
            }
          }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) s.ent[n_ent + __popc(bal & ((1u << lane) - 1u))] = te;
        n_ent += __popc(bal);
      }
      if (lane == 0) s.n_ent = n_ent;
    }
    __syncthreads();
    total_tiles = 0;
    for (int i = 0; i < s.n_ent; ++i) total_tiles += (s.ent[i].cnt + BN - 1) / BN;
  } else {
    i0 = blockIdx.x * BM;
    h = blockIdx.y;
    b = blockIdx.z;
    kvh = h / (a.H / a.H_kv);
    rows = min(BM, a.N - i0);
    qbase = a.q + (((int64_t)b * a.N + i0) * a.H + h) * D;
    q_stride = (int64_t)a.H * D;
    j_lo = max(0, i0 - a.w + 1);
    j_hi = i0 + rows;
    kbase = a.k + (((int64_t)b * a.N) * a.H_kv + kvh) * D;
    vbase = a.v + (((int64_t)b * a.N) * a.H_kv + kvh) * D;
    kv_stride = (int64_t)a.H_kv * D;
    for (int r = tid; r < BM; r += NT) s.qpos[r] = i0 + min(r, rows - 1);
    total_tiles = (j_hi - j_lo + BN - 1) / BN;
    __syncthreads();
  }

  // ---- tile loader (all threads) ----
  int ld_e = 0, ld_t = 0;  // long: current entry and tile inside it
  auto load_tile = [&](int stage, int tile) {
    int64_t row0;  // first key row (in units of rows of kv_stride)
    int valid, need_mask;
    const int* posp = nullptr;
    int pos0 = 0;
    if constexpr (LONG) {
      const TileEnt te = s.ent[ld_e];
      row0 = kv_head_row0 + te.start + (int64_t)ld_t * BN;
      valid = min(BN, te.cnt - ld_t * BN);
      need_mask = ld_t >= te.nfull;
      posp = P + te.start + ld_t * BN;
      if (++ld_t * BN >= te.cnt) { ++ld_e; ld_t = 0; }
    } else {
      const int j0 = j_lo + tile * BN;
      row0 = j0;
      valid = min(BN, j_hi - j0);
      pos0 = j0;
      const int i_last = i0 + rows - 1;
      need_mask = !(valid == BN && j0 + BN - 1 <= i0 && i_last - j0 < a.w);
    }
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    for (int idx = tid; idx < BN * CPR; idx += NT) {
      const int r = idx / CPR, c = idx % CPR;
      const bool ok = r < valid;
      const int64_t off = (row0 + (ok ? r : 0)) * kv_stride + c * 8;
      cp_async16(&s.k[stage][swz<D>(r, c) * 8], kbase + off, ok);
      cp_async16(&s.v[stage][swz<D>(r, c) * 8], vbase + off, ok);
    }
    for (int r = tid; r < BN; r += NT) {
      int pos = kKeySentinel;
      if (r < valid) pos = LONG ? __ldg(posp + r) : pos0 + r;
      s.kpos[stage][r] = pos;
    }
    if (tid == 0) s.tmask[stage] = need_mask;
  };

  {
    constexpr int CPR = D / 8;
    for (int idx = tid; idx < BM * CPR; idx += NT) {
      const int r = idx / CPR, c = idx % CPR;
      const bool ok = r < rows;
      cp_async16(&s.q[swz<D>(r, c) * 8], qbase + (ok ? r : 0) * q_stride + c * 8, ok);
    }
  }
  if (total_tiles > 0) load_tile(0, 0);
  cp_commit();

  const int g = lane >> 2, t4 = lane & 3;
  const int ra = warp * 16 + g, rb = ra + 8;
  uint32_t qf[D / 16][4];
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
  int qp_a = 0, qp_b = 0;

  const unsigned q_s = (unsigned)__cvta_generic_to_shared(s.q);
  for (int it = 0; it < total_tiles || it == 0; ++it) {
    if (it + 1 < total_tiles) {
      load_tile((it + 1) & 1, it + 1);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (it == 0) {
      qp_a = s.qpos[ra];
      qp_b = s.qpos[rb];
#pragma unroll
      for (int kc = 0; kc < D / 16; ++kc) {
        const int row = warp * 16 + (lane & 15);
        const int c = kc * 2 + (lane >> 4);
        ldsm_x4(q_s + swz<D>(row, c) * 16, qf[kc][0], qf[kc][1], qf[kc][2], qf[kc][3]);
      }
      if (total_tiles == 0) break;
    }
    const int st = it & 1;
    const unsigned k_s = (unsigned)__cvta_generic_to_shared(s.k[st]);
    const unsigned v_s = (unsigned)__cvta_generic_to_shared(s.v[st]);

    // S = Q K^T  (16 x 64 per warp)
    float sacc[BN / 8][4];
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
#pragma unroll
    for (int kc = 0; kc < D / 16; ++kc) {
#pragma unroll
      for (int nb2 = 0; nb2 < BN / 16; ++nb2) {
        const int row = nb2 * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kc * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(k_s + swz<D>(row, c) * 16, b0, b1, b2, b3);
        mma16816(sacc[2 * nb2], qf[kc], b0, b1);
        mma16816(sacc[2 * nb2 + 1], qf[kc], b2, b3);
      }
    }

    // scale, mask, online softmax (log2 domain)
    const bool need_mask = s.tmask[st] != 0;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < BN / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = sacc[nb][e] * a.sl2;
        if (need_mask) {
          const int kp = s.kpos[st][nb * 8 + 2 * t4 + (e & 1)];
          const int qp = (e < 2) ? qp_a : qp_b;
          bool ok;
          if constexpr (LONG) ok = (qp - kp) >= a.w;
          else ok = (qp - kp) >= 0 && (qp - kp) < a.w;
          if (!ok) x = -INFINITY;
        }
        sacc[nb][e] = x;
      }
      mx_a = fmaxf(mx_a, fmaxf(sacc[nb][0], sacc[nb][1]));
      mx_b = fmaxf(mx_b, fmaxf(sacc[nb][2], sacc[nb][3]));
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float ms_a = (mn_a == -INFINITY) ? 0.0f : mn_a;
    const float ms_b = (mn_b == -INFINITY) ? 0.0f : mn_b;
    const float al_a = exp2f(m_a - ms_a), al_b = exp2f(m_b - ms_b);
    m_a = mn_a;
    m_b = mn_b;
    float rs_a = 0.0f, rs_b = 0.0f;
#pragma unroll
    for (int nb = 0; nb < BN / 8; ++nb) {
      sacc[nb][0] = exp2f(sacc[nb][0] - ms_a);
      sacc[nb][1] = exp2f(sacc[nb][1] - ms_a);
      sacc[nb][2] = exp2f(sacc[nb][2] - ms_b);
      sacc[nb][3] = exp2f(sacc[nb][3] - ms_b);
      rs_a += sacc[nb][0] + sacc[nb][1];
      rs_b += sacc[nb][2] + sacc[nb][3];
    }
    l_a = l_a * al_a + rs_a;
    l_b = l_b * al_b + rs_b;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      oacc[i][0] *= al_a;
      oacc[i][1] *= al_a;
      oacc[i][2] *= al_b;
      oacc[i][3] *= al_b;
    }
    // O += P V
#pragma unroll
    for (int kc = 0; kc < BN / 16; ++kc) {
      uint32_t pa[4];
      pa[0] = pack_bf16(sacc[2 * kc][0], sacc[2 * kc][1]);
      pa[1] = pack_bf16(sacc[2 * kc][2], sacc[2 * kc][3]);
      pa[2] = pack_bf16(sacc[2 * kc + 1][0], sacc[2 * kc + 1][1]);
      pa[3] = pack_bf16(sacc[2 * kc + 1][2], sacc[2 * kc + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < D / 16; ++nd2) {
        const int row = kc * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = nd2 * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(v_s + swz<D>(row, c) * 16, b0, b1, b2, b3);
        mma16816(oacc[2 * nd2], pa, b0, b1);
        mma16816(oacc[2 * nd2 + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }

  // ---- epilogue ----
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rb : ra;
    if (r >= rows) continue;
    const float l = half ? l_b : l_a;
    const float m = half ? m_b : m_a;
    const int pos = half ? qp_b : qp_a;
    const int e0 = half ? 2 : 0;
    const int64_t orow = (((int64_t)b * a.N + pos) * a.H + h) * D;
    const int64_t lrow = ((int64_t)b * a.H + h) * a.N + pos;
    if constexpr (LONG) {
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const float lse = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = nd * 8 + 2 * t4;
        *reinterpret_cast<float2*>(a.o_lr + orow + col) =
            make_float2(oacc[nd][e0] * inv, oacc[nd][e0 + 1] * inv);
      }
      if (t4 == 0) a.lse_lr[lrow] = lse;
    } else {
      const float lse_w = (m + log2f(l)) * kLn2;
      const float lse_l = a.lse_lr[lrow];
      float ww, wl, lse;
      if (lse_l == -INFINITY) {
        ww = 1.0f / l;
        wl = 0.0f;
        lse = lse_w;
      } else {
        const float M = fmaxf(lse_w, lse_l);
        const float ew = expf(lse_w - M), el = expf(lse_l - M);
        const float tot = ew + el;
        lse = M + logf(tot);
        ww = ew / tot / l;
        wl = el / tot;
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = nd * 8 + 2 * t4;
        float2 ol = make_float2(0.0f, 0.0f);
        if (wl != 0.0f) ol = *reinterpret_cast<const float2*>(a.o_lr + orow + col);
        const float x0 = oacc[nd][e0] * ww + ol.x * wl;
        const float x1 = oacc[nd][e0 + 1] * ww + ol.y * wl;
        *reinterpret_cast<__nv_bfloat162*>(a.o + orow + col) = __floats2bfloat162_rn(x0, x1);
      }
      if (t4 == 0 && a.lse) a.lse[lrow] = lse;
    }
  }
}

template <int D, bool LONG>
cudaError_t launch(const AttnArgs& args, dim3 grid, int nseg, cudaStream_t s) {
  const size_t shm = sizeof(Smem<D>) + sizeof(TileEnt) * (LONG ? nseg : 0);
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, LONG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
  if (e != cudaSuccess) return e;
  attn_kernel<D, LONG><<<grid, NT, shm, s>>>(args);
  return cudaGetLastError();
}

AttnArgs make_args(const focus_params& p, const WsLayout& L, char* ws, float scale) {
  AttnArgs a{};
  a.B = p.B;
  a.N = p.N;
  a.H = p.H;
  a.H_kv = p.H_kv;
  a.R = p.R;
  a.w = p.w;
  a.nseg = L.nseg;
  a.sl2 = scale * kLog2e;
  a.perm = reinterpret_cast<const int*>(ws + L.perm);
  a.seg_off = reinterpret_cast<const int*>(ws + L.segoff);
  a.qtab = reinterpret_cast<const QBlock*>(ws + L.qtab);
  a.qtab_count = &reinterpret_cast<const WsHeader*>(ws)->qtab_count;
  a.o_lr = reinterpret_cast<float*>(ws + L.olr);
  a.lse_lr = reinterpret_cast<float*>(ws + L.lselr);
  return a;
}

}  // namespace

cudaError_t launch_attn_long(const focus_params& p, const WsLayout& L, const uint32_t* mask,
                             char* ws, float scale, cudaStream_t s) {
  AttnArgs a = make_args(p, L, ws, scale);
  a.q = reinterpret_cast<const bf16*>(ws + L.qp);
  a.k = reinterpret_cast<const bf16*>(ws + L.kp);
  a.v = reinterpret_cast<const bf16*>(ws + L.vp);
  a.mask = mask;
  const int64_t blocks = (int64_t)L.qtab_cap * (p.H / p.R);
  dim3 grid((unsigned)blocks);
  return p.d_head == 64 ? launch<64, true>(a, grid, L.nseg, s) : launch<128, true>(a, grid, L.nseg, s);
}

cudaError_t launch_attn_window(const focus_params& p, const WsLayout& L, const bf16* q,
                               const bf16* k, const bf16* v, char* ws, bf16* o, float* lse,
                               float scale, cudaStream_t s) {
  AttnArgs a = make_args(p, L, ws, scale);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  dim3 grid((p.N + BM - 1) / BM, p.H, p.B);
  return p.d_head == 64 ? launch<64, false>(a, grid, 0, s) : launch<128, false>(a, grid, 0, s);
}

}  // namespace focus
