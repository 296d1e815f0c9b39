// Router: logits on CUDA cores for small token counts (partial sums over
// slices of the hidden dimension), and the warp-per-token top-k_t selection
// with softmax / sigmoid gates.
//
// MoE-Prism (arXiv 2510.19366) §III-B2, expanded linear gate: a linear layer
// scores every sub-expert and the layer-wide top-k is taken over all of them;
// §III-C1: the budget k_i belongs to the request, so each token has its own k.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kTokPerCta = 8;

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(bf16lo(av[i]), bf16lo(bv[i]), acc);
    acc = fmaf(bf16hi(av[i]), bf16hi(bv[i]), acc);
  }
  return acc;
}

// Partial router logits over one slice of the hidden dimension:
//   P[s, t, u] = sum over h in slice s of x[t, h] * router_w[u, h]
// CTA = up to 8 tokens x 8 units x one slice of VS 16-byte vectors (at most
// kMaxSliceVec = 1024 columns).  Every thread issues all of its loads (the tokens' slice
// rows, staged in shared memory, and its warp's unit row slice) before it
// uses any, so the CTA costs one memory round trip; the grid spans tokens x
// units x slices, so a decode-sized batch still fills the GPU.  The top-k
// kernel adds the slices in order and the expert bias.
constexpr int kMaxSliceVec = 128;  // 1024 hidden columns
constexpr int kMaxLoads = kMaxSliceVec * kTokPerCta / 256;

__global__ void __launch_bounds__(256) router_logits_split_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ rw, int T, int nv, int E_r, int VS,
    float* __restrict__ P) {
  extern __shared__ uint4 xs[];  // [kTokPerCta][VS]
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.y * 8 + warp;
  const int t0 = blockIdx.x * kTokPerCta;
  const int nt = min(kTokPerCta, T - t0);
  const int v0 = blockIdx.z * VS;
  const int vn = min(VS, nv - v0);
  const int total = nt * vn;
  uint4 xr[kMaxLoads];
  uint4 wr[kMaxSliceVec / 32];
#pragma unroll
  for (int q = 0; q < kMaxLoads; ++q) {
    const int i = threadIdx.x + q * 256;
    if (i < total) {
      const int tt = i / vn, v = i - tt * vn;
      xr[q] = __ldg(x + static_cast<size_t>(t0 + tt) * nv + v0 + v);
    }
  }
  const uint4* wrow = rw + static_cast<size_t>(u < E_r ? u : 0) * nv + v0;
#pragma unroll
  for (int q = 0; q < kMaxSliceVec / 32; ++q) {
    const int v = lane + 32 * q;
    if (u < E_r && v < vn) wr[q] = __ldg(wrow + v);
  }
#pragma unroll
  for (int q = 0; q < kMaxLoads; ++q) {
    const int i = threadIdx.x + q * 256;
    if (i < total) {
      const int tt = i / vn, v = i - tt * vn;
      xs[tt * VS + v] = xr[q];
    }
  }
  __syncthreads();
  if (u >= E_r) return;
  float acc[kTokPerCta];
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) acc[i] = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxSliceVec / 32; ++q) {
    const int v = lane + 32 * q;
    if (v < vn) {
#pragma unroll
      for (int i = 0; i < kTokPerCta; ++i)
        if (i < nt) acc[i] = dot8_bf16(xs[i * VS + v], wr[q], acc[i]);
    }
  }
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) {
    float a = acc[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (lane == i) mine = a;
  }
  if (lane < nt)
    P[(static_cast<size_t>(blockIdx.z) * T + t0 + lane) * E_r + u] = mine;
}

// Total order used for selection: larger logit first; -0 == +0; NaN below
// every number.  The key is monotone in the logit.
__device__ __forceinline__ uint32_t order_key(float L) {
  if (L != L) return 0u;
  uint32_t b = __float_as_uint(L);
  if ((b & 0x7fffffffu) == 0u) b = 0u;  // -0 is +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp selects the k_t best units of one token.  Lane l holds units l,
// l+32, ... (IPL per lane); the token's logit of unit u is the sum of the S
// partial rows P[s] (s in order; S = 1 for finished logits) plus
// bias[u / n_sub] when bias is given, and is stored to lout[u] when lout is
// given.  Selection: a bitonic sort of all units on (key << 32 | ~u) in the
// warp's registers (key descending, lower index first on equal keys), so
// lane j < k ends up holding the j-th unit (*out_u) and its gate weight after
// renormalisation and route_scale (*out_w).
// Returns k.
template <int IPL>
__device__ __forceinline__ int warp_topk(const float* __restrict__ P, int S, size_t sstride,
                                         const float* __restrict__ bias, int n_sub,
                                         float* __restrict__ lout, int kt, int E_r, int k_max,
                                         int score, int renorm, float route_scale,
                                         int32_t* status, int lane, int* out_u,
                                         float* out_w) {
  int k = kt;
  if (k < 1 || k > k_max) {
    if (lane == 0) report(status, MOE_ERR_K_RANGE);
    k = min(max(k, 0), k_max);
  }
  k = min(k, E_r);
  float v[IPL];
  uint32_t key[IPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    if (u < E_r) {
      v[i] = P[u];
    } else {
      v[i] = 0.f;
    }
  }
  // add the remaining partial rows in slice order, SB slices' loads in flight
  constexpr int SB = IPL >= 8 ? 2 : 16 / IPL;
  for (int s0 = 1; s0 < S; s0 += SB) {
    float pv[SB][IPL];
#pragma unroll
    for (int j = 0; j < SB; ++j)
#pragma unroll
      for (int i = 0; i < IPL; ++i) {
        const int u = lane + 32 * i;
        pv[j][i] = (s0 + j < S && u < E_r) ? P[static_cast<size_t>(s0 + j) * sstride + u] : 0.f;
      }
#pragma unroll
    for (int j = 0; j < SB; ++j)
#pragma unroll
      for (int i = 0; i < IPL; ++i)
        if (s0 + j < S) v[i] += pv[j][i];
  }
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    if (u < E_r) {
      if (bias != nullptr) v[i] += bias[u / n_sub];
      if (lout != nullptr) lout[u] = v[i];
      bad |= !isfinite(v[i]);
      key[i] = order_key(v[i]);
    } else {
      key[i] = 0u;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(status, MOE_ERR_NONFINITE);

  float mx = -INFINITY, sum = 0.f;
  if (score == MOE_SCORE_SOFTMAX) {
#pragma unroll
    for (int i = 0; i < IPL; ++i)
      if (lane + 32 * i < E_r) mx = fmaxf(mx, v[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
#pragma unroll
    for (int i = 0; i < IPL; ++i)
      if (lane + 32 * i < E_r) sum += expf(v[i] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  }

  // Sort all 32 * IPL units best first: a bitonic network over positions
  // p = lane * IPL + i (strides below IPL inside a lane, the rest across
  // lanes) on (key << 32 | ~u), which orders equal keys by lower index.
  unsigned long long c[IPL];
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    c[i] = u < E_r ? (static_cast<unsigned long long>(key[i]) << 32) |
                         static_cast<uint32_t>(~static_cast<uint32_t>(u))
                   : 0ull;  // below every unit, NaN ones included
  }
  constexpr int N = 32 * IPL;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= IPL) {
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, c[i], stride / IPL);
          const int p = lane * IPL + i;
          const bool take_max = ((p & stride) == 0) == ((p & size) == 0);
          c[i] = take_max ? (o > c[i] ? o : c[i]) : (o < c[i] ? o : c[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
          if ((i & stride) == 0) {
            const int j = i | stride;
            const bool desc = ((lane * IPL + i) & size) == 0;
            const unsigned long long hi = c[i] > c[j] ? c[i] : c[j];
            const unsigned long long lo = c[i] > c[j] ? c[j] : c[i];
            c[i] = desc ? hi : lo;
            c[j] = desc ? lo : hi;
          }
        }
      }
    }
  }
  // lane j takes position j (held by lane j / IPL, item j % IPL)
  unsigned long long best = 0ull;
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const unsigned long long o = __shfl_sync(0xffffffffu, c[i], lane / IPL);
    if (i == lane % IPL) best = o;
  }
  int my_u = -1;
  float my_s = 0.f;
  if (lane < k) {
    my_u = static_cast<int>(~static_cast<uint32_t>(best & 0xffffffffull));
    const float L = key_to_logit(static_cast<uint32_t>(best >> 32));
    my_s = (score == MOE_SCORE_SOFTMAX) ? expf(L - mx) / sum : 1.f / (1.f + expf(-L));
  }
  float selsum = lane < k ? my_s : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) selsum += __shfl_xor_sync(0xffffffffu, selsum, off);
  *out_u = lane < k ? my_u : -1;
  *out_w = lane < k ? (renorm ? my_s / selsum : my_s) * route_scale : 0.f;
  return k;
}

// One warp per token, eight tokens per CTA.  P holds S partial logit arrays
// [T, E_r] one after another (S = 1: finished logits).  kpt == nullptr: every
// token keeps k_max units.
template <int IPL>
__global__ void __launch_bounds__(256) topk_gate_kernel(
    const float* __restrict__ P, int S, const float* __restrict__ bias, int n_sub,
    float* __restrict__ logits_out, const int32_t* __restrict__ kpt, int T, int E_r,
    int k_max, int score, int renorm, float route_scale, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* status) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  int u;
  float w;
  const size_t row = static_cast<size_t>(t) * E_r;
  warp_topk<IPL>(P + row, S, static_cast<size_t>(T) * E_r, bias, n_sub,
                 logits_out != nullptr ? logits_out + row : nullptr,
                 kpt != nullptr ? kpt[t] : k_max, E_r, k_max, score,
                 renorm, route_scale, status, lane, &u, &w);
  if (lane < k_max) {
    const size_t o = static_cast<size_t>(t) * k_max + lane;
    topk_idx[o] = u;
    topk_w[o] = w;
  }
}

}  // namespace

// Slices of the hidden dimension for a T x E_r router: at most 1024 columns
// each (one load round trip per CTA), and enough of them (up to one per 512
// columns) that the grid has about 304 CTAs.  Returns the slice count (0: H
// unsupported) and the 16-byte vectors per slice.
int router_slices(int T, int H, int E_r, int* vs) {
  const int nv = H / 8;
  if (nv <= 0) return 0;
  const int s_min = (nv + kMaxSliceVec - 1) / kMaxSliceVec;
  const int s_max = nv / 64 > s_min ? nv / 64 : s_min;
  const long long base = static_cast<long long>((T + kTokPerCta - 1) / kTokPerCta) * ((E_r + 7) / 8);
  long long want = base > 0 ? (304 + base - 1) / base : 1;
  want = want < s_min ? s_min : (want > s_max ? s_max : want);
  int v = static_cast<int>((nv + want - 1) / want);
  v = (v + 7) & ~7;
  if (v > kMaxSliceVec) v = kMaxSliceVec;
  *vs = v;
  return (nv + v - 1) / v;
}

int router_slices_max(int H) {
  const int nv = H / 8;
  const int s_min = (nv + kMaxSliceVec - 1) / kMaxSliceVec;
  return nv / 64 > s_min ? nv / 64 + 1 : s_min + 1;
}

cudaError_t launch_router_logits_small(const void* x, const void* router_w, int T, int H,
                                       int E_r, float* partial, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  int vs = 0;
  const int S = router_slices(T, H, E_r, &vs);
  if (S <= 0 || S > router_slices_max(H)) return cudaErrorInvalidValue;
  const int smem = kTokPerCta * vs * 16;
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(router_logits_split_kernel, kTokPerCta * kMaxSliceVec * 16,
                                attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid((T + kTokPerCta - 1) / kTokPerCta, (E_r + 7) / 8, S);
  return launch_pdl(router_logits_split_kernel, grid, dim3(256), smem, s,
                    static_cast<const uint4*>(x), static_cast<const uint4*>(router_w), T, H / 8,
                    E_r, vs, partial);
}

cudaError_t launch_topk_gate(const float* partial, int S, const float* bias, int n_sub,
                             float* logits_out, const int32_t* k_per_token, int T, int E_r,
                             int k_max, int score, int renorm, float route_scale,
                             int32_t* topk_idx, float* topk_w, int32_t* status,
                             cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int grid = (T + 7) / 8;
#define MOE_TOPK_LAUNCH(IPL)                                                                 \
  launch_pdl(topk_gate_kernel<IPL>, dim3(grid), dim3(256), 0, s, partial, S, bias, n_sub,     \
             logits_out, k_per_token, T, E_r, k_max, score, renorm, route_scale, topk_idx,    \
             topk_w, status)
  if (E_r <= 32) return MOE_TOPK_LAUNCH(1);
  if (E_r <= 64) return MOE_TOPK_LAUNCH(2);
  if (E_r <= 128) return MOE_TOPK_LAUNCH(4);
  return MOE_TOPK_LAUNCH(8);
#undef MOE_TOPK_LAUNCH
}

}  // namespace moe
