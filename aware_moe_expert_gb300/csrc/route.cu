// Router: logits on CUDA cores for small token counts, and the warp-per-token
// top-k_t selection with softmax / sigmoid gates.
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

// logits[t, u] = x_t . router_w[u] + bias[u / n_sub].  CTA = up to 8
// tokens x 8 units.  The CTA's x rows are first staged in shared memory
// (every thread's loads in flight at once); then one warp per unit streams
// its router row with eight independent 16-byte loads per lane per pass.
__global__ void __launch_bounds__(256) router_logits_small_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ rw,
    const float* __restrict__ bias, int T, int H, int E_r, int n_sub, int tok_per_cta,
    float* __restrict__ logits) {
  extern __shared__ uint4 xs[];  // [tok_per_cta][H / 8]
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.y * 8 + warp;
  const int t0 = blockIdx.x * tok_per_cta;
  const int nt = min(tok_per_cta, T - t0);
  const int nv = H / 8;
  const uint4* xg = reinterpret_cast<const uint4*>(x) + static_cast<size_t>(t0) * nv;
  // eight 16-byte loads per thread in flight before they are stored
  const int total = nt * nv;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * blockDim.x) {
    uint4 tmp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = i0 + q * blockDim.x;
      tmp[q] = i < total ? __ldg(xg + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = i0 + q * blockDim.x;
      if (i < total) xs[i] = tmp[q];
    }
  }
  __syncthreads();
  if (u >= E_r) return;
  float acc[kTokPerCta];
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) acc[i] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(rw + static_cast<size_t>(u) * H);
  for (int v0 = lane; v0 < nv; v0 += 256) {
    uint4 wv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      wv[q] = v0 + 32 * q < nv ? __ldg(wrow + v0 + 32 * q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (v0 + 32 * q < nv) {
#pragma unroll
        for (int i = 0; i < kTokPerCta; ++i)
          if (i < nt) acc[i] = dot8_bf16(xs[i * nv + v0 + 32 * q], wv[q], acc[i]);
      }
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
  if (lane < nt) {
    const float b = bias != nullptr ? bias[u / n_sub] : 0.f;
    logits[static_cast<size_t>(t0 + lane) * E_r + u] = mine + b;
  }
}

// Total order used for selection: larger logit first; -0 == +0; NaN below
// every number.  The key is monotone in the logit.
__device__ __forceinline__ uint32_t order_key(float L) {
  if (L != L) return 0u;
  uint32_t b = __float_as_uint(L);
  if ((b & 0x7fffffffu) == 0u) b = 0u;  // -0 is +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One warp selects the k_t best units of one token.  Lane l holds units l,
// l+32, ... (IPL per lane).  Round j picks the best remaining unit with a
// 64-bit warp max over (key << 32 | ~u), so equal keys resolve to the lower
// unit index.  On return lane j < k holds the j-th unit (*out_u) and its gate
// weight after renormalisation and route_scale (*out_w); returns k.
template <int IPL>
__device__ __forceinline__ int warp_topk(const float* __restrict__ row, int kt, int E_r, int k_max,
                                         int score, int renorm, float route_scale,
                                         int32_t* status, int lane, int* out_u, float* out_w) {
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
      const float L = row[u];
      bad |= !isfinite(L);
      v[i] = L;
      key[i] = order_key(L);
    } else {
      v[i] = 0.f;
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

  uint32_t taken = 0;
  int my_u = -1;
  float my_s = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
      const int u = lane + 32 * i;
      if (u < E_r && !((taken >> i) & 1u)) {
        const unsigned long long c =
            (static_cast<unsigned long long>(key[i]) << 32) | static_cast<uint32_t>(~u);
        best = c > best ? c : best;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    const int u = static_cast<int>(~static_cast<uint32_t>(best & 0xffffffffull));
    const int owner = u & 31, item = u >> 5;
    float s_local = 0.f;
    if (lane == owner) {
      float L = 0.f;
#pragma unroll
      for (int i = 0; i < IPL; ++i)
        if (i == item) L = v[i];
      taken |= 1u << item;
      s_local = (score == MOE_SCORE_SOFTMAX) ? expf(L - mx) / sum : 1.f / (1.f + expf(-L));
    }
    const float s = __shfl_sync(0xffffffffu, s_local, owner);
    if (lane == j) {
      my_u = u;
      my_s = s;
    }
  }
  float selsum = lane < k ? my_s : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) selsum += __shfl_xor_sync(0xffffffffu, selsum, off);
  *out_u = lane < k ? my_u : -1;
  *out_w = lane < k ? (renorm ? my_s / selsum : my_s) * route_scale : 0.f;
  return k;
}

// One warp per token, eight tokens per CTA.
template <int IPL>
__global__ void __launch_bounds__(256) topk_gate_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ kpt, int T, int E_r,
    int k_max, int score, int renorm, float route_scale, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* status) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  int u;
  float w;
  warp_topk<IPL>(logits + static_cast<size_t>(t) * E_r, kpt[t], E_r, k_max, score, renorm,
                 route_scale, status, lane, &u, &w);
  if (lane < k_max) {
    const size_t o = static_cast<size_t>(t) * k_max + lane;
    topk_idx[o] = u;
    topk_w[o] = w;
  }
}

}  // namespace

cudaError_t launch_router_logits_small(const void* x, const void* router_w,
                                       const float* expert_bias, int T, int H, int E_r,
                                       int n_sub, float* logits, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  // staged x rows: at most 96 KB of shared memory per CTA
  const int row_bytes = H * 2;
  int tpc = (96 * 1024) / row_bytes;
  tpc = tpc < 1 ? 1 : (tpc > kTokPerCta ? kTokPerCta : tpc);
  const int smem = tpc * row_bytes;
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(router_logits_small_kernel, 96 * 1024, attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid((T + tpc - 1) / tpc, (E_r + 7) / 8);
  return launch_pdl(router_logits_small_kernel, grid, dim3(256), smem, s,
                    static_cast<const __nv_bfloat16*>(x),
                    static_cast<const __nv_bfloat16*>(router_w), expert_bias, T, H, E_r, n_sub,
                    tpc, logits);
}

cudaError_t launch_topk_gate(const float* logits, const int32_t* k_per_token, int T, int E_r,
                             int k_max, int score, int renorm, float route_scale,
                             int32_t* topk_idx, float* topk_w, int32_t* status,
                             cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int grid = (T + 7) / 8;
  if (E_r <= 32)
    return launch_pdl(topk_gate_kernel<1>, dim3(grid), dim3(256), 0, s, logits, k_per_token, T,
                      E_r, k_max, score, renorm, route_scale, topk_idx, topk_w, status);
  else if (E_r <= 64)
    return launch_pdl(topk_gate_kernel<2>, dim3(grid), dim3(256), 0, s, logits, k_per_token, T,
                      E_r, k_max, score, renorm, route_scale, topk_idx, topk_w, status);
  else if (E_r <= 128)
    return launch_pdl(topk_gate_kernel<4>, dim3(grid), dim3(256), 0, s, logits, k_per_token, T,
                      E_r, k_max, score, renorm, route_scale, topk_idx, topk_w, status);
  else
    return launch_pdl(topk_gate_kernel<8>, dim3(grid), dim3(256), 0, s, logits, k_per_token, T,
                      E_r, k_max, score, renorm, route_scale, topk_idx, topk_w, status);
}

}  // namespace moe
