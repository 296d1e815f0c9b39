// Weighted combine: out_t = sum_{j < k_t} w_{t,j} * y_perm[inv_row(t,j)]
// (+ the shared expert's y_shared[t]), fp32 accumulation in j order, one
// rounding to bf16.  MoE-Prism (arXiv 2510.19366) §III-B2: the routed output
// of a token is the gate-weighted sum of its selected units' FFN outputs.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// One warp per token; lanes stride over H in 16-byte (8 x bf16) vectors.
// Lane j caches (row, weight) of slot j and broadcasts it in the j loop.
__global__ void __launch_bounds__(256) combine_kernel(
    const uint4* __restrict__ y_perm, const uint4* __restrict__ y_shared,
    const int32_t* __restrict__ inv_row, const float* __restrict__ topk_w,
    const int32_t* __restrict__ kpt, int T, int nv, int k_max, int n_rows,
    uint4* __restrict__ out, int32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int k = min(max(kpt[t], 0), k_max);
  int my_r = -1;
  float my_w = 0.f;
  if (lane < k) {
    my_r = inv_row[static_cast<size_t>(t) * k_max + lane];
    my_w = topk_w[static_cast<size_t>(t) * k_max + lane];
    if (my_r < 0 || my_r >= n_rows) {
      report(status, MOE_ERR_BAD_INDEX);
      my_r = -1;
    }
  }
  for (int v = lane; v < nv; v += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, my_r, j);
      const float w = __shfl_sync(0xffffffffu, my_w, j);
      if (r < 0) continue;
      const uint4 y = __ldg(y_perm + static_cast<size_t>(r) * nv + v);
      const uint32_t yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, bf16lo(yv[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, bf16hi(yv[i]), acc[2 * i + 1]);
      }
    }
    if (y_shared != nullptr) {
      const uint4 y = __ldg(y_shared + static_cast<size_t>(t) * nv + v);
      const uint32_t yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16lo(yv[i]);
        acc[2 * i + 1] += bf16hi(yv[i]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[static_cast<size_t>(t) * nv + v] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const void* y_perm, const void* y_shared, const int32_t* inv_row,
                           const float* topk_w, const int32_t* k_per_token, int T, int H,
                           int k_max, int n_rows, void* out, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  combine_kernel<<<(T + 7) / 8, 256, 0, s>>>(
      static_cast<const uint4*>(y_perm), static_cast<const uint4*>(y_shared), inv_row, topk_w,
      k_per_token, T, H / 8, k_max, n_rows, static_cast<uint4*>(out), status);
  return cudaGetLastError();
}

}  // namespace moe
