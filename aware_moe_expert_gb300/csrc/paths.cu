// Path-composed execution with source-grouped reuse.  "PCoMoE: Shifting MoE
// Inference from Monolithic Expert Selection to Fine-Grained Path
// Composition" (arXiv 2609.01024), "Source-Grouped Compute Reuse" (Fig. 8):
// a path (i, j) runs the expansion side of unit i (gate|up + SiLU product)
// and the projection side of unit j (down); paths of a token that share a
// source share one expansion.  The projection is linear, so the paths of a
// token that share a target share one projection too:
//     sum_i beta_ij D_j(U_i(h)) = D_j(sum_i beta_ij U_i(h)).
// The layer therefore runs the grouped gate|up over (token, distinct source)
// pairs and the grouped down over (token, distinct target) pairs, with two
// small kernels around them:
//   paths_sources_kernel   one warp per token: the distinct values of a slot
//                          list (sources, then targets) in first-occurrence
//                          order (__match_any_sync) and each path's position
//                          among them
//   paths_merge_kernel     one warp per token: for each of its distinct
//                          targets, the down input row = the beta-weighted
//                          sum (fp32, path order) of the expansion rows of
//                          the paths into that target, stored bf16, and the
//                          combine weight 1 of that row
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) paths_sources_kernel(
    const int32_t* __restrict__ src_idx, const int32_t* __restrict__ n_paths, int T, int k_max,
    int E_r, int32_t* __restrict__ srcs, int32_t* __restrict__ n_src, int32_t* __restrict__ slot,
    int32_t* status) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int kt = n_paths[t];
  if ((kt < 1 || kt > k_max) && lane == 0) report(status, MOE_ERR_K_RANGE);
  const int k = min(max(kt, 0), k_max);
  int s = -1 - lane;   // distinct for lanes without a path
  if (lane < k) {
    const int v = src_idx[static_cast<size_t>(t) * k_max + lane];
    if (v >= 0 && v < E_r)
      s = v;
    else
      report(status, MOE_ERR_BAD_INDEX);
  }
  const uint32_t same = __match_any_sync(0xffffffffu, s);
  const int first = __ffs(same) - 1;
  const bool lead = s >= 0 && first == lane;
  const uint32_t leads = __ballot_sync(0xffffffffu, lead);
  const int pos_first = __popc(leads & ((1u << first) - 1u));   // position of my source
  const size_t o = static_cast<size_t>(t) * k_max;
  if (lead) srcs[o + pos_first] = s;
  const int ns = __popc(leads);
  if (lane >= ns && lane < k_max) srcs[o + lane] = -1;
  if (lane < k_max) slot[o + lane] = (lane < k && s >= 0) ? pos_first : -1;
  if (lane == 0) n_src[t] = ns;
}

__global__ void __launch_bounds__(256) paths_merge_kernel(
    const int32_t* __restrict__ n_paths, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ tslot, const int32_t* __restrict__ n_tgt,
    const float* __restrict__ beta, const int32_t* __restrict__ inv_src,
    const int32_t* __restrict__ inv_tgt, const uint4* __restrict__ act_src, int T, int k_max,
    int I_sub, long long n_src_rows, long long n_tgt_rows, uint4* __restrict__ act_tgt,
    float* __restrict__ w_tgt, int32_t* status) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const size_t o = static_cast<size_t>(t) * k_max;
  const int k = min(max(n_paths[t], 0), k_max);
  const int nt = min(max(n_tgt[t], 0), k_max);
  // lane j holds path j: its target slot, the expansion row it reads, beta
  int my_ts = -1, my_row = -1;
  float my_b = 0.0f;
  if (lane < k) {
    my_ts = tslot[o + lane];
    const int sl = slot[o + lane];
    if (sl >= 0 && sl < k_max) my_row = inv_src[o + sl];
    my_b = beta[o + lane];
    if (my_ts < 0 || my_row < 0 || my_row >= n_src_rows) {
      report(status, MOE_ERR_BAD_INDEX);
      my_ts = -1;
    }
  }
  const int vecs = I_sub / 8;   // 16-byte vectors of 8 bf16 per row
  for (int ts = 0; ts < nt; ++ts) {
    const int pos = inv_tgt[o + ts];
    if (pos < 0 || pos >= n_tgt_rows) {
      if (lane == 0) report(status, MOE_ERR_BAD_INDEX);
      continue;
    }
    const uint32_t members = __ballot_sync(0xffffffffu, my_ts == ts);
    // every lane runs every iteration (the shuffles need the whole warp);
    // lanes past the row's end load and store nothing
    for (int v0 = 0; v0 < vecs; v0 += 32) {
      const int v = v0 + lane;
      const bool live = v < vecs;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
      uint32_t m = members;
      while (m != 0u) {
        const int j = __ffs(m) - 1;
        m &= m - 1u;
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        const float b = __shfl_sync(0xffffffffu, my_b, j);
        if (live) {
          const uint4 q = act_src[static_cast<size_t>(row) * vecs + v];
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(b, __uint_as_float(w4[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(b, __uint_as_float(w4[e] & 0xffff0000u), acc[2 * e + 1]);
          }
        }
      }
      if (live) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
        act_tgt[static_cast<size_t>(pos) * vecs + v] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    if (lane == 0) w_tgt[o + ts] = 1.0f;
  }
}

}  // namespace

cudaError_t launch_paths_sources(const int32_t* src_idx, const int32_t* n_paths, int T, int k_max,
                                 int E_r, int32_t* srcs, int32_t* n_src, int32_t* slot,
                                 int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (k_max > 32) return cudaErrorInvalidValue;
  return launch_pdl(paths_sources_kernel, dim3((T + 7) / 8), dim3(256), 0, s, src_idx, n_paths, T,
                    k_max, E_r, srcs, n_src, slot, status);
}

cudaError_t launch_paths_merge(const int32_t* n_paths, const int32_t* slot, const int32_t* tslot,
                               const int32_t* n_tgt, const float* beta, const int32_t* inv_src,
                               const int32_t* inv_tgt, const void* act_src, int T, int k_max,
                               int I_sub, long long n_src_rows, long long n_tgt_rows,
                               void* act_tgt, float* w_tgt, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (k_max > 32 || I_sub % 8 != 0) return cudaErrorInvalidValue;
  return launch_pdl(paths_merge_kernel, dim3((T + 7) / 8), dim3(256), 0, s, n_paths, slot, tslot,
                    n_tgt, beta, inv_src, inv_tgt, static_cast<const uint4*>(act_src), T, k_max,
                    I_sub, n_src_rows, n_tgt_rows, static_cast<uint4*>(act_tgt), w_tgt, status);
}

}  // namespace moe
