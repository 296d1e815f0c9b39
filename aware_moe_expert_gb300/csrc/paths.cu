// Path-composed execution with source-grouped reuse.  "PCoMoE: Shifting MoE
// Inference from Monolithic Expert Selection to Fine-Grained Path
// Composition" (arXiv 2609.01024), "Source-Grouped Compute Reuse" (Fig. 8):
// a path (i, j) runs the expansion side of unit i (gate|up + SiLU product)
// and the projection side of unit j (down); paths of a token that share a
// source share one expansion.  The layer therefore runs the grouped gate|up
// over (token, unique source) pairs and the grouped down over paths, with two
// small kernels in between:
//   paths_sources_kernel   one warp per token: the distinct sources in
//                          first-occurrence order (__match_any_sync) and each
//                          path's position among them
//   paths_rows_kernel      one thread per path: the expansion row (in the
//                          source-sorted order) the path's down row reads
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

__global__ void __launch_bounds__(256) paths_rows_kernel(
    const int32_t* __restrict__ n_paths, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ inv_src, const int32_t* __restrict__ inv_tgt, int T, int k_max,
    int32_t* __restrict__ row_of) {
  pdl_wait_and_trigger();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(T) * k_max) return;
  const int t = static_cast<int>(i / k_max), j = static_cast<int>(i - static_cast<long long>(t) * k_max);
  const int k = min(max(n_paths[t], 0), k_max);
  if (j >= k) return;
  const int pos = inv_tgt[i];
  const int sl = slot[i];
  if (pos < 0 || sl < 0) return;
  row_of[pos] = inv_src[static_cast<size_t>(t) * k_max + sl];
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

cudaError_t launch_paths_rows(const int32_t* n_paths, const int32_t* slot, const int32_t* inv_src,
                              const int32_t* inv_tgt, int T, int k_max, int32_t* row_of,
                              cudaStream_t s) {
  const long long n = static_cast<long long>(T) * k_max;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(paths_rows_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    s, n_paths, slot, inv_src, inv_tgt, T, k_max, row_of);
}

}  // namespace moe
