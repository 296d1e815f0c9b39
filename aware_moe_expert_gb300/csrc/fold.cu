// Decode expert-pool folding: rewrites a batch's routing so that only a pool
// of D units runs.  "ExFold: Unified Expert Folding for Training-Free MoE
// Prefill-Decode Acceleration" (arXiv 2608.24938), "Phase-Specific Routing and
// Folding": decode cost follows the distinct experts a batch activates, so
// the batch keeps a pool of D experts (dynamic: ranked by aggregate routed
// contribution; or static) and every other route is remapped to its
// minimum-loss pool target, its router weight scaled by the calibrated
// scalar S[source, target]; routes of a token that land on one target are
// coalesced so the target runs once.  Folding changes routing metadata only.
//
//   fold_score_kernel   one CTA per 64-token block: the block's routed weight
//                       per unit, summed token by token (a dense [64, E_r]
//                       tile in shared memory, each column added in order)
//   fold_pool_kernel    one CTA: block sums added in block order, times the
//                       unit scale; pool = the D best units (score descending,
//                       lower index on ties: rank by counting)
//   fold_map_kernel     one warp per unit: its target (itself, or the pool
//                       member of least L, lower index on ties) and scale
//                       S[u, target]
//   fold_remap_kernel   one warp per token: remap each route, merge the routes
//                       to one target in slot order (__match_any_sync), pack
//                       the targets in first-occurrence order; new k_t
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kFoldBlock = 64;   // tokens per partial score

__global__ void __launch_bounds__(256) fold_score_kernel(const int32_t* __restrict__ topk_idx,
                                                         const float* __restrict__ topk_w,
                                                         const int32_t* __restrict__ kpt, int T,
                                                         int k_max, int E_r,
                                                         float* __restrict__ part,
                                                         int32_t* status) {
  extern __shared__ float tile[];  // [kFoldBlock][E_r]
  pdl_wait_and_trigger();
  const int t0 = blockIdx.x * kFoldBlock;
  const int nt = min(kFoldBlock, T - t0);
  for (int i = threadIdx.x; i < kFoldBlock * E_r; i += blockDim.x) tile[i] = 0.f;
  __syncthreads();
  for (int i = threadIdx.x; i < nt * k_max; i += blockDim.x) {
    const int tt = i / k_max, j = i - tt * k_max;
    const int t = t0 + tt;
    const int k = kpt[t];
    if (k < 1 || k > k_max) {
      if (j == 0) report(status, MOE_ERR_K_RANGE);
      continue;
    }
    if (j >= k) continue;
    const int u = topk_idx[static_cast<size_t>(t) * k_max + j];
    if (u < 0 || u >= E_r) {
      report(status, MOE_ERR_BAD_INDEX);
      continue;
    }
    // the units of one token are distinct, so no two slots share a cell
    tile[tt * E_r + u] = topk_w[static_cast<size_t>(t) * k_max + j];
  }
  __syncthreads();
  for (int u = threadIdx.x; u < E_r; u += blockDim.x) {
    float s = 0.f;
    for (int tt = 0; tt < nt; ++tt) s += tile[tt * E_r + u];
    part[static_cast<size_t>(blockIdx.x) * E_r + u] = s;
  }
}

__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;
  uint32_t b = __float_as_uint(s);
  if ((b & 0x7fffffffu) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One CTA of 256 threads, thread u <-> unit u: the pool (in_pool flags and
// the members in ascending order, n of them).
__global__ void __launch_bounds__(256) fold_pool_kernel(
    const float* __restrict__ part, int n_blocks, int E_r, int D,
    const int32_t* __restrict__ pool_in, const float* __restrict__ unit_scale,
    int32_t* __restrict__ in_pool, int32_t* __restrict__ pool_list, int32_t* __restrict__ n_out,
    int32_t* __restrict__ pool_out, int32_t* status) {
  __shared__ uint32_t s_key[256];
  __shared__ int s_in[256];
  __shared__ int s_wcnt[8];
  pdl_wait_and_trigger();
  const int u = threadIdx.x, warp = u >> 5, lane = u & 31;
  if (pool_in == nullptr) {
    float sc = 0.f;
    if (u < E_r) {
      for (int b = 0; b < n_blocks; ++b) sc += part[static_cast<size_t>(b) * E_r + u];
      if (unit_scale != nullptr) sc *= unit_scale[u];
    }
    s_key[u] = u < E_r ? score_key(sc) : 0u;
    __syncthreads();
    int rank = 0;
    if (u < E_r) {
      const uint32_t ku = s_key[u];
      for (int v = 0; v < E_r; ++v) {
        const uint32_t kv = s_key[v];
        rank += (kv > ku || (kv == ku && v < u)) ? 1 : 0;
      }
    }
    s_in[u] = (u < E_r && rank < D) ? 1 : 0;
  } else {
    s_in[u] = 0;
    __syncthreads();
    if (u < D) {
      const int p = pool_in[u];
      if (p < 0 || p >= E_r || atomicExch(&s_in[p], 1) != 0) report(status, MOE_ERR_BAD_INDEX);
    }
  }
  __syncthreads();
  // members in ascending order: warp ballots, then the counts of earlier warps
  const int flag = s_in[u];
  const uint32_t m = __ballot_sync(0xffffffffu, flag != 0);
  if (lane == 0) s_wcnt[warp] = __popc(m);
  __syncthreads();
  int before = 0, n = 0;
  for (int w2 = 0; w2 < 8; ++w2) {
    before += w2 < warp ? s_wcnt[w2] : 0;
    n += s_wcnt[w2];
  }
  if (u < E_r) in_pool[u] = flag;
  if (flag) {
    const int pos = before + __popc(m & ((1u << lane) - 1u));
    pool_list[pos] = u;
    if (pool_out != nullptr) pool_out[pos] = u;
  }
  if (u == 0) *n_out = n;
}

// One warp per unit: the target (itself when in the pool, else the pool
// member of least L[u, p], a NaN loss counting as +inf, lower index on ties)
// and the scale S[u, target].
__global__ void __launch_bounds__(256) fold_map_kernel(
    int E_r, const int32_t* __restrict__ in_pool, const int32_t* __restrict__ pool_list,
    const int32_t* __restrict__ n_in, const float* __restrict__ S, const float* __restrict__ L,
    int32_t* __restrict__ tgt, float* __restrict__ scale) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * 8 + warp;
  if (u >= E_r) return;
  if (in_pool[u]) {
    if (lane == 0) {
      tgt[u] = u;
      scale[u] = 1.f;
    }
    return;
  }
  const int n = *n_in;
  float best = INFINITY;
  int bp = 0x7fffffff;
  for (int i = lane; i < n; i += 32) {
    const int p = pool_list[i];
    float l = L[static_cast<size_t>(u) * E_r + p];
    if (l != l) l = INFINITY;
    if (l < best || (l == best && p < bp)) {
      best = l;
      bp = p;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ol = __shfl_xor_sync(0xffffffffu, best, off);
    const int op = __shfl_xor_sync(0xffffffffu, bp, off);
    if (ol < best || (ol == best && op < bp)) {
      best = ol;
      bp = op;
    }
  }
  if (lane == 0) {
    const int t = bp < E_r ? bp : u;
    tgt[u] = t;
    scale[u] = t == u ? 1.f : S[static_cast<size_t>(u) * E_r + t];
  }
}

// One warp per token.
__global__ void __launch_bounds__(256) fold_remap_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ kpt, int T, int k_max, int E_r, const int32_t* __restrict__ tgt,
    const float* __restrict__ scale, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
    int32_t* __restrict__ k_out, int32_t* status) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int kt = kpt[t];
  if ((kt < 1 || kt > k_max) && lane == 0) report(status, MOE_ERR_K_RANGE);
  const int k = min(max(kt, 0), k_max);
  int v = -1 - lane;   // distinct for inactive lanes
  float w = 0.f;
  if (lane < k) {
    const int u = topk_idx[static_cast<size_t>(t) * k_max + lane];
    if (u >= 0 && u < E_r) {
      v = tgt[u];
      w = topk_w[static_cast<size_t>(t) * k_max + lane];
      if (v != u) w = w * scale[u];
    } else {
      report(status, MOE_ERR_BAD_INDEX);
    }
  }
  const uint32_t same = __match_any_sync(0xffffffffu, v);
  const bool lead = v >= 0 && (__ffs(same) - 1) == lane;
  // merge the lanes of one target in slot (lane) order, starting from the first
  float acc = 0.f;
  bool first = true;
  for (int s = 0; s < 32; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (lead && ((same >> s) & 1u)) {
      acc = first ? ws : acc + ws;
      first = false;
    }
  }
  const uint32_t leads = __ballot_sync(0xffffffffu, lead);
  const int kn = __popc(leads);
  const size_t o = static_cast<size_t>(t) * k_max;
  if (lead) {
    const int pos = __popc(leads & ((1u << lane) - 1u));
    idx_out[o + pos] = v;
    w_out[o + pos] = acc;
  }
  if (lane >= kn && lane < k_max) {
    idx_out[o + lane] = -1;
    w_out[o + lane] = 0.f;
  }
  if (lane == 0) k_out[t] = kn;
}

}  // namespace

size_t fold_workspace_bytes(int T, int E_r) {
  const size_t nb = static_cast<size_t>((T + kFoldBlock - 1) / kFoldBlock);
  return nb * E_r * 4 + 4 * static_cast<size_t>(E_r) * 4 + 16;
}

cudaError_t launch_fold_decode(const int32_t* topk_idx, const float* topk_w,
                               const int32_t* k_per_token, int T, int k_max, int E_r, int D,
                               const int32_t* pool_in, const float* unit_scale, const float* S,
                               const float* L, int32_t* idx_out, float* w_out, int32_t* k_out,
                               int32_t* pool_out, void* ws, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (E_r > 256 || k_max > 32) return cudaErrorInvalidValue;
  const int nb = (T + kFoldBlock - 1) / kFoldBlock;
  float* part = static_cast<float*>(ws);
  int32_t* tgt = reinterpret_cast<int32_t*>(part + static_cast<size_t>(nb) * E_r);
  float* scale = reinterpret_cast<float*>(tgt + E_r);
  int32_t* in_pool = reinterpret_cast<int32_t*>(scale + E_r);
  int32_t* pool_list = in_pool + E_r;
  int32_t* n_pool = pool_list + E_r;
  cudaError_t e;
  if (pool_in == nullptr) {
    const int smem = kFoldBlock * E_r * 4;
    static bool attr_done[64] = {false};
    e = set_smem_once(fold_score_kernel, kFoldBlock * 256 * 4, attr_done);
    if (e != cudaSuccess) return e;
    e = launch_pdl(fold_score_kernel, dim3(nb), dim3(256), smem, s, topk_idx, topk_w,
                   k_per_token, T, k_max, E_r, part, status);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(fold_pool_kernel, dim3(1), dim3(256), 0, s, static_cast<const float*>(part), nb,
                 E_r, D, pool_in, unit_scale, in_pool, pool_list, n_pool, pool_out, status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fold_map_kernel, dim3((E_r + 7) / 8), dim3(256), 0, s, E_r,
                 static_cast<const int32_t*>(in_pool), static_cast<const int32_t*>(pool_list),
                 static_cast<const int32_t*>(n_pool), S, L, tgt, scale);
  if (e != cudaSuccess) return e;
  return launch_pdl(fold_remap_kernel, dim3((T + 7) / 8), dim3(256), 0, s, topk_idx, topk_w,
                    k_per_token, T, k_max, E_r, static_cast<const int32_t*>(tgt),
                    static_cast<const float*>(scale), idx_out, w_out, k_out, status);
}

}  // namespace moe
