// Permutation of the routed assignments into unit-contiguous rows, and the
// row gather that feeds the grouped GEMM.
//
// MoE-Prism (arXiv 2510.19366) §II-D: grouped-GEMM MoE kernels need the
// token rows of one expert contiguous.  The order is fixed so the result is
// bit-reproducible: unit ascending, token ascending inside a unit.
//
// Deterministic without position atomics: a membership bitmap
// bitmap[u][w] (bit b of word w = token 32w+b selected u) is built per
// 32-token block in shared memory (atomicOr only merges bits, so the result
// does not depend on order).  One CTA then turns per-word popcounts into
// per-unit word prefixes and the unit offsets, and the rank of (t, u) inside
// unit u is offsets[u] + prefix[u][t/32] + popcount(bits of earlier tokens).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// One CTA per 32-token word.  bits[u] collects the tokens of this word that
// selected unit u; invalid or repeated unit indices are reported.
__global__ void __launch_bounds__(256) bitmap_kernel(const int32_t* __restrict__ topk_idx,
                                                      const int32_t* __restrict__ kpt, int T,
                                                      int k_max, int E_r, int W,
                                                      uint32_t* __restrict__ bitmap,
                                                      int32_t* status) {
  __shared__ uint32_t bits[256];
  pdl_wait_and_trigger();
  for (int u = threadIdx.x; u < E_r; u += blockDim.x) bits[u] = 0u;
  __syncthreads();
  const int word = blockIdx.x;
  // a thread's slots (at most 32 * 32 / 256 = 4): every load in flight at once
  constexpr int kPer = 4;
  int kk[kPer], uu[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int i = threadIdx.x + r * blockDim.x;
    const int t = word * 32 + i / k_max;
    const bool in = i < 32 * k_max && t < T;
    kk[r] = in ? kpt[t] : 0;
    uu[r] = in ? topk_idx[static_cast<size_t>(word) * 32 * k_max + i] : -1;
  }
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int i = threadIdx.x + r * blockDim.x;
    const int tl = i / k_max, j = i - tl * k_max;
    const int t = word * 32 + tl;
    if (i >= 32 * k_max || t >= T) continue;
    int k = kk[r];
    if (k < 1 || k > k_max) {
      if (j == 0) report(status, MOE_ERR_K_RANGE);
      k = min(max(k, 0), k_max);
    }
    if (j >= k) continue;
    const int u = uu[r];
    if (u < 0 || u >= E_r) {
      report(status, MOE_ERR_BAD_INDEX);
      continue;
    }
    const uint32_t bit = 1u << tl;
    const uint32_t old = atomicOr(&bits[u], bit);
    if (old & bit) report(status, MOE_ERR_BAD_INDEX);
  }
  __syncthreads();
  for (int u = threadIdx.x; u < E_r; u += blockDim.x)
    bitmap[static_cast<size_t>(u) * W + word] = bits[u];
}

// One warp per unit: per-word popcounts of the unit's bitmap row turned
// into exclusive word prefixes, and the unit's count.
__global__ void __launch_bounds__(256) unit_scan_kernel(const uint32_t* __restrict__ bitmap,
                                                         int E_r, int W,
                                                         int32_t* __restrict__ wprefix,
                                                         int32_t* __restrict__ counts) {
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * 8 + warp;
  if (u >= E_r) return;
  const uint32_t* row = bitmap + static_cast<size_t>(u) * W;
  int32_t* pre = wprefix + static_cast<size_t>(u) * W;
  int running = 0;
  for (int w0 = 0; w0 < W; w0 += 32) {
    const int w = w0 + lane;
    const int c = w < W ? __popc(row[w]) : 0;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (w < W) pre[w] = running + incl - c;
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) counts[u] = running;
}

// Exclusive scan of counts[0..E_r) by warp 0 into s_off[0..E_r].
__device__ __forceinline__ void scan_counts(const int32_t* counts, int E_r, int32_t* s_off,
                                            int lane) {
  const int per = (E_r + 31) / 32;
  const int u0 = lane * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (u0 + i < E_r) local += counts[u0 + i];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - local;
  for (int i = 0; i < per; ++i) {
    const int u = u0 + i;
    if (u < E_r) {
      s_off[u] = run;
      run += counts[u];
    }
  }
  if (lane == 31) s_off[E_r] = incl;
}

// One thread per (t, j) slot.  Every CTA rebuilds the unit offsets from the
// counts (E_r <= 256) in shared memory; CTA 0 also stores them.
__global__ void __launch_bounds__(256) scatter_kernel(
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ kpt, int T, int k_max,
    int E_r, int W, const uint32_t* __restrict__ bitmap, const int32_t* __restrict__ wprefix,
    const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_row,
    int32_t* __restrict__ zero_ptr, int zero_n) {
  __shared__ int32_t s_off[257];
  pdl_wait_and_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_n; i += gridDim.x * blockDim.x)
    zero_ptr[i] = 0;
  if (threadIdx.x < 32) scan_counts(counts, E_r, s_off, threadIdx.x);
  __syncthreads();
  if (blockIdx.x == 0)
    for (int u = threadIdx.x; u <= E_r; u += blockDim.x) offsets[u] = s_off[u];
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(T) * k_max) return;
  const int t = static_cast<int>(i / k_max), j = static_cast<int>(i - static_cast<long long>(t) * k_max);
  const int kt = kpt[t];
  const int u = topk_idx[i];   // read with k_t (unused past it)
  const int k = min(max(kt, 0), k_max);
  int pos = -1;
  if (j < k) {
    if (u >= 0 && u < E_r) {
      const int w = t >> 5;
      const uint32_t below = (1u << (t & 31)) - 1u;
      const size_t o = static_cast<size_t>(u) * W + w;
      pos = s_off[u] + wprefix[o] + __popc(bitmap[o] & below);
      sorted_token[pos] = t;
    }
  }
  inv_row[i] = pos;
}

// x_perm[r] = x[sorted_token[r]] for r < offsets[E_r]; one warp per row,
// 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ sorted_token,
                                                           const int32_t* __restrict__ offsets,
                                                           int E_r, int T, int nv, int n_cap,
                                                           uint4* __restrict__ x_perm,
                                                           int32_t* status,
                                                           int32_t* __restrict__ zero_ptr,
                                                           int zero_n) {
  pdl_wait_and_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_n; i += gridDim.x * blockDim.x)
    zero_ptr[i] = 0;
  const int n = min(offsets[E_r], n_cap);
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int r = gw; r < n; r += nw) {
    const int t = sorted_token[r];
    uint4* dst = x_perm + static_cast<size_t>(r) * nv;
    if (t < 0 || t >= T) {
      if (lane == 0) report(status, MOE_ERR_BAD_INDEX);
      for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* src = x + static_cast<size_t>(t) * nv;
    for (int v = lane; v < nv; v += 32) dst[v] = __ldg(src + v);
  }
}

// Decode-sized batches in one CTA (1024 threads): bitmap, word prefixes,
// offsets and scatter all in shared memory (W = ceil(T/32) <= 8 words per
// unit, T < kPermuteBitmapMinT).  Same result as bitmap_kernel + scan_kernel +
// scatter_kernel.
__global__ void __launch_bounds__(1024) permute_small_kernel(
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ kpt, int T, int k_max,
    int E_r, int W, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_row, int32_t* status,
    int32_t* __restrict__ zero_ptr, int zero_n) {
  extern __shared__ uint32_t sm[];
  uint32_t* bits = sm;
  int32_t* pre = reinterpret_cast<int32_t*>(sm + E_r * W);
  int32_t* s_cnt = pre + E_r * W;
  int32_t* s_off = s_cnt + 256;
  pdl_wait_and_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < zero_n; i += blockDim.x) zero_ptr[i] = 0;
  for (int i = tid; i < E_r * W; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  const int slots = T * k_max;
  for (int i = tid; i < slots; i += blockDim.x) {
    const int t = i / k_max, j = i - (i / k_max) * k_max;
    int k = kpt[t];
    if (k < 1 || k > k_max) {
      if (j == 0) report(status, MOE_ERR_K_RANGE);
      k = min(max(k, 0), k_max);
    }
    if (j >= k) continue;
    const int u = topk_idx[i];
    if (u < 0 || u >= E_r) {
      report(status, MOE_ERR_BAD_INDEX);
      continue;
    }
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bits[u * W + (t >> 5)], bit) & bit) report(status, MOE_ERR_BAD_INDEX);
  }
  __syncthreads();
  for (int u = warp; u < E_r; u += 32) {
    const int c = lane < W ? __popc(bits[u * W + lane]) : 0;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane < W) pre[u * W + lane] = incl - c;
    if (lane == 31) s_cnt[u] = incl;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (E_r + 31) / 32;
    const int u0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
      if (u0 + i < E_r) local += s_cnt[u0 + i];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int u = u0 + i;
      if (u < E_r) {
        s_off[u] = run;
        offsets[u] = run;
        counts[u] = s_cnt[u];
        run += s_cnt[u];
      }
    }
    if (lane == 31) offsets[E_r] = incl;
  }
  __syncthreads();
  for (int i = tid; i < slots; i += blockDim.x) {
    const int t = i / k_max, j = i - (i / k_max) * k_max;
    const int k = min(max(kpt[t], 0), k_max);
    int pos = -1;
    if (j < k) {
      const int u = topk_idx[i];
      if (u >= 0 && u < E_r) {
        const int o = u * W + (t >> 5);
        pos = s_off[u] + pre[o] + __popc(bits[o] & ((1u << (t & 31)) - 1u));
        sorted_token[pos] = t;
      }
    }
    inv_row[i] = pos;
  }
}

}  // namespace

cudaError_t launch_permute(const int32_t* topk_idx, const int32_t* k_per_token, int T,
                           int k_max, int E_r, uint32_t* bitmap, int32_t* wprefix,
                           int32_t* counts, int32_t* offsets, int32_t* sorted_token,
                           int32_t* inv_row, int32_t* status, cudaStream_t s,
                           bool bitmap_ready, int32_t* zero_ptr, int zero_n) {
  const int W = (T + 31) / 32;
  static_assert(kPermuteBitmapMinT <= 8 * 32 + 1, "the one-CTA path takes W <= 8");
  if (T > 0 && T < kPermuteBitmapMinT) {
    const int smem = (2 * E_r * W + 256 + 257) * 4;
    static bool attr_done[64] = {false};
    cudaError_t e = set_smem_once(permute_small_kernel, (2 * 256 * 8 + 256 + 257) * 4, attr_done);
    if (e != cudaSuccess) return e;
    return launch_pdl(permute_small_kernel, dim3(1), dim3(1024), smem, s, topk_idx, k_per_token,
                      T, k_max, E_r, W, counts, offsets, sorted_token, inv_row, status, zero_ptr,
                      zero_n);
  }
  if (W > 0 && !bitmap_ready) {
    cudaError_t e = launch_pdl(bitmap_kernel, dim3(W), dim3(256), 0, s, topk_idx, k_per_token, T,
                               k_max, E_r, W, bitmap, status);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(unit_scan_kernel, dim3((E_r + 7) / 8), dim3(256), 0, s,
                             static_cast<const uint32_t*>(bitmap), E_r, W, wprefix, counts);
  if (e != cudaSuccess) return e;
  const long long slots = static_cast<long long>(T) * k_max;
  const unsigned blocks = static_cast<unsigned>(slots > 0 ? (slots + 255) / 256 : 1);
  e = launch_pdl(scatter_kernel, dim3(blocks), dim3(256), 0, s, topk_idx, k_per_token, T, k_max,
                 E_r, W, static_cast<const uint32_t*>(bitmap),
                 static_cast<const int32_t*>(wprefix), static_cast<const int32_t*>(counts),
                 offsets, sorted_token, inv_row, zero_ptr, zero_n);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, const int32_t* sorted_token,
                               const int32_t* offsets, int E_r, int T, int H, int n_cap,
                               void* x_perm, int32_t* status, int sm_count, cudaStream_t s,
                               int32_t* zero_ptr, int zero_n) {
  if (n_cap <= 0) return cudaSuccess;
  const int warps_needed = n_cap;
  int blocks = (warps_needed + 7) / 8;
  blocks = blocks < sm_count * 8 ? blocks : sm_count * 8;
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s,
                    static_cast<const uint4*>(x), sorted_token, offsets, E_r, T, H / 8, n_cap,
                    static_cast<uint4*>(x_perm), status, zero_ptr, zero_n);
}

}  // namespace moe
