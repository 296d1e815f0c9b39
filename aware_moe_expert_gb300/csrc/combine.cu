// Weighted combine: out_t = sum_{j < k_t} w_{t,j} * y_perm[inv_row(t,j)]
// (+ the shared expert's y_shared[t]), fp32 accumulation in j order, one
// rounding to bf16.  MoE-Prism (arXiv 2510.19366) §III-B2: the routed output
// of a token is the gate-weighted sum of its selected units' FFN outputs.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 y) {
  const uint32_t yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(w, bf16lo(yv[i]), acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, bf16hi(yv[i]), acc[2 * i + 1]);
  }
}

// One thread per (token, 16-byte column vector), 128 threads per CTA.  The
// k_t rows a thread reads are independent, so they are loaded four at a time
// before they are accumulated (in j order); the grid spans T * H/8 threads so
// enough loads are in flight even for a handful of tokens.  y_perm is read
// once and out written once: both use the streaming (evict-first) cache
// policy, which leaves L2 to the rows still being read (Qwen3-30B-A3B-shaped
// prefill: 41 -> 33 us).
__global__ void __launch_bounds__(128) combine_kernel(
    const uint4* __restrict__ y_perm, const uint4* __restrict__ y_shared,
    const int32_t* __restrict__ inv_row, const float* __restrict__ topk_w,
    const int32_t* __restrict__ kpt, int T, int nv, int k_max, int n_rows,
    uint4* __restrict__ out, int32_t* status) {
  pdl_wait_and_trigger();
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int t = static_cast<int>(gid / nv);
  const int v = static_cast<int>(gid - static_cast<long long>(t) * nv);
  if (t >= T) return;
  const int32_t* ir = inv_row + static_cast<size_t>(t) * k_max;
  const float* tw = topk_w + static_cast<size_t>(t) * k_max;
  // the first four slots' indices are loaded with k_t (slots past k_t are
  // read but not used), so the row loads wait for one round trip, not two
  int r[4];
  float w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    r[q] = q < k_max ? __ldg(ir + q) : -1;
    w[q] = q < k_max ? __ldg(tw + q) : 0.f;
  }
  const int k = min(max(kpt[t], 0), k_max);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool bad = false;
  for (int j0 = 0; j0 < k; j0 += 4) {
    uint4 y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q;
      if (j0 > 0) {
        r[q] = j < k ? __ldg(ir + j) : -1;
        w[q] = j < k ? __ldg(tw + j) : 0.f;
      } else if (j >= k) {
        r[q] = -1;
      }
      if (j < k && (r[q] < 0 || r[q] >= n_rows)) {
        bad = true;
        r[q] = -1;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      y[q] = r[q] >= 0 ? __ldcs(y_perm + static_cast<size_t>(r[q]) * nv + v)
                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (r[q] >= 0) fma8(acc, w[q], y[q]);
  }
  if (bad && v == 0) report(status, MOE_ERR_BAD_INDEX);
  if (y_shared != nullptr) {
    const uint4 s = __ldg(y_shared + static_cast<size_t>(t) * nv + v);
    const uint32_t sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16lo(sv[i]);
      acc[2 * i + 1] += bf16hi(sv[i]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  __stcs(out + static_cast<size_t>(t) * nv + v, o);
}

// Small batches (the whole grid resident at once: latency, not bandwidth,
// sets the time): a thread loads KB indices and gates of its token with k_t
// in one round trip, then those rows of y_perm in the next (KB >= k_max:
// two round trips in all), instead of four at a time.  Same sum, same order, same rounding as
// combine_kernel.
template <int KB>
__global__ void __launch_bounds__(128) combine_wide_kernel(
    const uint4* __restrict__ y_perm, const uint4* __restrict__ y_shared,
    const int32_t* __restrict__ inv_row, const float* __restrict__ topk_w,
    const int32_t* __restrict__ kpt, int T, int nv, int k_max, int n_rows,
    uint4* __restrict__ out, int32_t* status) {
  pdl_wait_and_trigger();
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int t = static_cast<int>(gid / nv);
  const int v = static_cast<int>(gid - static_cast<long long>(t) * nv);
  if (t >= T) return;
  const int32_t* ir = inv_row + static_cast<size_t>(t) * k_max;
  const float* tw = topk_w + static_cast<size_t>(t) * k_max;
  // the first KB indices and gates are loaded with k_t (slots past k_t are
  // read but not used)
  int r[KB];
  float w[KB];
#pragma unroll
  for (int q = 0; q < KB; ++q) {
    r[q] = q < k_max ? __ldg(ir + q) : -1;
    w[q] = q < k_max ? __ldg(tw + q) : 0.f;
  }
  const int k = min(max(kpt[t], 0), k_max);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool bad = false;
  for (int j0 = 0; j0 < k; j0 += KB) {
    if (j0 > 0) {
#pragma unroll
      for (int q = 0; q < KB; ++q) {
        r[q] = j0 + q < k_max ? __ldg(ir + j0 + q) : -1;
        w[q] = j0 + q < k_max ? __ldg(tw + j0 + q) : 0.f;
      }
    }
    uint4 y[KB];
#pragma unroll
    for (int q = 0; q < KB; ++q) {
      const int j = j0 + q;
      if (j >= k) {
        r[q] = -1;
      } else if (r[q] < 0 || r[q] >= n_rows) {
        bad = true;
        r[q] = -1;
      }
      y[q] = r[q] >= 0 ? __ldcs(y_perm + static_cast<size_t>(r[q]) * nv + v)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < KB; ++q)
      if (r[q] >= 0) fma8(acc, w[q], y[q]);
  }
  if (bad && v == 0) report(status, MOE_ERR_BAD_INDEX);
  if (y_shared != nullptr) {
    const uint4 sh = __ldg(y_shared + static_cast<size_t>(t) * nv + v);
    const uint32_t sv[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16lo(sv[i]);
      acc[2 * i + 1] += bf16hi(sv[i]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  __stcs(out + static_cast<size_t>(t) * nv + v, o);
}

// Threads of `kern` (128 per CTA) the device holds at once.
template <typename K>
long long resident_threads(K kern, long long (&cache)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int sms = 0, blocks = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, 128, 0) == cudaSuccess)
      cache[dev] = static_cast<long long>(sms) * blocks * 128;
    (void)cudaGetLastError();
  }
  return cache[dev];
}

}  // namespace

cudaError_t launch_combine(const void* y_perm, const void* y_shared, const int32_t* inv_row,
                           const float* topk_w, const int32_t* k_per_token, int T, int H,
                           int k_max, int n_rows, void* out, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const long long threads = static_cast<long long>(T) * (H / 8);
  // From 32 tokens up to one wave of the wide kernel (latency-bound: all of a
  // thread's loads at once).  Same-box A/B of the decode layer: T = 64
  // -1.65 us, T = 256 -0.55, Mixtral-shaped T = 64 -0.25, but T = 8 +0.67 and
  // T = 1 unchanged, so smaller batches keep combine_kernel.
  static long long res8[64] = {0}, res16[64] = {0};
  const unsigned grid = static_cast<unsigned>((threads + 127) / 128);
  const bool wide = T >= 32;
  if (wide && k_max <= 8 && threads <= resident_threads(combine_wide_kernel<8>, res8))
    return launch_pdl(combine_wide_kernel<8>, dim3(grid), dim3(128), 0, s,
                      static_cast<const uint4*>(y_perm), static_cast<const uint4*>(y_shared),
                      inv_row, topk_w, k_per_token, T, H / 8, k_max, n_rows,
                      static_cast<uint4*>(out), status);
  if (wide && k_max <= 16 && threads <= resident_threads(combine_wide_kernel<16>, res16))
    return launch_pdl(combine_wide_kernel<16>, dim3(grid), dim3(128), 0, s,
                      static_cast<const uint4*>(y_perm), static_cast<const uint4*>(y_shared),
                      inv_row, topk_w, k_per_token, T, H / 8, k_max, n_rows,
                      static_cast<uint4*>(out), status);
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>((threads + 127) / 128)), dim3(128),
                    0, s, static_cast<const uint4*>(y_perm), static_cast<const uint4*>(y_shared),
                    inv_row, topk_w, k_per_token, T, H / 8, k_max, n_rows,
                    static_cast<uint4*>(out), status);
}

}  // namespace moe
