// Training-free proxy router (CG): the original router keeps m experts per
// token; gate-neuron activations of each kept expert's sub-experts give proxy
// scores; the kappa_j best sub-experts of expert j are routed with the
// expert's weight.  MoE-Prism (arXiv 2510.19366) §III-B2, "Training-Free
// Proxy Gating" (Fig. 7, left).
//
// GPU layout: the gate neurons of all units are packed once (model set-up)
// into proxy_w = bf16 [E_r * r * 2, H]: row (u * r + i) * 2 is the gate row of
// unit u's i-th gate neuron, the next row its up row.  At routing time the
// pre-activations P = x . proxy_w^T (fp32 [T, E_r * 2r], possibly as slice
// partials) come from the router kernels; cg_select_kernel then forms
//   s_n = (1/r) sum_i |SiLU(g_i) * u_i|
// for the n_sub sub-experts of each kept expert and picks the kappa_j best.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float silu32(float g) { return g / (1.0f + expf(-g)); }

// Same total order as the unit selection: larger first, -0 == +0, NaN last.
__device__ __forceinline__ uint32_t cg_key(float v) {
  if (v != v) return 0u;
  uint32_t b = __float_as_uint(v);
  if ((b & 0x7fffffffu) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One warp per packed row; 16-byte copies.
__global__ void __launch_bounds__(256) pack_proxy_kernel(
    const uint4* __restrict__ w_gate_up, const int32_t* __restrict__ G, int E_r, int r,
    int I_sub, int nv, uint4* __restrict__ proxy_w, int32_t* status) {
  pdl_wait_and_trigger();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= E_r * r * 2) return;
  const int u = row / (2 * r), i = (row >> 1) % r, up = row & 1;
  const int c = G[u * r + i];
  uint4* dst = proxy_w + static_cast<size_t>(row) * nv;
  if (c < 0 || c >= I_sub) {
    if (lane == 0) report(status, MOE_ERR_BAD_INDEX);
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* src =
      w_gate_up + (static_cast<size_t>(u) * 2 * I_sub + static_cast<size_t>(up) * I_sub + c) * nv;
  for (int v = lane; v < nv; v += 32) dst[v] = __ldg(src + v);
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(bf16lo(av[i]), bf16lo(bv[i]), acc);
    acc = fmaf(bf16hi(av[i]), bf16hi(bv[i]), acc);
  }
  return acc;
}

// Gate-neuron pre-activations of the kept experts only (decode-sized T):
//   out[t, j, row] = x_t . proxy_w[e_j * rows_e + row],  row < rows_e = N * 2r
// CTA = up to tpc (<= 8) tokens x one expert e x kRowsPerCta of its rows; it
// returns at once if none of its tokens kept e.  The kept tokens' x rows are
// staged in shared memory (eight loads per thread in flight); each warp takes
// two rows, one at a time, with up to kVecBatch 16-byte loads per lane of the
// row in flight together.
constexpr int kTpcMax = 8;
constexpr int kRowsPerCta = 16;
constexpr int kVecBatch = 8;

__global__ void __launch_bounds__(256) proxy_gemv_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ proxy_w,
    const int32_t* __restrict__ expert_idx, int T, int nv, int m, int rows_e, int tpc,
    float* __restrict__ out) {
  extern __shared__ uint4 xs[];  // [tpc][nv]
  __shared__ int jpos[kTpcMax];
  __shared__ int kept[kTpcMax];   // token slots (in the block) that kept e, compacted
  __shared__ int any_kept;
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y;
  const int t0 = blockIdx.x * tpc;
  const int nt = min(tpc, T - t0);
  if (threadIdx.x == 0) any_kept = 0;
  __syncthreads();
  if (threadIdx.x < nt) {
    int jp = -1;
    for (int j = 0; j < m; ++j)
      if (expert_idx[static_cast<size_t>(t0 + threadIdx.x) * m + j] == e) jp = j;
    jpos[threadIdx.x] = jp;
    if (jp >= 0) atomicOr(&any_kept, 1);
  } else if (threadIdx.x < kTpcMax) {
    jpos[threadIdx.x] = -1;
  }
  __syncthreads();
  if (!any_kept) return;
  int nk = 0;
  for (int i = 0; i < nt; ++i)
    if (jpos[i] >= 0) {
      if (threadIdx.x == 0) kept[nk] = i;
      ++nk;
    }
  // stage the kept tokens' rows, eight 16-byte loads per thread in flight
  const int total = nt * nv;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * 256) {
    uint4 tmp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = i0 + q * 256;
      const int tt = i / nv;
      tmp[q] = (i < total && jpos[tt] >= 0)
                   ? __ldg(x + static_cast<size_t>(t0 + tt) * nv + (i - tt * nv))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = i0 + q * 256;
      if (i < total) xs[i] = tmp[q];
    }
  }
  __syncthreads();
  const int row_end = min(rows_e, static_cast<int>(blockIdx.z + 1) * kRowsPerCta);
  for (int row = blockIdx.z * kRowsPerCta + warp; row < row_end; row += 8) {
    const uint4* w = proxy_w + (static_cast<size_t>(e) * rows_e + row) * nv;
    float acc[kTpcMax];
#pragma unroll
    for (int i = 0; i < kTpcMax; ++i) acc[i] = 0.f;
    for (int v0 = lane; v0 < nv; v0 += 32 * kVecBatch) {
      uint4 wv[kVecBatch];
#pragma unroll
      for (int q = 0; q < kVecBatch; ++q)
        wv[q] = v0 + 32 * q < nv ? __ldg(w + v0 + 32 * q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < kVecBatch; ++q) {
        if (v0 + 32 * q >= nv) continue;
        float wf[8];                                   // the weight vector, unpacked once
        const uint32_t wr[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          wf[2 * h] = bf16lo(wr[h]);
          wf[2 * h + 1] = bf16hi(wr[h]);
        }
#pragma unroll
        for (int i = 0; i < kTpcMax; ++i) {
          if (i >= nk) continue;
          const uint4 xv = xs[kept[i] * nv + v0 + 32 * q];
          const uint32_t xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            acc[i] = fmaf(bf16lo(xr[h]), wf[2 * h], acc[i]);
            acc[i] = fmaf(bf16hi(xr[h]), wf[2 * h + 1], acc[i]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kTpcMax; ++i) {
      if (i >= nk) continue;
      float a = acc[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      if (lane == 0) {
        const int ti = kept[i];
        out[(static_cast<size_t>(t0 + ti) * m + jpos[ti]) * rows_e + row] = a;
      }
    }
  }
}

// One warp per token.  The m * N * r (expert, sub-expert, gate neuron) pairs
// of the token are shared by the 32 lanes: a lane adds the S slice partials
// of its pairs' gate and up pre-activations (all loads of a pair issued
// together) and stores |SiLU(g) * u| in shared memory; then lane n < N sums
// sub-expert n's r values in neuron order.  P holds S partial arrays [T, R]
// (R = E_r * 2r), or, with `compact`, one array [T, m, N * 2r] of the kept
// experts only; P == nullptr (n_sub == 1, no proxy_out) skips the scores: the
// single sub-expert of a kept expert needs none.
constexpr int kSliceBatch = 8;

__global__ void __launch_bounds__(256) cg_select_kernel(
    const float* __restrict__ P, int S, int R, const int32_t* __restrict__ expert_idx,
    const float* __restrict__ expert_w, const int32_t* __restrict__ kappa,
    const int32_t* __restrict__ kpt, int T, int m, int N, int r, int k_max, int n_experts,
    int compact, float* __restrict__ proxy_out, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* status) {
  extern __shared__ float act_s[];  // [8 warps][m * N * r]
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float* act = act_s + warp * (m * N * r);
  int k = kpt[t];
  bool ok = true;
  if (k < 1 || k > k_max) {
    ok = false;
    k = min(max(k, 0), k_max);
  }
  // validate the allocation row kappa[k]
  int ksum = 0;
  for (int j = 0; j < m; ++j) {
    const int kj = kappa[k * m + j];
    ok &= kj >= 0 && kj <= N;
    ksum += kj;
  }
  ok &= ksum == k;
  if (!ok && lane == 0) report(status, MOE_ERR_K_RANGE);
  // the kept experts (lane j holds expert j)
  const int my_e = lane < m ? expert_idx[static_cast<size_t>(t) * m + lane] : 0;
  const float my_w = lane < m ? expert_w[static_cast<size_t>(t) * m + lane] : 0.f;
  if (__any_sync(0xffffffffu, lane < m && (my_e < 0 || my_e >= n_experts))) {
    if (lane == 0) report(status, MOE_ERR_BAD_INDEX);
    ok = false;
  }
  if (ok && P != nullptr) {
    const int pairs = m * N * r, per_e = N * r;
#pragma unroll 4
    for (int p0 = 0; p0 < pairs; p0 += 32) {       // warp-uniform trip count
      const int p = p0 + lane;
      const int j = min(p, pairs - 1) / per_e;
      const int e = __shfl_sync(0xffffffffu, my_e, j);
      if (p < pairs) {
        const size_t off =
            compact ? (static_cast<size_t>(t) * m + j) * 2 * per_e + 2 * (p - j * per_e)
                    : static_cast<size_t>(t) * R + static_cast<size_t>(e) * 2 * per_e +
                          2 * (p - j * per_e);
        float g = 0.f, u = 0.f;
        for (int q0 = 0; q0 < S; q0 += kSliceBatch) {   // kSliceBatch loads in flight
          float2 v[kSliceBatch];
#pragma unroll
          for (int q = 0; q < kSliceBatch; ++q)
            if (q0 + q < S)
              v[q] = *reinterpret_cast<const float2*>(P + static_cast<size_t>(q0 + q) * T * R +
                                                      off);
#pragma unroll
          for (int q = 0; q < kSliceBatch; ++q)
            if (q0 + q < S) {
              g = (q0 + q == 0) ? v[q].x : g + v[q].x;
              u = (q0 + q == 0) ? v[q].y : u + v[q].y;
            }
        }
        act[p] = fabsf(silu32(g) * u);
      }
    }
    __syncwarp();
  }
  int slot = 0;
  const float inv_r = 1.0f / static_cast<float>(r);
  for (int j = 0; ok && j < m; ++j) {
    const int e = __shfl_sync(0xffffffffu, my_e, j);
    const float wj = __shfl_sync(0xffffffffu, my_w, j);
    float s = 0.f;
    if (P != nullptr && lane < N) {
      const float* a = act + (j * N + lane) * r;
      float acc = 0.f;
      for (int i = 0; i < r; ++i) acc += a[i];
      s = acc * inv_r;
      if (proxy_out != nullptr) proxy_out[(static_cast<size_t>(t) * m + j) * N + lane] = s;
    }
    // rank of lane's sub-expert among the N: key descending, lower index first
    const uint32_t key = lane < N ? cg_key(s) : 0u;
    int rank = 0;
    for (int o = 0; o < N; ++o) {
      const uint32_t ko = __shfl_sync(0xffffffffu, key, o);
      rank += (ko > key || (ko == key && o < lane)) ? 1 : 0;
    }
    const int kj = kappa[k * m + j];
    if (lane < N && rank < kj) {
      const size_t o = static_cast<size_t>(t) * k_max + slot + rank;
      topk_idx[o] = e * N + lane;
      topk_w[o] = wj;
    }
    slot += kj;
  }
  if (!ok) slot = 0;
  for (int sl = slot + lane; sl < k_max; sl += 32) {
    topk_idx[static_cast<size_t>(t) * k_max + sl] = -1;
    topk_w[static_cast<size_t>(t) * k_max + sl] = 0.f;
  }
}

}  // namespace

cudaError_t launch_pack_proxy(const void* w_gate_up, const int32_t* gate_neurons, int E_r, int r,
                              int I_sub, int H, void* proxy_w, int32_t* status, cudaStream_t s) {
  const int rows = E_r * r * 2;
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(pack_proxy_kernel, dim3((rows + 7) / 8), dim3(256), 0, s,
                    static_cast<const uint4*>(w_gate_up), gate_neurons, E_r, r, I_sub, H / 8,
                    static_cast<uint4*>(proxy_w), status);
}

cudaError_t launch_proxy_gemv(const void* x, const void* proxy_w, const int32_t* expert_idx,
                              int T, int H, int n_experts, int m, int rows_e, float* out,
                              cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int row_bytes = H * 2;
  int tpc = (96 * 1024) / row_bytes;
  tpc = tpc < 1 ? 1 : (tpc > kTpcMax ? kTpcMax : tpc);
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(proxy_gemv_kernel, 96 * 1024, attr_done);
  if (e != cudaSuccess) return e;
  const dim3 grid((T + tpc - 1) / tpc, n_experts, (rows_e + kRowsPerCta - 1) / kRowsPerCta);
  return launch_pdl(proxy_gemv_kernel, grid, dim3(256),
                    static_cast<size_t>(tpc) * row_bytes, s, static_cast<const uint4*>(x),
                    static_cast<const uint4*>(proxy_w), expert_idx, T, H / 8, m, rows_e, tpc,
                    out);
}

cudaError_t launch_cg_select(const float* partial, int S, int R, bool compact,
                             const int32_t* expert_idx, const float* expert_w,
                             const int32_t* kappa, const int32_t* kpt, int T, int m, int N,
                             int r, int k_max, int n_experts, float* proxy_out, int32_t* topk_idx,
                             float* topk_w, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (m * N * r > kMaxProxyPairs) return cudaErrorInvalidValue;
  const int smem = 8 * m * N * r * static_cast<int>(sizeof(float));
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(cg_select_kernel, 8 * kMaxProxyPairs * 4, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(cg_select_kernel, dim3((T + 7) / 8), dim3(256), smem, s, partial, S, R,
                    expert_idx, expert_w, kappa, kpt, T, m, N, r, k_max, n_experts,
                    compact ? 1 : 0, proxy_out,
                    topk_idx, topk_w, status);
}

}  // namespace moe
