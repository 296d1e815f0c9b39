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

// Descending compare-exchange of two packed (key << 32 | ~unit) entries.
__device__ __forceinline__ void cas_desc(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Sorts a lane's IPL entries in descending order (Batcher's odd-even merge
// networks for 2, 4 and 8 entries: 1, 5 and 19 compare-exchanges).
template <int IPL>
__device__ __forceinline__ void lane_sort_desc(unsigned long long (&e)[IPL]) {
  if constexpr (IPL == 2) {
    cas_desc(e[0], e[1]);
  } else if constexpr (IPL == 4) {
    cas_desc(e[0], e[1]); cas_desc(e[2], e[3]);
    cas_desc(e[0], e[2]); cas_desc(e[1], e[3]);
    cas_desc(e[1], e[2]);
  } else if constexpr (IPL == 8) {
    cas_desc(e[0], e[1]); cas_desc(e[2], e[3]); cas_desc(e[4], e[5]); cas_desc(e[6], e[7]);
    cas_desc(e[0], e[2]); cas_desc(e[1], e[3]); cas_desc(e[4], e[6]); cas_desc(e[5], e[7]);
    cas_desc(e[1], e[2]); cas_desc(e[5], e[6]);
    cas_desc(e[0], e[4]); cas_desc(e[1], e[5]); cas_desc(e[2], e[6]); cas_desc(e[3], e[7]);
    cas_desc(e[2], e[4]); cas_desc(e[3], e[5]);
    cas_desc(e[1], e[2]); cas_desc(e[3], e[4]); cas_desc(e[5], e[6]);
  } else {
    static_assert(IPL == 1, "IPL is 1, 2, 4 or 8");
  }
}

// The k best of the 32 * IPL units a warp holds (lane l holds units l,
// l + 32, ...; key[i] = order_key of unit lane + 32 i, units >= E_r absent),
// best first, ties to the lower index.  Lane j < k returns
// (key << 32) | ~u of the j-th unit; other lanes return 0.
//
// Every unit is packed as (key << 32) | ~u, so the packed order is the
// selection order (larger key first, then lower index); absent units pack
// as 0, below every unit.  Each lane sorts its entries; then k rounds take
// the warp's largest head (two 32-bit warp max reductions: key, then ~u among
// the heads with that key) and the lane that held it drops its head.
template <int IPL>
__device__ __forceinline__ unsigned long long warp_select_topk(const uint32_t (&key)[IPL],
                                                               int E_r, int k, int lane) {
  unsigned long long e[IPL];
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    e[i] = u < E_r ? (static_cast<unsigned long long>(key[i]) << 32) |
                         static_cast<uint32_t>(~static_cast<uint32_t>(u))
                   : 0ull;
  }
  lane_sort_desc<IPL>(e);
  unsigned long long best = 0ull;
  for (int j = 0; j < k; ++j) {
    const uint32_t hk = static_cast<uint32_t>(e[0] >> 32);
    const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t lo = hk == mk ? static_cast<uint32_t>(e[0]) : 0u;
    const uint32_t ml = __reduce_max_sync(0xffffffffu, lo);
    const unsigned long long win = (static_cast<unsigned long long>(mk) << 32) | ml;
    if (lane == j) best = win;
    const bool pop = e[0] == win;
#pragma unroll
    for (int i = 0; i + 1 < IPL; ++i) e[i] = pop ? e[i + 1] : e[i];
    if (pop) e[IPL - 1] = 0ull;
  }
  return best;
}

// One warp selects the k_t best units of one token.  Lane l holds units l,
// l+32, ... (IPL per lane); the token's logit of unit u is the sum of the S
// partial rows P[s] (s in order; S = 1 for finished logits) plus
// bias[u / n_sub] when bias is given, and is stored to lout[u] when lout is
// given.  Lane j < k ends up holding the j-th unit (*out_u) and its gate
// weight after renormalisation and route_scale (*out_w).  Returns k.
// Softmax statistics of one token's logits held IPL per lane: the maximum and
// sum of exp(v - max) over the E_r units, reduced across the warp in a fixed
// order (bit-identical wherever it runs).
template <int IPL>
__device__ __forceinline__ void softmax_stats(const float (&v)[IPL], int E_r, int lane, float* mx_out,
                                              float* sum_out) {
  float mx = -INFINITY, sum = 0.f;
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
  *mx_out = mx;
  *sum_out = sum;
}

// One token's logits in a lane's IPL registers: the first partial row plus
// the rest in slice order (SB slices' loads in flight), plus bias[u / n_sub].
template <int IPL, int SB>
__device__ __forceinline__ void load_logits(const float* __restrict__ P, int S, size_t sstride,
                                            const float* __restrict__ bias, int n_sub, int E_r,
                                            int lane, float (&v)[IPL]) {
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    v[i] = u < E_r ? P[u] : 0.f;
  }
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
    if (u < E_r && bias != nullptr) v[i] += bias[u / n_sub];
  }
}

// stats (nullable): softmax maximum and sum computed by a helper warp, read
// after named barrier stats_bar (64 threads: this warp and the helper).
template <int IPL, int SB = 2>
__device__ __forceinline__ int warp_topk(const float* __restrict__ P, int S, size_t sstride,
                                         const float* __restrict__ bias, int n_sub,
                                         float* __restrict__ lout, int kt, int E_r, int k_max,
                                         int score, int renorm, float route_scale,
                                         int32_t* status, int lane, int* out_u, float* out_w,
                                         const volatile float* stats = nullptr,
                                         int stats_bar = 0) {
  int k = kt;
  if (k < 1 || k > k_max) {
    if (lane == 0) report(status, MOE_ERR_K_RANGE);
    k = min(max(k, 0), k_max);
  }
  k = min(k, E_r);
  float v[IPL];
  uint32_t key[IPL];
  bool bad = false;
  load_logits<IPL, SB>(P, S, sstride, bias, n_sub, E_r, lane, v);
#pragma unroll
  for (int i = 0; i < IPL; ++i) {
    const int u = lane + 32 * i;
    if (u < E_r) {
      if (lout != nullptr) lout[u] = v[i];
      bad |= !isfinite(v[i]);
      key[i] = order_key(v[i]);
    } else {
      key[i] = 0u;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(status, MOE_ERR_NONFINITE);

  float mx = -INFINITY, sum = 0.f;
  if (score == MOE_SCORE_SOFTMAX && stats == nullptr) softmax_stats<IPL>(v, E_r, lane, &mx, &sum);

  const unsigned long long best = warp_select_topk<IPL>(key, E_r, k, lane);
  if (score == MOE_SCORE_SOFTMAX && stats != nullptr) {
    asm volatile("bar.sync %0, 64;" ::"r"(stats_bar) : "memory");
    mx = stats[0];
    sum = stats[1];
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
//
// HELP (softmax scores): warps 8-15 compute the softmax maximum and exp-sum
// of token (warp - 8) with the code warp_topk would run (same bits) while
// warp (warp - 8) selects; they meet at named barrier 1 + (warp - 8).
//
// bitmap != nullptr: the CTA also writes its byte of the permutation's unit
// membership bitmap (bit j of byte b of row u = token 8 b + j selected u;
// rows of row_bytes = 4 * ceil(T / 32) bytes, the uint32 words the scan
// reads), so the permutation needs no pass of its own over topk_idx.  The
// last CTA also zeroes the row bytes past the last token group.
template <int IPL, int SB, bool HELP = false>
__global__ void __launch_bounds__(HELP ? 512 : 256) topk_gate_kernel(
    const float* __restrict__ P, int S, const float* __restrict__ bias, int n_sub,
    float* __restrict__ logits_out, const int32_t* __restrict__ kpt, int T, int E_r,
    int k_max, int score, int renorm, float route_scale, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* status, uint8_t* __restrict__ bitmap,
    int row_bytes) {
  __shared__ uint32_t s_bits[256];
  __shared__ float s_stat_raw[16];
  volatile float* s_stat = s_stat_raw;
  pdl_wait_and_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tw = warp & 7;
  const int t = blockIdx.x * 8 + tw;
  const bool helped = HELP && score == MOE_SCORE_SOFTMAX;
  if (bitmap != nullptr) {
    for (int v = threadIdx.x; v < E_r; v += blockDim.x) s_bits[v] = 0u;
    __syncthreads();
  }
  if (HELP && warp >= 8) {
    if (helped && t < T) {
      float v[IPL], mx, sum;
      load_logits<IPL, SB>(P + static_cast<size_t>(t) * E_r, S, static_cast<size_t>(T) * E_r,
                           bias, n_sub, E_r, lane, v);
      softmax_stats<IPL>(v, E_r, lane, &mx, &sum);
      if (lane == 0) {
        s_stat[2 * tw] = mx;
        s_stat[2 * tw + 1] = sum;
      }
      asm volatile("bar.sync %0, 64;" ::"r"(1 + tw) : "memory");
    }
  } else if (t < T) {
    int u;
    float w;
    const size_t row = static_cast<size_t>(t) * E_r;
    warp_topk<IPL, SB>(P + row, S, static_cast<size_t>(T) * E_r, bias, n_sub,
                       logits_out != nullptr ? logits_out + row : nullptr,
                       kpt != nullptr ? kpt[t] : k_max, E_r, k_max, score,
                       renorm, route_scale, status, lane, &u, &w,
                       helped ? s_stat + 2 * tw : nullptr, 1 + tw);
    if (lane < k_max) {
      const size_t o = static_cast<size_t>(t) * k_max + lane;
      topk_idx[o] = u;
      topk_w[o] = w;
    }
    if (bitmap != nullptr && u >= 0) atomicOr(&s_bits[u], 1u << tw);
  }
  if (bitmap != nullptr) {
    __syncthreads();
    for (int v = threadIdx.x; v < E_r; v += blockDim.x) {
      uint8_t* r = bitmap + static_cast<size_t>(v) * row_bytes;
      r[blockIdx.x] = static_cast<uint8_t>(s_bits[v]);
      if (blockIdx.x + 1 == gridDim.x)
        for (int b = blockIdx.x + 1; b < row_bytes; ++b) r[b] = 0;
    }
  }
}

// ---------------------------------------------------------------- cluster router
// Logits and top-k_t of up to eight tokens in one launch.  A cluster of C
// CTAs (16, else 8) splits the units; each CTA stages its units' router rows
// and the eight tokens' x rows in shared memory, chunk by chunk of the hidden
// dimension (cp.async, two chunks in flight), and its 16 warps split every
// chunk's k-steps between them: per k-step one mma.sync m16n8k16 (16 units x
// 8 tokens, bf16 in, fp32 out).  The warps' partial tiles are added in warp
// order, and each CTA pushes its logits into CTA 0's shared memory.  After a
// cluster barrier CTA 0 runs the warp top-k per token.  With a single cluster
// holding every token (T <= 8) CTA 0 also builds the permutation in shared
// memory, writes it out and zeroes the next kernel's counters, while the
// other CTAs have already exited.
constexpr int kClTok = 8;
constexpr int kClThreads = 512;
constexpr int kClWarps = kClThreads / 32;
static_assert(kClWarps >= 2 * 8, "a selecting warp and a helper warp per token of a cluster block");
constexpr int kClMaxMt = 2;                      // 16-unit m-tiles per CTA (C >= 8, E_r <= 256)
constexpr uint32_t kClStageBudget = 208 * 1024;  // staged rows, all chunks in flight

struct ClusterRouteParams {
  const uint4* x;
  const uint4* rw;
  const float* bias;
  int n_sub;
  const int32_t* kpt;
  int T, nv, E_r, k_max, score, renorm;
  float route_scale;
  float* logits_out;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* status;
  int C;                 // CTAs per cluster
  int MT;                // 16-unit m-tiles per CTA: ceil(ceil(E_r / C) / 16)
  int kc;                // hidden columns per staged chunk (multiple of 16)
  int ns;                // chunk buffers (1: all of H at once, or 2)
  // fused permutation (nullptr: route only); zero_ptr: counters of the next
  // kernel that this launch zeroes
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_token;
  int32_t* inv_row;
  int32_t* zero_ptr;
  int zero_n;
};

struct ClusterSmem {
  uint32_t pitch, rows, stage, red, all, bits, off, wt, bias, stat, total;
};

// Staged rows per buffer: MT * 16 unit rows, then the eight token rows, each
// kc columns plus 16 bytes of padding (conflict-free ldmatrix).  The warps'
// partial tiles reuse the staging area once the last chunk is consumed.
__host__ __device__ inline ClusterSmem cluster_smem(int E_r, int MT, int kc, int ns) {
  ClusterSmem o;
  o.pitch = static_cast<uint32_t>(kc) * 2 + 16;
  o.rows = static_cast<uint32_t>(MT * 16 + kClTok);
  uint32_t b = 0;
  o.stage = b;
  o.red = b;                                     // [warp][m-tile][16 x 8] fp32
  const uint32_t st = static_cast<uint32_t>(ns) * o.rows * o.pitch;
  const uint32_t red = static_cast<uint32_t>(kClWarps * MT * 128 * 4);
  b += st > red ? st : red;
  b = (b + 15) & ~15u;
  o.all = b;
  b += kClTok * E_r * 4;
  o.bits = b;
  b += 256 * 4;
  o.off = b;
  b += 260 * 4;
  o.wt = b;
  b += kClWarps * 4;
  o.bias = b;
  b += 256 * 4;
  o.stat = b;
  b += kClTok * 2 * 4;
  o.total = b;
  return o;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int IPL>
__global__ void __launch_bounds__(kClThreads, 1) route_cluster_kernel(const ClusterRouteParams p) {
  extern __shared__ __align__(16) uint8_t csm[];
  const ClusterSmem L = cluster_smem(p.E_r, p.MT, p.kc, p.ns);
  float* s_red = reinterpret_cast<float*>(csm + L.red);
  float* s_all = reinterpret_cast<float*>(csm + L.all);
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(csm + L.bits);
  int32_t* s_off = reinterpret_cast<int32_t*>(csm + L.off);
  int32_t* s_wt = reinterpret_cast<int32_t*>(csm + L.wt);
  float* s_bias = reinterpret_cast<float*>(csm + L.bias);
  volatile float* s_stat = reinterpret_cast<volatile float*>(csm + L.stat);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool fused = p.counts != nullptr;
  const int t0 = blockIdx.y * kClTok;
  const int nt = min(kClTok, p.T - t0);
  const int nv = p.nv, E_r = p.E_r, MT = p.MT;
  const int U = (E_r + p.C - 1) / p.C;           // units per CTA (<= MT * 16)
  const int u0 = static_cast<int>(rank) * U;
  const int nu = max(0, min(U, E_r - u0));
  const int n_mt = (nu + 15) / 16;
  const uint32_t pitch = L.pitch;
  const uint32_t stage_bytes = L.rows * pitch;
  const uint32_t tok_row0 = static_cast<uint32_t>(MT * 16);
  if (fused && rank == 0)
    for (int u = tid; u < 256; u += kClThreads) s_bits[u] = 0u;
  // rows no chunk writes (units past nu, tokens past nt) are zero in every buffer
  {
    const int zrows_u = MT * 16 - nu, zrows_t = kClTok - nt;
    const int vpr = p.kc / 8;
    const int total = p.ns * (zrows_u + zrows_t) * vpr;
    for (int i = tid; i < total; i += kClThreads) {
      const int per = (zrows_u + zrows_t) * vpr;
      const int s = i / per, j = i - s * per;
      const int zr = j / vpr, v = j - zr * vpr;
      const int row = zr < zrows_u ? nu + zr : MT * 16 + nt + (zr - zrows_u);
      *reinterpret_cast<uint4*>(csm + L.stage + s * stage_bytes + row * pitch + v * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // chunk c -> buffer c % ns: unit rows [0, nu), token rows [MT * 16, + nt)
  const int vc = p.kc / 8;                       // 16-byte vectors per chunk row
  const int n_chunks = (nv + vc - 1) / vc;
  const uint32_t stage0 = smem_u32(csm + L.stage);
  auto issue_rows = [&](int c, int r0, int nr, const uint4* base_src, uint32_t srow0) {
    const uint32_t base = stage0 + static_cast<uint32_t>((c % p.ns) * stage_bytes);
    const int v0 = c * vc, nvc = min(vc, nv - v0);
    const int total = nr * nvc;
    for (int i = tid; i < total; i += kClThreads) {
      const int r = i / nvc, v = i - r * nvc;
      cp_async16(base + (srow0 + static_cast<uint32_t>(r)) * pitch + static_cast<uint32_t>(v * 16),
                 base_src + static_cast<size_t>(r0 + r) * nv + v0 + v);
    }
  };
  auto issue_w = [&](int c) { issue_rows(c, u0, nu, p.rw, 0u); };
  auto issue_x = [&](int c) { issue_rows(c, t0, nt, p.x, tok_row0); };
  const bool two = n_chunks > 1 && p.ns > 1;
  // The router rows and the expert bias are layer parameters, not outputs of
  // the kernel this launch may overlap, so their loads go out before the
  // dependency wait; the token rows (and k_t) are read after it.
  if (nu > 0) {
    issue_w(0);
    if (two) issue_w(1);
  }
  if (rank == 0)
    for (int u = tid; u < E_r; u += kClThreads)
      s_bias[u] = p.bias != nullptr ? __ldg(p.bias + u / p.n_sub) : 0.f;
  pdl_wait_and_trigger();
  const int kt_pre =
      (rank == 0 && warp < nt) ? (p.kpt != nullptr ? __ldg(p.kpt + t0 + warp) : p.k_max) : 0;
  if (nu > 0) {
    issue_x(0);
    cp_async_commit();                           // group 0: rows of chunk 0 (and chunk 1's units)
    if (two) {
      issue_x(1);
      cp_async_commit();
    }
  }
  auto issue = [&](int c) {
    issue_w(c);
    issue_x(c);
    cp_async_commit();
  };
  float acc[kClMaxMt][4];
#pragma unroll
  for (int m = 0; m < kClMaxMt; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;
  for (int c = 0; c < n_chunks && nu > 0; ++c) {
    if (c + 1 < n_chunks && p.ns > 1)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    const uint32_t base = stage0 + static_cast<uint32_t>((c % p.ns) * stage_bytes);
    const int ks = min(vc, nv - c * vc) / 2;     // 16-column k-steps in this chunk
    // A (units, row-major): matrix i = lane / 8 -> rows (i & 1) * 8 + lane % 8, k + (i >> 1) * 8
    const uint32_t a_off = ((lane & 7) + ((lane >> 3) & 1) * 8) * pitch + (lane >> 4) * 16;
    // B (tokens, k contiguous): matrix i = (lane / 8) & 1 -> token lane % 8, k + i * 8
    const uint32_t b_off = (tok_row0 + (lane & 7)) * pitch + ((lane >> 3) & 1) * 16;
    for (int k = warp; k < ks; k += kClWarps) {
      uint32_t b[2];
      ldsm_x2(base + b_off + static_cast<uint32_t>(k * 32), b);
#pragma unroll
      for (int m = 0; m < kClMaxMt; ++m) {
        if (m < n_mt) {
          uint32_t a[4];
          ldsm_x4(base + a_off + static_cast<uint32_t>(m * 16) * pitch + static_cast<uint32_t>(k * 32), a);
          mma_16816(acc[m], a, b);
        }
      }
    }
    __syncthreads();
    if (c + p.ns < n_chunks) issue(c + p.ns);
  }
  // partial tiles -> s_red[warp][m][row][col] (over the staging area); C
  // fragment: c0,c1 at row lane/4, cols 2(lane%4)+{0,1}; c2,c3 at row lane/4 + 8
#pragma unroll
  for (int m = 0; m < kClMaxMt; ++m) {
    if (m < MT) {
      float* t = s_red + (warp * MT + m) * 128;
      const int r = lane >> 2, cc = (lane & 3) * 2;
      t[r * 8 + cc] = acc[m][0];
      t[r * 8 + cc + 1] = acc[m][1];
      t[(r + 8) * 8 + cc] = acc[m][2];
      t[(r + 8) * 8 + cc + 1] = acc[m][3];
    }
  }
  __syncthreads();
  // warps in order -> CTA 0's s_all[token][unit]
  const uint32_t all0 = mapa_shared(smem_u32(s_all), 0u);
  for (int i = tid; i < nt * nu; i += kClThreads) {
    const int tt = i / nu, ul = i - tt * nu;
    const int m = ul >> 4, r = ul & 15;
    float v = 0.f;
    for (int w = 0; w < kClWarps; ++w) v += s_red[(w * MT + m) * 128 + r * 8 + tt];
    st_cluster_f32(all0 + static_cast<uint32_t>((tt * E_r + u0 + ul) * 4), v);
  }
  cluster_sync_all();

  if (rank == 0) {
    int my_u = -1, k = 0;
    // Softmax: warp kClTok + j computes token j's maximum and exp-sum (the
    // code warp_topk would run, so the same bits) while warp j selects, and
    // hands them over at named barrier 1 + j.
    const bool helped = p.score == MOE_SCORE_SOFTMAX;
    if (helped && warp >= kClTok && warp < kClTok + nt) {
      const int j = warp - kClTok;
      float v[IPL], mx, sum;
      load_logits<IPL, 2>(s_all + j * E_r, 1, 0, p.bias != nullptr ? s_bias : nullptr, 1, E_r,
                          lane, v);
      softmax_stats<IPL>(v, E_r, lane, &mx, &sum);
      if (lane == 0) {
        s_stat[2 * j] = mx;
        s_stat[2 * j + 1] = sum;
      }
      asm volatile("bar.sync %0, 64;" ::"r"(1 + j) : "memory");
    }
    if (warp < nt) {
      const int t = t0 + warp;
      const size_t row = static_cast<size_t>(t) * E_r;
      float w;
      k = warp_topk<IPL>(s_all + warp * E_r, 1, 0, p.bias != nullptr ? s_bias : nullptr, 1,
                         p.logits_out != nullptr ? p.logits_out + row : nullptr,
                         kt_pre, E_r, p.k_max, p.score,
                         p.renorm, p.route_scale, p.status, lane, &my_u, &w,
                         helped ? s_stat + 2 * warp : nullptr, 1 + warp);
      if (lane < p.k_max) {
        const size_t o = static_cast<size_t>(t) * p.k_max + lane;
        p.topk_idx[o] = my_u;
        p.topk_w[o] = w;
      }
      if (fused && lane < k) atomicOr(&s_bits[my_u], 1u << warp);
    }
    if (fused) {
      __syncthreads();
      // counts and exclusive offsets over the units (E_r <= 256 <= threads)
      const int c = tid < E_r ? __popc(s_bits[tid]) : 0;
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) s_wt[warp] = incl;
      __syncthreads();
      int before = 0;
      for (int w2 = 0; w2 < warp; ++w2) before += s_wt[w2];
      if (tid < E_r) {
        const int ex = before + incl - c;
        s_off[tid] = ex;
        p.offsets[tid] = ex;
        p.counts[tid] = c;
        if (tid == E_r - 1) {
          s_off[E_r] = ex + c;
          p.offsets[E_r] = ex + c;
        }
      }
      __syncthreads();
      if (warp < nt && lane < p.k_max) {
        const int t = t0 + warp;
        int pos = -1;
        if (lane < k) {
          pos = s_off[my_u] + __popc(s_bits[my_u] & ((1u << warp) - 1u));
          p.sorted_token[pos] = t;
        }
        p.inv_row[static_cast<size_t>(t) * p.k_max + lane] = pos;
      }
    }
  }
  // CTA 0 alone finishes: no other CTA reads its shared memory after the
  // barrier above, so the others may already have exited
  if (fused && rank == 0)
    for (int i = tid; i < p.zero_n; i += kClThreads) p.zero_ptr[i] = 0;
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

bool route_cluster_supports(int H, int E_r) { return H % 16 == 0 && E_r <= 256; }

namespace {

// Most 16-CTA clusters of the router that can be resident at once (0: the
// device does not allow 16-CTA clusters; 8-CTA clusters are used instead).
template <int IPL>
cudaError_t route_clusters16(int* out) {
  static int cached[64];
  static bool known[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!known[dev]) {
    auto kern = route_cluster_kernel<IPL>;
    const int smem_max = static_cast<int>(kClStageBudget + 16 * 1024);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return e;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kClThreads);
      cfg.dynamicSmemBytes = smem_max;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    cached[dev] = n;
    known[dev] = true;
  }
  *out = cached[dev];
  return cudaSuccess;
}

template <int IPL>
cudaError_t run_route_cluster(ClusterRouteParams p, cudaStream_t s) {
  int n16 = 0;
  cudaError_t e = route_clusters16<IPL>(&n16);
  if (e != cudaSuccess) return e;
  const int n_clusters = (p.T + kClTok - 1) / kClTok;
  // 16-CTA clusters while they all fit at once, else 8-CTA clusters
  const int C = (n16 > 0 && n_clusters <= n16) ? 16 : 8;
  const int U = (p.E_r + C - 1) / C;
  p.C = C;
  p.MT = (U + 15) / 16;
  const int rows = p.MT * 16 + kClTok;
  const int H = p.nv * 8;
  if (static_cast<uint32_t>(rows) * (2u * H + 16u) <= kClStageBudget) {
    p.kc = H;
    p.ns = 1;
  } else {
    int kc = 4096;
    while (kc > 128 && 2u * rows * (2u * kc + 16u) > kClStageBudget) kc >>= 1;
    p.kc = kc;
    p.ns = 2;
  }
  const int smem = static_cast<int>(cluster_smem(p.E_r, p.MT, p.kc, p.ns).total);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, n_clusters);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, route_cluster_kernel<IPL>, p);
}

}  // namespace

cudaError_t launch_route_cluster(const void* x, const void* router_w, const float* bias,
                                 int n_sub, const int32_t* k_per_token, int T, int H, int E_r,
                                 int k_max, int score, int renorm, float route_scale,
                                 float* logits_out, int32_t* topk_idx, float* topk_w,
                                 int32_t* status, const RoutePermuteOut* fuse, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (!route_cluster_supports(H, E_r)) return cudaErrorInvalidValue;
  if (fuse != nullptr && T > kClTok) return cudaErrorInvalidValue;
  ClusterRouteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.rw = static_cast<const uint4*>(router_w);
  p.bias = bias;
  p.n_sub = n_sub;
  p.kpt = k_per_token;
  p.T = T;
  p.nv = H / 8;
  p.E_r = E_r;
  p.k_max = k_max;
  p.score = score;
  p.renorm = renorm;
  p.route_scale = route_scale;
  p.logits_out = logits_out;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.status = status;
  if (fuse != nullptr) {
    p.counts = fuse->counts;
    p.offsets = fuse->offsets;
    p.sorted_token = fuse->sorted_token;
    p.inv_row = fuse->inv_row;
    p.zero_ptr = fuse->zero_ptr;
    p.zero_n = fuse->zero_ptr != nullptr ? fuse->zero_n : 0;
  }
  if (E_r <= 32) return run_route_cluster<1>(p, s);
  if (E_r <= 64) return run_route_cluster<2>(p, s);
  if (E_r <= 128) return run_route_cluster<4>(p, s);
  return run_route_cluster<8>(p, s);
}

namespace {
// Multiprocessors of the current device (0 when it cannot be read).
int topk_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached[dev] = n;
  }
  return cached[dev];
}
}  // namespace

cudaError_t launch_topk_gate(const float* partial, int S, const float* bias, int n_sub,
                             float* logits_out, const int32_t* k_per_token, int T, int E_r,
                             int k_max, int score, int renorm, float route_scale,
                             int32_t* topk_idx, float* topk_w, int32_t* status,
                             cudaStream_t s, uint32_t* bitmap) {
  if (T <= 0) return cudaSuccess;
  if (E_r > 256) return cudaErrorInvalidValue;
  const int grid = (T + 7) / 8;
  uint8_t* bm = reinterpret_cast<uint8_t*>(bitmap);
  const int row_bytes = 4 * ((T + 31) / 32);
  // many partial slices (split-K routers of small batches): every slice's
  // loads in one round trip; otherwise two at a time (fewer registers).  With
  // softmax scores and at most one CTA per SM, a second warp per token
  // computes the softmax statistics while the first selects.
  const bool help = S > 2 && score == MOE_SCORE_SOFTMAX && grid <= topk_sm_count();
#define MOE_TOPK_LAUNCH(IPL)                                                                 \
  launch_pdl(help ? topk_gate_kernel<IPL, 8, true>                                           \
                  : (S > 2 ? topk_gate_kernel<IPL, 8> : topk_gate_kernel<IPL, 2>),            \
             dim3(grid), dim3(help ? 512 : 256), 0, s, partial, S, bias, n_sub,               \
             logits_out, k_per_token, T, E_r, k_max, score, renorm, route_scale, topk_idx,    \
             topk_w, status, bm, row_bytes)
  if (E_r <= 32) return MOE_TOPK_LAUNCH(1);
  if (E_r <= 64) return MOE_TOPK_LAUNCH(2);
  if (E_r <= 128) return MOE_TOPK_LAUNCH(4);
  return MOE_TOPK_LAUNCH(8);
#undef MOE_TOPK_LAUNCH
}

}  // namespace moe
