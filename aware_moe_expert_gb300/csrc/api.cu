// C ABI of libmoe.so (declared in include/moe.h): argument validation,
// workspace carving and launch sequencing on the caller's stream.  No call
// here allocates, frees or synchronises, except moe_get_device_status.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

using moe::GemmArgs;

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte offsets of every workspace region for one desc.
struct Layout {
  size_t logits, router_partial, topk_idx, topk_w, counts, offsets, sorted_token, inv_row, bitmap,
      wprefix, xperm, act, yperm, act_sh, ysh, split_word, partial, chunk_done, ffn_part,
      fold_ws, fold_idx, fold_w, fold_k, p_srcs, p_nsrc, p_slot, p_counts, p_offsets, p_sorted,
      p_inv, p_tgts, p_ntgt, p_tslot, p_wtgt, p_act, total;
  int router_slices;   // slices of the CUDA-core router (0: the tensor-core router runs)
  int max_split;       // K splits the decode gate|up kernel may use (1: none)
  int max_split_down;  // K splits the decode down kernel may use
};

// Budget of the decode kernel's fp32 split-K partial buffer.
constexpr size_t kPartialBudget = size_t(256) << 20;
constexpr int kMaxSplit = 8;

// The tensor-core GEMM computes the router logits for T >= 128 tokens when
// E_r is one of its tile widths; otherwise CUDA cores do, in slices of H.
bool router_on_tensor_cores(const moe_layer_desc& d) {
  return d.T >= 128 && moe::gemm_supports_f32_router(d.n_experts * d.n_sub);
}

inline int E_r_of(const moe_layer_desc* d) { return d->n_experts * d->n_sub; }

// Decode-shaped batches (at most 64 rows per routing unit on average, from
// the T * k_max bound) run the swap-AB kernels; desc->path forces either.
bool use_decode_path(const moe_layer_desc* d, int n_out, bool gate_up) {
  if (!moe::decode_gemm_supports(n_out, gate_up)) return false;
  if (d->path == MOE_PATH_DECODE) return true;
  if (d->path == MOE_PATH_PREFILL) return false;
  return static_cast<long long>(d->T) * d->k_max <= 64ll * E_r_of(d);
}

bool use_decode_ffn(const moe_layer_desc* d) {
  return use_decode_path(d, d->I_sub, true) && use_decode_path(d, d->H, false) &&
         moe::decode_ffn_supports(d->H, d->I_sub);
}
inline bool decode_ffn_path(const moe_layer_desc& d) { return use_decode_ffn(&d); }

Layout layout_of(const moe_layer_desc& d) {
  const size_t T = static_cast<size_t>(d.T), E_r = static_cast<size_t>(d.n_experts) * d.n_sub;
  const size_t n_cap = T * d.k_max, W = (T + 31) / 32;
  Layout l;
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  l.logits = take(T * E_r * 4);
  l.router_slices = 0;
  if (!router_on_tensor_cores(d)) {
    int vs = 0;
    l.router_slices = moe::router_slices(d.T, d.H, static_cast<int>(E_r), &vs);
  } else {
    int bn = 0, S = 1;
    moe::router_gemm_shape(d.T, d.H, static_cast<int>(E_r), &bn, &S);
    l.router_slices = S > 1 ? S : 0;
  }
  l.router_partial = take(static_cast<size_t>(l.router_slices) * T * E_r * 4);
  l.topk_idx = take(n_cap * 4);
  l.topk_w = take(n_cap * 4);
  l.counts = take(E_r * 4);
  l.offsets = take((E_r + 1) * 4);
  l.sorted_token = take(n_cap * 4);
  l.inv_row = take(n_cap * 4);
  l.bitmap = take(E_r * W * 4);
  l.wprefix = take(E_r * W * 4);
  l.xperm = take(n_cap * d.H * 2);
  l.act = take(n_cap * d.I_sub * 2);
  l.yperm = take(n_cap * d.H * 2);
  l.act_sh = take(T * static_cast<size_t>(d.I_shared) * 2);
  l.ysh = take(T * static_cast<size_t>(d.H) * 2);
  l.split_word = take(16);
  // fused decode FFN: chunk counters, the work counter and the split
  // counters (zeroed together), and the split partial sums
  l.chunk_done = take((n_cap / 16 + E_r + 1 + 1 + moe::kFfnPartSlots / 2) * 4);
  l.ffn_part = take(decode_ffn_path(d) ? static_cast<size_t>(moe::kFfnPartSlots) * 64 * 128 * 4 : 0);
  auto splits = [](size_t per_split) {
    size_t ms = per_split > 0 ? kPartialBudget / per_split : 1;
    return static_cast<int>(ms < 1 ? 1 : (ms > kMaxSplit ? kMaxSplit : ms));
  };
  const size_t per_gu = n_cap * 2 * static_cast<size_t>(d.I_sub) * 4;
  const size_t per_dn = n_cap * static_cast<size_t>(d.H) * 4;
  l.max_split = splits(per_gu);
  l.max_split_down = splits(per_dn);
  const size_t need_gu = l.max_split > 1 ? l.max_split * per_gu : 0;
  const size_t need_dn = l.max_split_down > 1 ? l.max_split_down * per_dn : 0;
  l.partial = take(need_gu > need_dn ? need_gu : need_dn);
  // decode expert-pool folding: block scores and target map, folded routing
  l.fold_ws = take(moe::fold_workspace_bytes(d.T, static_cast<int>(E_r)));
  l.fold_idx = take(n_cap * 4);
  l.fold_w = take(n_cap * 4);
  l.fold_k = take(T * 4);
  // path-composed execution: distinct sources and their permutation,
  // distinct targets, the combine weights of the target rows, and the
  // target-ordered down input rows (in the permuted-x region when it is wide
  // enough: x_perm is free by then)
  l.p_srcs = take(n_cap * 4);
  l.p_nsrc = take(T * 4);
  l.p_slot = take(n_cap * 4);
  l.p_counts = take(E_r * 4);
  l.p_offsets = take((E_r + 1) * 4);
  l.p_sorted = take(n_cap * 4);
  l.p_inv = take(n_cap * 4);
  l.p_tgts = take(n_cap * 4);
  l.p_ntgt = take(T * 4);
  l.p_tslot = take(n_cap * 4);
  l.p_wtgt = take(n_cap * 4);
  l.p_act = d.I_sub <= d.H ? l.xperm : take(n_cap * d.I_sub * 2);
  l.total = o;
  return l;
}

template <typename P>
inline P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

moe_status validate(const moe_layer_desc* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARGUMENT;
  if (d->T < 0 || d->H <= 0 || d->n_experts <= 0 || d->n_sub <= 0 || d->I_sub <= 0 ||
      d->k_max <= 0 || d->I_shared < 0)
    return MOE_ERR_INVALID_ARGUMENT;
  if (d->score != MOE_SCORE_SOFTMAX && d->score != MOE_SCORE_SIGMOID)
    return MOE_ERR_INVALID_ARGUMENT;
  const long long E_r = static_cast<long long>(d->n_experts) * d->n_sub;
  if (d->H % 64 != 0 || d->I_sub % 64 != 0 || d->I_shared % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->H > 49152) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (E_r > 256 || d->k_max > E_r || d->k_max > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(d->T) * d->k_max > (1ll << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->I_shared > 0 && (d->w_shared_gate_up == nullptr || d->w_shared_down == nullptr))
    return MOE_ERR_INVALID_ARGUMENT;
  if (d->I_shared > 0 && (!aligned16(d->w_shared_gate_up) || !aligned16(d->w_shared_down)))
    return MOE_ERR_INVALID_ARGUMENT;
  return MOE_OK;
}

moe_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARGUMENT;
  return MOE_OK;
}

// int32 / fp32 arrays only need 4-byte alignment
moe_status check_ptrs4(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) != 0) return MOE_ERR_INVALID_ARGUMENT;
  return MOE_OK;
}

moe_status check_ws(const void* ws) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cache[dev] = n;
  }
  return cache[dev];
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                      \
  do {                                     \
    const moe_status _st = (expr);         \
    if (_st != MOE_OK) return _st;         \
  } while (0)

// Tokens per weight-stationary item: 64 when units hold few rows (decode),
// else larger chunks so each weight tile is reused across more tokens.
int decode_chunk(const moe_layer_desc* d) {
  return static_cast<long long>(d->T) * d->k_max <= 64ll * E_r_of(d) ? 64 : 128;
}

// ---- the steps, without argument checks (callers check)

// Router logits into dst: tcgen05 GEMM for T >= 128 with E_r in {64,128,256},
// else the CUDA-core kernel.
// Finished logits (with bias) into dst on the tensor cores.
// splits > 1: the K-split partial sums go to dst + s * T * E_r (no bias).
moe_status do_logits_gemm(const moe_layer_desc* d, const void* x, const void* router_w,
                          float* dst, int32_t* status, cudaStream_t s, int splits = 1,
                          int bn = 0) {
  const int E_r = E_r_of(d);
  GemmArgs g{};
  g.epi = moe::EPI_F32;
  g.a = x;
  g.a_rows = d->T;
  g.b = router_w;
  g.b_rows = E_r;
  g.K = d->H;
  g.offsets = nullptr;
  g.n_groups = 1;
  g.dense_rows = d->T;
  g.n_out = E_r;
  g.b_group_rows = 0;
  g.out = dst;
  g.ld_out = E_r;
  g.out_rows = d->T;
  g.bias = d->expert_bias;
  g.bias_div = d->n_sub;
  g.status = status;
  g.debug_flags = 0;
  g.sm_count = sm_count();
  g.max_rows_hint = d->T;
  // small batches: 64-column tiles for more CTAs; large ones: one n-tile,
  // so x is read once
  g.bn_hint = bn > 0 ? bn : (d->T < 4096 ? 64 : 0);
  g.k_splits = splits;
  g.split_stride = static_cast<long long>(d->T) * E_r;
  return cuda_status(moe::launch_gemm(g, s));
}

// bitmap_done (nullable): ask the top-k kernel to write the permutation's
// bitmap as well (layer forward, T >= kPermuteBitmapMinT); *bitmap_done says whether it did.
moe_status do_route(const moe_layer_desc* d, const void* x, const void* router_w,
                    const float* logits_in, const int32_t* kpt, float* logits_out,
                    int32_t* topk_idx, float* topk_w, int32_t* status, void* ws,
                    cudaStream_t s, bool* bitmap_done = nullptr) {
  if (bitmap_done != nullptr) *bitmap_done = false;
  const int E_r = E_r_of(d);
  const Layout l = layout_of(*d);
  const float* P = logits_in;   // what the top-k kernel sums
  int S = 1;
  const float* bias = nullptr;
  float* lout = nullptr;
  if (P == nullptr) {
    if (router_on_tensor_cores(*d)) {
      int bn = 0, splits = 1;
      moe::router_gemm_shape(d->T, d->H, E_r, &bn, &splits);
      if (splits > 1) {
        // K-split partial sums; the top-k kernel adds them in order, then the bias
        float* part = at<float>(ws, l.router_partial);
        MOE_TRY(do_logits_gemm(d, x, router_w, part, status, s, splits, bn));
        P = part;
        S = splits;
        bias = d->expert_bias;
        lout = logits_out;
      } else {
        float* dst = logits_out != nullptr ? logits_out : at<float>(ws, l.logits);
        MOE_TRY(do_logits_gemm(d, x, router_w, dst, status, s, 1, bn));
        P = dst;
      }
    } else if (moe::route_cluster_supports(d->H, E_r)) {
      return cuda_status(moe::launch_route_cluster(
          x, router_w, d->expert_bias, d->n_sub, kpt, d->T, d->H, E_r, d->k_max, d->score,
          d->renorm, d->route_scale, logits_out, topk_idx, topk_w, status, nullptr, s));
    } else {
      float* part = at<float>(ws, l.router_partial);
      MOE_TRY(cuda_status(
          moe::launch_router_logits_small(x, router_w, d->T, d->H, E_r, part, s)));
      P = part;
      S = l.router_slices;
      bias = d->expert_bias;
      lout = logits_out;
    }
  }
  uint32_t* bm = nullptr;
  if (bitmap_done != nullptr && d->T >= moe::kPermuteBitmapMinT) {
    bm = at<uint32_t>(ws, l.bitmap);
    *bitmap_done = true;
  }
  return cuda_status(moe::launch_topk_gate(P, S, bias, d->n_sub, lout, kpt, d->T, E_r, d->k_max,
                                           d->score, d->renorm, d->route_scale, topk_idx, topk_w,
                                           status, s, bm));
}

// Counters of the fused decode FFN kernel (one per token chunk, the work
// counter, the split counters), zeroed by the launch that precedes the FFN.
// Tokens per fused-decode-FFN item: 16 when no unit can hold more than 16
// rows (T <= 16), else 64.
inline int decode_ffn_chunk(const moe_layer_desc* d) { return d->T <= 16 ? 16 : 64; }
inline int decode_ffn_chunks(const moe_layer_desc* d) {
  return static_cast<int>(static_cast<long long>(d->T) * d->k_max / decode_ffn_chunk(d) +
                          E_r_of(d) + 1);
}
inline int decode_ffn_counters(const moe_layer_desc* d) {
  return decode_ffn_chunks(d) + 1 + moe::kFfnPartSlots / 2;
}

// zero_ffn: the permutation also zeroes the fused decode FFN's counters (the
// layer forward, whose FFN then gathers its token rows itself).
moe_status do_permute(const moe_layer_desc* d, const int32_t* topk_idx, const int32_t* kpt,
                      int32_t* counts, int32_t* offsets, int32_t* sorted_token,
                      int32_t* inv_row, int32_t* status, void* ws, cudaStream_t s,
                      bool bitmap_ready = false, bool zero_ffn = false) {
  const Layout l = layout_of(*d);
  return cuda_status(moe::launch_permute(
      topk_idx, kpt, d->T, d->k_max, E_r_of(d), at<uint32_t>(ws, l.bitmap),
      at<int32_t>(ws, l.wprefix), counts, offsets, sorted_token, inv_row, status, s,
      bitmap_ready, zero_ffn ? at<int32_t>(ws, l.chunk_done) : nullptr,
      zero_ffn ? decode_ffn_counters(d) : 0));
}

moe_status do_gate_up(const moe_layer_desc* d, const void* x, const int32_t* sorted_token,
                      const int32_t* offsets, const void* w_gate_up, void* act, int32_t* status,
                      void* ws, cudaStream_t s) {
  const Layout l = layout_of(*d);
  const int E_r = E_r_of(d);
  const long long n_cap = static_cast<long long>(d->T) * d->k_max;
  if (n_cap == 0) return MOE_OK;
  void* xperm = at<void>(ws, l.xperm);
  const bool decode = use_decode_path(d, d->I_sub, true);
  const bool pair = (d->debug_flags & MOE_DEBUG_FORCE_PAIR) != 0u;
  // the prefill kernels (single CTAs or CTA pairs) gather their A rows
  // themselves; the decode kernels read the permuted copy
  if (decode)
    MOE_TRY(cuda_status(moe::launch_gather_rows(x, sorted_token, offsets, E_r, d->T, d->H,
                                                static_cast<int>(n_cap), xperm, status,
                                                sm_count(), s)));
  if (decode) {
    moe::DecodeGemmArgs a{};
    a.gate_up = true;
    a.w = w_gate_up;
    a.w_rows = static_cast<long long>(E_r) * 2 * d->I_sub;
    a.x = xperm;
    a.x_rows = n_cap;
    a.K = d->H;
    a.offsets = offsets;
    a.n_groups = E_r;
    a.n_out = d->I_sub;
    a.w_group_rows = 2 * d->I_sub;
    a.out = act;
    a.out_rows = n_cap;
    a.partial = at<float>(ws, l.partial);
    a.split_word = at<int32_t>(ws, l.split_word);
    a.max_split = l.max_split;
    a.status = status;
    a.debug_flags = d->debug_flags;
    a.sm_count = sm_count();
    a.chunk = decode_chunk(d);
    return cuda_status(moe::launch_decode_gemm(a, s));
  }
  GemmArgs g{};
  g.epi = moe::EPI_SWIGLU;
  g.a = xperm;
  g.a_rows = n_cap;
  g.b = w_gate_up;
  g.b_rows = static_cast<long long>(E_r) * 2 * d->I_sub;
  g.K = d->H;
  g.offsets = offsets;
  g.n_groups = E_r;
  g.n_out = d->I_sub;
  g.b_group_rows = 2 * d->I_sub;
  g.out = act;
  g.ld_out = d->I_sub;
  g.out_rows = n_cap;
  g.status = status;
  g.debug_flags = d->debug_flags;
  g.force_pair = pair;
  g.gather_x = x;
  g.gather_tok = sorted_token;
  g.gather_rows = d->T;
  g.sm_count = sm_count();
  g.max_rows_hint = static_cast<int>(n_cap);
  return cuda_status(moe::launch_gemm(g, s));
}

moe_status do_down(const moe_layer_desc* d, const void* act, const int32_t* offsets,
                   const void* w_down, void* y_perm, int32_t* status, void* ws, cudaStream_t s) {
  const int E_r = E_r_of(d);
  const long long n_cap = static_cast<long long>(d->T) * d->k_max;
  if (n_cap == 0) return MOE_OK;
  if (use_decode_path(d, d->H, false)) {
    moe::DecodeGemmArgs a{};
    a.gate_up = false;
    a.w = w_down;
    a.w_rows = static_cast<long long>(E_r) * d->H;
    a.x = act;
    a.x_rows = n_cap;
    a.K = d->I_sub;
    a.offsets = offsets;
    a.n_groups = E_r;
    a.n_out = d->H;
    a.w_group_rows = d->H;
    const Layout l = layout_of(*d);
    a.out = y_perm;
    a.out_rows = n_cap;
    a.partial = at<float>(ws, l.partial);
    a.split_word = at<int32_t>(ws, l.split_word) + 1;
    a.max_split = l.max_split_down;
    a.status = status;
    a.debug_flags = 0;
    a.sm_count = sm_count();
    a.chunk = decode_chunk(d);
    return cuda_status(moe::launch_decode_gemm(a, s));
  }
  GemmArgs g{};
  g.epi = moe::EPI_BF16;
  g.a = act;
  g.a_rows = n_cap;
  g.b = w_down;
  g.b_rows = static_cast<long long>(E_r) * d->H;
  g.K = d->I_sub;
  g.offsets = offsets;
  g.n_groups = E_r;
  g.n_out = d->H;
  g.b_group_rows = d->H;
  g.out = y_perm;
  g.ld_out = d->H;
  g.out_rows = n_cap;
  g.status = status;
  g.debug_flags = 0;
  // The down projection reads act through TMA (no row gather), so CTA pairs
  // apply as they are: with K = I_sub >= 1024 their main loops are long
  // enough to win (DeepSeek-V3 shape, I_sub 2048: 2444 -> 2370 us measured
  // on GB300); with short K (Qwen3-30B-A3B shape, I_sub 768) single CTAs
  // stay ahead (140 vs 147 us).
  g.force_pair = (d->debug_flags & MOE_DEBUG_FORCE_PAIR) != 0u || d->I_sub >= 1024;
  g.sm_count = sm_count();
  g.max_rows_hint = static_cast<int>(n_cap);
  return cuda_status(moe::launch_gemm(g, s));
}

// Both FFN projections.  Decode-shaped batches with H and I_sub multiples of
// 128 run the fused kernel (gate|up and down overlapped in one launch);
// otherwise gate|up then down.
// gather_in_ffn: the decode FFN reads its token rows from x itself and its
// counters are already zero (the router or the permutation zeroed them);
// otherwise a row-gather launch writes x_perm and zeroes them.
moe_status do_grouped_ffn(const moe_layer_desc* d, const void* x, const int32_t* sorted_token,
                          const int32_t* offsets, const void* w_gate_up, const void* w_down,
                          void* y_perm, int32_t* status, void* ws, cudaStream_t s,
                          bool gather_in_ffn = false) {
  const Layout l = layout_of(*d);
  void* act = at<void>(ws, l.act);
  const long long n_cap = static_cast<long long>(d->T) * d->k_max;
  if (n_cap == 0) return MOE_OK;
  if (use_decode_ffn(d)) {
    const int E_r = E_r_of(d);
    void* xperm = at<void>(ws, l.xperm);
    int32_t* done = at<int32_t>(ws, l.chunk_done);
    // the counters are zeroed by the launch that precedes the FFN: the row
    // gather, or the fused router or the permutation (gather_in_ffn)
    if (!gather_in_ffn)
      MOE_TRY(cuda_status(moe::launch_gather_rows(x, sorted_token, offsets, E_r, d->T, d->H,
                                                  static_cast<int>(n_cap), xperm, status,
                                                  sm_count(), s, done, decode_ffn_counters(d))));
    moe::DecodeFfnArgs a{};
    a.x_perm = xperm;
    a.x_rows = n_cap;
    a.w_gate_up = w_gate_up;
    a.w_down = w_down;
    a.offsets = offsets;
    a.n_groups = E_r;
    a.H = d->H;
    a.I = d->I_sub;
    a.act = act;
    a.y = y_perm;
    a.chunk = decode_ffn_chunk(d);
    a.done = done;
    a.work = done + decode_ffn_chunks(d);
    a.split_cnt = a.work + 1;
    a.part = at<float>(ws, l.ffn_part);
    a.rows = n_cap;
    a.status = status;
    a.debug_flags = d->debug_flags;
    a.sm_count = sm_count();
    if (gather_in_ffn) {
      a.gather_x = x;
      a.gather_tok = sorted_token;
      a.gather_rows = d->T;
    }
    return cuda_status(moe::launch_decode_ffn(a, s));
  }
  MOE_TRY(do_gate_up(d, x, sorted_token, offsets, w_gate_up, act, status, ws, s));
  return do_down(d, act, offsets, w_down, y_perm, status, ws, s);
}

moe_status do_shared(const moe_layer_desc* d, const void* x, void* y_shared, int32_t* status,
                     void* ws, cudaStream_t s) {
  if (d->T == 0) return MOE_OK;
  const Layout l = layout_of(*d);
  void* act = at<void>(ws, l.act_sh);
  GemmArgs g{};
  g.epi = moe::EPI_SWIGLU;
  g.a = x;
  g.a_rows = d->T;
  g.b = d->w_shared_gate_up;
  g.b_rows = 2ll * d->I_shared;
  g.K = d->H;
  g.offsets = nullptr;
  g.n_groups = 1;
  g.dense_rows = d->T;
  g.n_out = d->I_shared;
  g.b_group_rows = 2 * d->I_shared;
  g.out = act;
  g.ld_out = d->I_shared;
  g.out_rows = d->T;
  g.status = status;
  g.sm_count = sm_count();
  g.max_rows_hint = d->T;
  MOE_TRY(cuda_status(moe::launch_gemm(g, s)));
  GemmArgs h{};
  h.epi = moe::EPI_BF16;
  h.a = act;
  h.a_rows = d->T;
  h.b = d->w_shared_down;
  h.b_rows = d->H;
  h.K = d->I_shared;
  h.offsets = nullptr;
  h.n_groups = 1;
  h.dense_rows = d->T;
  h.n_out = d->H;
  h.b_group_rows = d->H;
  h.out = y_shared;
  h.ld_out = d->H;
  h.out_rows = d->T;
  h.status = status;
  h.sm_count = sm_count();
  h.max_rows_hint = d->T;
  return cuda_status(moe::launch_gemm(h, s));
}

moe_status do_combine(const moe_layer_desc* d, const void* y_perm, const void* y_shared,
                      const int32_t* inv_row, const float* topk_w, const int32_t* kpt, void* out,
                      int32_t* status, cudaStream_t s) {
  const long long n_cap = static_cast<long long>(d->T) * d->k_max;
  return cuda_status(moe::launch_combine(y_perm, y_shared, inv_row, topk_w, kpt, d->T, d->H,
                                         d->k_max, static_cast<int>(n_cap), out, status, s));
}

// ---------------------------------------------------------------- expert-pool folding

moe_status validate_fold(const moe_layer_desc* d, const moe_fold_desc* f) {
  MOE_TRY(validate(d));
  if (f == nullptr) return MOE_ERR_INVALID_ARGUMENT;
  if (f->D < 1 || f->D > E_r_of(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  MOE_TRY(check_ptrs4({f->S, f->L}));
  if (f->pool != nullptr) MOE_TRY(check_ptrs4({f->pool}));
  if (f->unit_scale != nullptr) MOE_TRY(check_ptrs4({f->unit_scale}));
  return MOE_OK;
}

moe_status do_fold(const moe_layer_desc* d, const moe_fold_desc* f, const int32_t* topk_idx,
                   const float* topk_w, const int32_t* kpt, int32_t* idx_out, float* w_out,
                   int32_t* k_out, int32_t* pool_out, int32_t* status, void* ws, cudaStream_t s) {
  const Layout l = layout_of(*d);
  return cuda_status(moe::launch_fold_decode(topk_idx, topk_w, kpt, d->T, d->k_max, E_r_of(d),
                                             f->D, f->pool, f->unit_scale, f->S, f->L, idx_out,
                                             w_out, k_out, pool_out, at<void>(ws, l.fold_ws),
                                             status, s));
}

// ---------------------------------------------------------------- composed paths

moe_status do_layer_paths(const moe_layer_desc* d, const void* x, const void* w_gate_up,
                          const void* w_down, const int32_t* src_idx, const int32_t* tgt_idx,
                          const float* beta, const int32_t* n_paths, void* out,
                          int32_t* status, void* ws, cudaStream_t s) {
  const Layout l = layout_of(*d);
  const int E_r = E_r_of(d);
  const long long n_cap = static_cast<long long>(d->T) * d->k_max;
  int32_t* srcs = at<int32_t>(ws, l.p_srcs);
  int32_t* nsrc = at<int32_t>(ws, l.p_nsrc);
  int32_t* slot = at<int32_t>(ws, l.p_slot);
  int32_t* offs_s = at<int32_t>(ws, l.p_offsets);
  int32_t* sorted_s = at<int32_t>(ws, l.p_sorted);
  int32_t* inv_s = at<int32_t>(ws, l.p_inv);
  int32_t* tgts = at<int32_t>(ws, l.p_tgts);
  int32_t* ntgt = at<int32_t>(ws, l.p_ntgt);
  int32_t* tslot = at<int32_t>(ws, l.p_tslot);
  float* wtgt = at<float>(ws, l.p_wtgt);
  int32_t* counts = at<int32_t>(ws, l.counts);
  int32_t* offsets = at<int32_t>(ws, l.offsets);
  int32_t* sorted_token = at<int32_t>(ws, l.sorted_token);
  int32_t* inv_row = at<int32_t>(ws, l.inv_row);
  void* act_s = at<void>(ws, l.act);
  void* act_p = at<void>(ws, l.p_act);
  void* yperm = at<void>(ws, l.yperm);
  // expansions: one per (token, distinct source)
  MOE_TRY(cuda_status(moe::launch_paths_sources(src_idx, n_paths, d->T, d->k_max, E_r, srcs,
                                                nsrc, slot, status, s)));
  MOE_TRY(do_permute(d, srcs, nsrc, at<int32_t>(ws, l.p_counts), offs_s, sorted_s, inv_s, status,
                     ws, s));
  MOE_TRY(do_gate_up(d, x, sorted_s, offs_s, w_gate_up, act_s, status, ws, s));
  // projections: one per (token, distinct target); its input row is the
  // beta-weighted sum of the expansions of the paths into that target
  MOE_TRY(cuda_status(moe::launch_paths_sources(tgt_idx, n_paths, d->T, d->k_max, E_r, tgts,
                                                ntgt, tslot, status, s)));
  MOE_TRY(do_permute(d, tgts, ntgt, counts, offsets, sorted_token, inv_row, status, ws, s));
  MOE_TRY(cuda_status(moe::launch_paths_merge(n_paths, slot, tslot, ntgt, beta, inv_s, inv_row,
                                              act_s, d->T, d->k_max, d->I_sub, n_cap, n_cap,
                                              act_p, wtgt, status, s)));
  MOE_TRY(do_down(d, act_p, offsets, w_down, yperm, status, ws, s));
  void* ysh = d->I_shared > 0 ? at<void>(ws, l.ysh) : nullptr;
  if (ysh != nullptr) MOE_TRY(do_shared(d, x, ysh, status, ws, s));
  return do_combine(d, yperm, ysh, inv_row, wtgt, ntgt, out, status, s);
}

// ---------------------------------------------------------------- proxy router

moe_status validate_cg(const moe_layer_desc* d, const moe_cg_router* cg) {
  MOE_TRY(validate(d));
  if (cg == nullptr) return MOE_ERR_INVALID_ARGUMENT;
  if (cg->m < 1 || cg->m > d->n_experts || cg->m > 32 || cg->r < 1 || cg->r > d->I_sub)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->n_sub > 32 || d->k_max > cg->m * d->n_sub) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (cg->m * d->n_sub * cg->r > moe::kMaxProxyPairs) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// The expert-level router: the layer's desc with one unit per expert and the
// native m as k.
moe_layer_desc expert_desc(const moe_layer_desc& d, int m) {
  moe_layer_desc e = d;
  e.n_sub = 1;
  e.k_max = m;
  e.I_shared = 0;
  return e;
}

struct CgLayout {
  size_t e_logits, e_part, e_idx, e_w, p_buf, total;
  int e_slices;   // 0: expert logits on the tensor cores
  bool p_dense;   // proxy pre-activations of every unit on the tensor cores (else kept
                  // experts only, on CUDA cores)
  int R;          // packed proxy rows = E_r * 2r
};

bool proxy_on_tensor_cores(const moe_layer_desc& d, int R) { return d.T >= 128 && R % 64 == 0; }

// Placed after the layer's own workspace layout.
CgLayout cg_layout_of(const moe_layer_desc& d, const moe_cg_router& cg) {
  const size_t T = static_cast<size_t>(d.T), E = static_cast<size_t>(d.n_experts);
  const moe_layer_desc ed = expert_desc(d, cg.m);
  CgLayout c;
  size_t o = layout_of(d).total;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  int vs = 0;
  c.R = E_r_of(&d) * 2 * cg.r;
  c.e_slices = router_on_tensor_cores(ed) ? 0 : moe::router_slices(d.T, d.H, d.n_experts, &vs);
  c.p_dense = proxy_on_tensor_cores(d, c.R);
  c.e_logits = take(T * E * 4);
  c.e_part = take(static_cast<size_t>(c.e_slices) * T * E * 4);
  c.e_idx = take(T * cg.m * 4);
  c.e_w = take(T * cg.m * 4);
  const size_t rows_e = static_cast<size_t>(d.n_sub) * 2 * cg.r;   // per kept expert
  c.p_buf = take(c.p_dense ? T * c.R * 4 : T * cg.m * rows_e * 4);
  c.total = o;
  return c;
}

moe_status do_route_cg(const moe_layer_desc* d, const moe_cg_router* cg, const void* x,
                       const int32_t* kpt, float* expert_logits_out, float* proxy_out,
                       int32_t* topk_idx, float* topk_w, int32_t* status, void* ws,
                       cudaStream_t s) {
  const CgLayout c = cg_layout_of(*d, *cg);
  const moe_layer_desc ed = expert_desc(*d, cg->m);
  int32_t* eidx = at<int32_t>(ws, c.e_idx);
  float* ew = at<float>(ws, c.e_w);
  // 1. the original router keeps m experts per token
  if (c.e_slices == 0) {
    float* dst = expert_logits_out != nullptr ? expert_logits_out : at<float>(ws, c.e_logits);
    MOE_TRY(do_logits_gemm(&ed, x, cg->router_w_expert, dst, status, s));
    MOE_TRY(cuda_status(moe::launch_topk_gate(dst, 1, nullptr, 1, nullptr, nullptr, d->T,
                                              d->n_experts, cg->m, d->score, d->renorm,
                                              d->route_scale, eidx, ew, status, s)));
  } else {
    float* part = at<float>(ws, c.e_part);
    MOE_TRY(cuda_status(moe::launch_router_logits_small(x, cg->router_w_expert, d->T, d->H,
                                                        d->n_experts, part, s)));
    MOE_TRY(cuda_status(moe::launch_topk_gate(part, c.e_slices, d->expert_bias, 1,
                                              expert_logits_out, nullptr, d->T, d->n_experts,
                                              cg->m, d->score, d->renorm, d->route_scale, eidx,
                                              ew, status, s)));
  }
  // 2. gate-neuron pre-activations of every unit (not needed when every
  // expert has a single sub-expert and nobody asks for the scores)
  float* pre = at<float>(ws, c.p_buf);
  int S = 1;
  if (d->n_sub == 1 && proxy_out == nullptr) {
    pre = nullptr;
  } else if (c.p_dense) {
    GemmArgs g{};
    g.epi = moe::EPI_F32;
    g.a = x;
    g.a_rows = d->T;
    g.b = cg->proxy_w;
    g.b_rows = c.R;
    g.K = d->H;
    g.offsets = nullptr;
    g.n_groups = 1;
    g.dense_rows = d->T;
    g.n_out = c.R;
    g.b_group_rows = 0;
    g.out = pre;
    g.ld_out = c.R;
    g.out_rows = d->T;
    g.bias = nullptr;
    g.bias_div = 1;
    g.status = status;
    g.sm_count = sm_count();
    g.max_rows_hint = d->T;
    g.bn_hint = c.R % 256 == 0 ? 256 : (c.R % 128 == 0 ? 128 : 64);
    MOE_TRY(cuda_status(moe::launch_gemm(g, s)));
  } else {
    MOE_TRY(cuda_status(moe::launch_proxy_gemv(x, cg->proxy_w, eidx, d->T, d->H, d->n_experts,
                                               cg->m, d->n_sub * 2 * cg->r, pre, s)));
  }
  // 3. proxy scores and the per-expert top-kappa_j
  return cuda_status(moe::launch_cg_select(pre, S, c.R, !c.p_dense, eidx, ew, cg->kappa, kpt,
                                           d->T, cg->m,
                                           d->n_sub, cg->r, d->k_max, d->n_experts, proxy_out,
                                           topk_idx, topk_w, status, s));
}

}  // namespace

namespace moe {
moe_status validate_desc(const moe_layer_desc* d) { return validate(d); }
}  // namespace moe

extern "C" {

size_t moe_workspace_size(const moe_layer_desc* desc) {
  if (validate(desc) != MOE_OK) return 0;
  return layout_of(*desc).total;
}

moe_status moe_route(const moe_layer_desc* desc, const void* x, const void* router_w,
                     const float* logits_in, const int32_t* k_per_token, float* logits_out,
                     int32_t* topk_idx, float* topk_w, int32_t* dev_status, void* workspace,
                     void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs4({k_per_token, topk_idx, topk_w, dev_status}));
  if (logits_in != nullptr) {
    MOE_TRY(check_ptrs4({logits_in}));
  } else {
    MOE_TRY(check_ptrs({x, router_w}));
    if (logits_out != nullptr) MOE_TRY(check_ptrs({logits_out}));
    MOE_TRY(check_ws(workspace));
  }
  return do_route(desc, x, router_w, logits_in, k_per_token, logits_out, topk_idx, topk_w,
                  dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_layer_desc* desc, const int32_t* topk_idx,
                       const int32_t* k_per_token, int32_t* counts, int32_t* offsets,
                       int32_t* sorted_token, int32_t* inv_row, int32_t* dev_status,
                       void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  MOE_TRY(check_ptrs4({counts, offsets, dev_status}));
  if (desc->T > 0) MOE_TRY(check_ptrs4({topk_idx, k_per_token, sorted_token, inv_row}));
  MOE_TRY(check_ws(workspace));
  return do_permute(desc, topk_idx, k_per_token, counts, offsets, sorted_token, inv_row,
                    dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_gate_up(const moe_layer_desc* desc, const void* x, const int32_t* sorted_token,
                       const int32_t* offsets, const void* w_gate_up, void* act,
                       int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, w_gate_up, act}));
  MOE_TRY(check_ptrs4({sorted_token, offsets, dev_status}));
  MOE_TRY(check_ws(workspace));
  return do_gate_up(desc, x, sorted_token, offsets, w_gate_up, act, dev_status, workspace,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_down(const moe_layer_desc* desc, const void* act, const int32_t* offsets,
                    const void* w_down, void* y_perm, int32_t* dev_status, void* workspace,
                    void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({act, w_down, y_perm}));
  MOE_TRY(check_ptrs4({offsets, dev_status}));
  MOE_TRY(check_ws(workspace));
  return do_down(desc, act, offsets, w_down, y_perm, dev_status, workspace,
                 static_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_ffn(const moe_layer_desc* desc, const void* x,
                           const int32_t* sorted_token, const int32_t* offsets,
                           const void* w_gate_up, const void* w_down, void* y_perm,
                           int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, w_gate_up, w_down, y_perm}));
  MOE_TRY(check_ptrs4({sorted_token, offsets, dev_status}));
  MOE_TRY(check_ws(workspace));
  return do_grouped_ffn(desc, x, sorted_token, offsets, w_gate_up, w_down, y_perm, dev_status,
                        workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_shared_ffn(const moe_layer_desc* desc, const void* x, void* y_shared,
                          int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->I_shared <= 0) return MOE_ERR_INVALID_ARGUMENT;
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, y_shared}));
  MOE_TRY(check_ptrs4({dev_status}));
  MOE_TRY(check_ws(workspace));
  return do_shared(desc, x, y_shared, dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_layer_desc* desc, const void* y_perm, const void* y_shared,
                       const int32_t* inv_row, const float* topk_w, const int32_t* k_per_token,
                       void* out, int32_t* dev_status, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({y_perm, out}));
  if (y_shared != nullptr) MOE_TRY(check_ptrs({y_shared}));
  MOE_TRY(check_ptrs4({inv_row, topk_w, k_per_token, dev_status}));
  return do_combine(desc, y_perm, y_shared, inv_row, topk_w, k_per_token, out, dev_status,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, const void* router_w,
                             const void* w_gate_up, const void* w_down,
                             const int32_t* k_per_token, void* out, int32_t* dev_status,
                             void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, router_w, w_gate_up, w_down, out}));
  MOE_TRY(check_ptrs4({k_per_token, dev_status}));
  MOE_TRY(check_ws(workspace));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout l = layout_of(*desc);
  int32_t* topk_idx = at<int32_t>(workspace, l.topk_idx);
  float* topk_w = at<float>(workspace, l.topk_w);
  int32_t* counts = at<int32_t>(workspace, l.counts);
  int32_t* offsets = at<int32_t>(workspace, l.offsets);
  int32_t* sorted_token = at<int32_t>(workspace, l.sorted_token);
  int32_t* inv_row = at<int32_t>(workspace, l.inv_row);
  void* act = at<void>(workspace, l.act);
  void* yperm = at<void>(workspace, l.yperm);
  void* ysh = desc->I_shared > 0 ? at<void>(workspace, l.ysh) : nullptr;
  const int E_r = E_r_of(desc);
  // the fused decode FFN gathers its token rows from x itself; the launch
  // before it (router or permutation) zeroes its counters
  const bool gather_in_ffn = use_decode_ffn(desc);
  if (desc->T <= moe::kRouteFuseMaxT && !router_on_tensor_cores(*desc) &&
      moe::route_cluster_supports(desc->H, E_r)) {
    // small batch: logits, top-k and permutation in one launch
    moe::RoutePermuteOut f{counts, offsets, sorted_token, inv_row,
                           gather_in_ffn ? at<int32_t>(workspace, l.chunk_done) : nullptr,
                           gather_in_ffn ? decode_ffn_counters(desc) : 0};
    MOE_TRY(cuda_status(moe::launch_route_cluster(
        x, router_w, desc->expert_bias, desc->n_sub, k_per_token, desc->T, desc->H, E_r,
        desc->k_max, desc->score, desc->renorm, desc->route_scale, nullptr, topk_idx, topk_w,
        dev_status, &f, s)));
  } else {
    bool bitmap_done = false;
    MOE_TRY(do_route(desc, x, router_w, nullptr, k_per_token, nullptr, topk_idx, topk_w,
                     dev_status, workspace, s, &bitmap_done));
    MOE_TRY(do_permute(desc, topk_idx, k_per_token, counts, offsets, sorted_token, inv_row,
                       dev_status, workspace, s, bitmap_done, gather_in_ffn));
  }
  if (ysh != nullptr) MOE_TRY(do_shared(desc, x, ysh, dev_status, workspace, s));
  MOE_TRY(do_grouped_ffn(desc, x, sorted_token, offsets, w_gate_up, w_down, yperm, dev_status,
                         workspace, s, gather_in_ffn));
  return do_combine(desc, yperm, ysh, inv_row, topk_w, k_per_token, out, dev_status, s);
}

moe_status moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host,
                                  const int32_t* k_host, void* out_host, void* x_dev,
                                  int32_t* k_dev, void* out_dev, const void* router_w,
                                  const void* w_gate_up, const void* w_down,
                                  int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  if (x_host == nullptr || k_host == nullptr || out_host == nullptr)
    return MOE_ERR_INVALID_ARGUMENT;
  MOE_TRY(check_ptrs({x_dev, router_w, w_gate_up, w_down, out_dev}));
  MOE_TRY(check_ptrs4({k_dev, dev_status}));
  MOE_TRY(check_ws(workspace));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t act_bytes = static_cast<size_t>(desc->T) * desc->H * 2;
  MOE_TRY(cuda_status(cudaMemcpyAsync(x_dev, x_host, act_bytes, cudaMemcpyHostToDevice, s)));
  MOE_TRY(cuda_status(cudaMemcpyAsync(k_dev, k_host, static_cast<size_t>(desc->T) * 4,
                                      cudaMemcpyHostToDevice, s)));
  MOE_TRY(moe_layer_forward(desc, x_dev, router_w, w_gate_up, w_down, k_dev, out_dev,
                            dev_status, workspace, stream));
  return cuda_status(cudaMemcpyAsync(out_host, out_dev, act_bytes, cudaMemcpyDeviceToHost, s));
}

size_t moe_cg_workspace_size(const moe_layer_desc* desc, const moe_cg_router* cg) {
  if (validate_cg(desc, cg) != MOE_OK) return 0;
  return cg_layout_of(*desc, *cg).total;
}

moe_status moe_pack_proxy_rows(const moe_layer_desc* desc, int32_t r, const void* w_gate_up,
                               const int32_t* gate_neurons, void* proxy_w, int32_t* dev_status,
                               void* stream) {
  MOE_TRY(validate(desc));
  if (r < 1 || r > desc->I_sub) return MOE_ERR_UNSUPPORTED_SHAPE;
  MOE_TRY(check_ptrs({w_gate_up, proxy_w}));
  MOE_TRY(check_ptrs4({gate_neurons, dev_status}));
  return cuda_status(moe::launch_pack_proxy(w_gate_up, gate_neurons, E_r_of(desc), r,
                                            desc->I_sub, desc->H, proxy_w, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_cg(const moe_layer_desc* desc, const moe_cg_router* cg, const void* x,
                        const int32_t* k_per_token, float* expert_logits_out, float* proxy_out,
                        int32_t* topk_idx, float* topk_w, int32_t* dev_status, void* workspace,
                        void* stream) {
  MOE_TRY(validate_cg(desc, cg));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, cg->router_w_expert, cg->proxy_w}));
  MOE_TRY(check_ptrs4({cg->kappa, k_per_token, topk_idx, topk_w, dev_status}));
  if (expert_logits_out != nullptr) MOE_TRY(check_ptrs4({expert_logits_out}));
  if (proxy_out != nullptr) MOE_TRY(check_ptrs4({proxy_out}));
  MOE_TRY(check_ws(workspace));
  return do_route_cg(desc, cg, x, k_per_token, expert_logits_out, proxy_out, topk_idx, topk_w,
                     dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward_cg(const moe_layer_desc* desc, const moe_cg_router* cg,
                                const void* x, const void* w_gate_up, const void* w_down,
                                const int32_t* k_per_token, void* out, int32_t* dev_status,
                                void* workspace, void* stream) {
  MOE_TRY(validate_cg(desc, cg));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, cg->router_w_expert, cg->proxy_w, w_gate_up, w_down, out}));
  MOE_TRY(check_ptrs4({cg->kappa, k_per_token, dev_status}));
  MOE_TRY(check_ws(workspace));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout l = layout_of(*desc);
  int32_t* topk_idx = at<int32_t>(workspace, l.topk_idx);
  float* topk_w = at<float>(workspace, l.topk_w);
  int32_t* counts = at<int32_t>(workspace, l.counts);
  int32_t* offsets = at<int32_t>(workspace, l.offsets);
  int32_t* sorted_token = at<int32_t>(workspace, l.sorted_token);
  int32_t* inv_row = at<int32_t>(workspace, l.inv_row);
  void* yperm = at<void>(workspace, l.yperm);
  void* ysh = desc->I_shared > 0 ? at<void>(workspace, l.ysh) : nullptr;
  MOE_TRY(do_route_cg(desc, cg, x, k_per_token, nullptr, nullptr, topk_idx, topk_w, dev_status,
                      workspace, s));
  MOE_TRY(do_permute(desc, topk_idx, k_per_token, counts, offsets, sorted_token, inv_row,
                     dev_status, workspace, s));
  if (ysh != nullptr) MOE_TRY(do_shared(desc, x, ysh, dev_status, workspace, s));
  MOE_TRY(do_grouped_ffn(desc, x, sorted_token, offsets, w_gate_up, w_down, yperm, dev_status,
                         workspace, s));
  return do_combine(desc, yperm, ysh, inv_row, topk_w, k_per_token, out, dev_status, s);
}

moe_status moe_fold_decode(const moe_layer_desc* desc, const moe_fold_desc* fold,
                           const int32_t* topk_idx, const float* topk_w,
                           const int32_t* k_per_token, int32_t* topk_idx_out,
                           float* topk_w_out, int32_t* k_out, int32_t* pool_out,
                           int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate_fold(desc, fold));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs4({topk_idx, topk_w, k_per_token, topk_idx_out, topk_w_out, k_out,
                       dev_status}));
  if (pool_out != nullptr) MOE_TRY(check_ptrs4({pool_out}));
  MOE_TRY(check_ws(workspace));
  return do_fold(desc, fold, topk_idx, topk_w, k_per_token, topk_idx_out, topk_w_out, k_out,
                 pool_out, dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward_fold(const moe_layer_desc* desc, const moe_fold_desc* fold,
                                  const void* x, const void* router_w, const void* w_gate_up,
                                  const void* w_down, const int32_t* k_per_token, void* out,
                                  int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate_fold(desc, fold));
  if (desc->T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, router_w, w_gate_up, w_down, out}));
  MOE_TRY(check_ptrs4({k_per_token, dev_status}));
  MOE_TRY(check_ws(workspace));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout l = layout_of(*desc);
  int32_t* topk_idx = at<int32_t>(workspace, l.topk_idx);
  float* topk_w = at<float>(workspace, l.topk_w);
  int32_t* fidx = at<int32_t>(workspace, l.fold_idx);
  float* fw = at<float>(workspace, l.fold_w);
  int32_t* fk = at<int32_t>(workspace, l.fold_k);
  int32_t* counts = at<int32_t>(workspace, l.counts);
  int32_t* offsets = at<int32_t>(workspace, l.offsets);
  int32_t* sorted_token = at<int32_t>(workspace, l.sorted_token);
  int32_t* inv_row = at<int32_t>(workspace, l.inv_row);
  void* yperm = at<void>(workspace, l.yperm);
  void* ysh = desc->I_shared > 0 ? at<void>(workspace, l.ysh) : nullptr;
  MOE_TRY(do_route(desc, x, router_w, nullptr, k_per_token, nullptr, topk_idx, topk_w,
                   dev_status, workspace, s));
  MOE_TRY(do_fold(desc, fold, topk_idx, topk_w, k_per_token, fidx, fw, fk, nullptr, dev_status,
                  workspace, s));
  MOE_TRY(do_permute(desc, fidx, fk, counts, offsets, sorted_token, inv_row, dev_status,
                     workspace, s));
  if (ysh != nullptr) MOE_TRY(do_shared(desc, x, ysh, dev_status, workspace, s));
  MOE_TRY(do_grouped_ffn(desc, x, sorted_token, offsets, w_gate_up, w_down, yperm, dev_status,
                         workspace, s));
  return do_combine(desc, yperm, ysh, inv_row, fw, fk, out, dev_status, s);
}

moe_status moe_layer_forward_paths(const moe_layer_desc* desc, const void* x,
                                   const void* w_gate_up, const void* w_down,
                                   const int32_t* src_idx, const int32_t* tgt_idx,
                                   const float* beta, const int32_t* n_paths, void* out,
                                   int32_t* dev_status, void* workspace, void* stream) {
  MOE_TRY(validate(desc));
  if (desc->T == 0) return MOE_OK;
  if (desc->I_sub % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  MOE_TRY(check_ptrs({x, w_gate_up, w_down, out}));
  MOE_TRY(check_ptrs4({src_idx, tgt_idx, beta, n_paths, dev_status}));
  MOE_TRY(check_ws(workspace));
  return do_layer_paths(desc, x, w_gate_up, w_down, src_idx, tgt_idx, beta, n_paths, out,
                        dev_status, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_get_device_status(const int32_t* dev_status, void* stream) {
  if (dev_status == nullptr) return MOE_ERR_INVALID_ARGUMENT;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARGUMENT: return "MOE_ERR_INVALID_ARGUMENT";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE";
    case MOE_ERR_K_RANGE: return "MOE_ERR_K_RANGE";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX";
  }
  return "MOE_ERR_UNKNOWN";
}

}  // extern "C"
