// Host-side launchers of the libmoe kernels (internal; the public ABI is
// include/moe.h).  Each launcher enqueues on `stream` and returns the
// cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- api.cu
// Host validation of a layer descriptor: the status every entry point of
// include/moe.h returns for an invalid or unsupported descriptor.
moe_status validate_desc(const moe_layer_desc* d);

// ---- route.cu
// Partial logits P[s, t, u] over router_slices(T, H, E_r) slices of the
// hidden dimension (no bias); P: fp32 [S, T, E_r], S <= router_slices_max(H).
int router_slices(int T, int H, int E_r, int* vec_per_slice);
int router_slices_max(int H);
cudaError_t launch_router_logits_small(const void* x, const void* router_w, int T, int H,
                                       int E_r, float* partial, cudaStream_t s);
// Top-k_t and gates from the sum of S partial logit arrays [S, T, E_r] (S = 1:
// finished logits) plus bias[u / n_sub] (nullable); logits_out (nullable)
// receives the summed logits; k_per_token == nullptr keeps k_max per token.
// bitmap (nullable): also write the permutation's unit membership bitmap
// ([E_r][ceil(T/32)] uint32, the layout launch_permute builds), so that
// launch_permute can be told it is ready.
cudaError_t launch_topk_gate(const float* partial, int S, const float* bias, int n_sub,
                             float* logits_out, const int32_t* k_per_token, int T, int E_r,
                             int k_max, int score, int renorm, float route_scale,
                             int32_t* topk_idx, float* topk_w, int32_t* status,
                             cudaStream_t s, uint32_t* bitmap = nullptr);

// Logits and top-k_t of clusters of eight tokens in one launch (mma.sync
// tiles, H % 16 == 0, E_r <= 256).  With `fuse` (T <= 8 only) the same launch also
// writes the permutation (counts, offsets, sorted_token, inv_row) and zeroes
// zero_ptr[0, zero_n).  Router rows and the expert bias are read before the
// launch's dependency wait (they are layer parameters); x and k after it.
struct RoutePermuteOut {
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_token;
  int32_t* inv_row;
  int32_t* zero_ptr;   // counters of the kernel that follows, zeroed here (nullable)
  int zero_n;
};
bool route_cluster_supports(int H, int E_r);
constexpr int kRouteFuseMaxT = 8;
cudaError_t launch_route_cluster(const void* x, const void* router_w, const float* bias,
                                 int n_sub, const int32_t* k_per_token, int T, int H, int E_r,
                                 int k_max, int score, int renorm, float route_scale,
                                 float* logits_out, int32_t* topk_idx, float* topk_w,
                                 int32_t* status, const RoutePermuteOut* fuse, cudaStream_t s);

// ---- cg_router.cu: training-free proxy router
constexpr int kMaxProxyPairs = 2048;   // m * n_sub * r per token (8 KB of scores per warp)
cudaError_t launch_pack_proxy(const void* w_gate_up, const int32_t* gate_neurons, int E_r, int r,
                              int I_sub, int H, void* proxy_w, int32_t* status, cudaStream_t s);
// Pre-activations of the kept experts' gate-neuron rows only: out fp32
// [T, m, rows_e] (rows_e = n_sub * 2r); H <= 49152.
cudaError_t launch_proxy_gemv(const void* x, const void* proxy_w, const int32_t* expert_idx,
                              int T, int H, int n_experts, int m, int rows_e, float* out,
                              cudaStream_t s);
// partial: S arrays [T, R] (R = E_r * 2r), or with compact one [T, m, n_sub * 2r]
cudaError_t launch_cg_select(const float* partial, int S, int R, bool compact,
                             const int32_t* expert_idx, const float* expert_w,
                             const int32_t* kappa, const int32_t* kpt, int T, int m, int N,
                             int r, int k_max, int n_experts, float* proxy_out, int32_t* topk_idx,
                             float* topk_w, int32_t* status, cudaStream_t s);

// ---- fold.cu: decode expert-pool folding
// Workspace bytes: ceil(T/64) * E_r fp32 block scores + target map.
size_t fold_workspace_bytes(int T, int E_r);
// pool_in == nullptr: dynamic pool of D units; S, L: fp32 [E_r, E_r];
// unit_scale nullable; pool_out nullable ([D], ascending).
cudaError_t launch_fold_decode(const int32_t* topk_idx, const float* topk_w,
                               const int32_t* k_per_token, int T, int k_max, int E_r, int D,
                               const int32_t* pool_in, const float* unit_scale, const float* S,
                               const float* L, int32_t* idx_out, float* w_out, int32_t* k_out,
                               int32_t* pool_out, void* ws, int32_t* status, cudaStream_t s);

// ---- paths.cu: path-composed execution
// Distinct values of a per-path unit list (sources or targets) per token in
// first-occurrence order, their count, and each path's position among them
// (all [T, k_max] / [T]).
cudaError_t launch_paths_sources(const int32_t* src_idx, const int32_t* n_paths, int T, int k_max,
                                 int E_r, int32_t* srcs, int32_t* n_src, int32_t* slot,
                                 int32_t* status, cudaStream_t s);
// Down input of every (token, distinct target) row: act_tgt[inv_tgt[t, ts]] =
// bf16(sum over the token's paths j with tslot[t, j] == ts, in path order, of
// beta[t, j] * act_src[inv_src[t, slot[t, j]]]) in fp32; w_tgt[t, ts] = 1.
cudaError_t launch_paths_merge(const int32_t* n_paths, const int32_t* slot, const int32_t* tslot,
                               const int32_t* n_tgt, const float* beta, const int32_t* inv_src,
                               const int32_t* inv_tgt, const void* act_src, int T, int k_max,
                               int I_sub, long long n_src_rows, long long n_tgt_rows,
                               void* act_tgt, float* w_tgt, int32_t* status, cudaStream_t s);

// ---- permute.cu
// bitmap_ready: the top-k kernel already wrote `bitmap` (T >= kPermuteBitmapMinT only).
// Also zeroes zero_ptr[0, zero_n) (counters of the kernel that follows).
cudaError_t launch_permute(const int32_t* topk_idx, const int32_t* k_per_token, int T,
                           int k_max, int E_r, uint32_t* bitmap, int32_t* wprefix,
                           int32_t* counts, int32_t* offsets, int32_t* sorted_token,
                           int32_t* inv_row, int32_t* status, cudaStream_t s,
                           bool bitmap_ready = false, int32_t* zero_ptr = nullptr,
                           int zero_n = 0);
// T from which launch_permute uses the bitmap kernels (below: one CTA, no bitmap).
// Measured on the Qwen3-30B-A3B-shaped decode at T = 256: the one-CTA kernel
// took 7.2 us in the layer, the bitmap path (top-k writes the bitmap, then
// scan and scatter) ~4 us at T = 1024.
constexpr int kPermuteBitmapMinT = 129;
// also zeroes zero_ptr[0, zero_n) (counters for the kernel that follows)
cudaError_t launch_gather_rows(const void* x, const int32_t* sorted_token,
                               const int32_t* offsets, int E_r, int T, int H, int n_cap,
                               void* x_perm, int32_t* status, int sm_count, cudaStream_t s,
                               int32_t* zero_ptr = nullptr, int zero_n = 0);

// ---- combine.cu
cudaError_t launch_combine(const void* y_perm, const void* y_shared, const int32_t* inv_row,
                           const float* topk_w, const int32_t* k_per_token, int T, int H,
                           int k_max, int n_rows, void* out, int32_t* status, cudaStream_t s);

// ---- gemm.cu
enum GemmEpi { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_F32 = 2 };

struct GemmArgs {
  int epi;                   // GemmEpi
  const void* a;             // bf16 [a_rows, K]
  long long a_rows;
  const void* b;             // bf16 [b_rows, K]
  long long b_rows;
  int K;                     // multiple of 64
  const int32_t* offsets;    // [n_groups + 1] device, or nullptr for one dense group
  int n_groups;
  int dense_rows;            // rows of the dense group (offsets == nullptr)
  int n_out;                 // output columns per group (SWIGLU: I; BF16: H; F32: E_r)
  int b_group_rows;          // B rows per group (SWIGLU: 2I; BF16: H; F32: 0)
  void* out;                 // SWIGLU/BF16: bf16, F32: fp32
  long long ld_out;          // elements
  long long out_rows;        // rows the output buffer holds (stores beyond are dropped)
  const float* bias;         // F32 only, nullable
  int bias_div;
  int32_t* status;
  uint32_t debug_flags;
  int sm_count;
  int max_rows_hint;         // upper bound of total rows (grid sizing)
  int bn_hint;               // EPI_F32: output columns per tile (64/128/256), 0 = all
  int k_splits;              // EPI_F32: K split S ways (S divides K / 64); partial sums of
  long long split_stride;    //   split s at out + s * split_stride, no bias; 0/1 = no split
  bool force_pair;           // grouped SWIGLU/BF16: use the CTA-pair kernel
  const void* gather_x;      // grouped SWIGLU, single-CTA kernel: A row r is
  const int32_t* gather_tok; //   gather_x[gather_tok[r]] (no permuted copy); nullptr: A
  int gather_rows;           //   rows of gather_x
};

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s);

// ---- gemm_pair.cu: the same grouped GEMM on CTA pairs (tcgen05 cta_group::2)
bool gemm_pair_supports(int epi, int n_out);
cudaError_t launch_gemm_pair(const GemmArgs& g, cudaStream_t s);

// ---- gemm_decode.cu
struct DecodeGemmArgs {
  bool gate_up;              // true: gate|up + SwiGLU; false: down
  const void* w;             // bf16 weights [w_rows, K]
  long long w_rows;
  const void* x;             // bf16 rows [x_rows, K] (x_perm or act)
  long long x_rows;
  int K;
  const int32_t* offsets;    // [n_groups + 1]
  int n_groups;
  int n_out;                 // gate|up: I_sub; down: H (multiple of 128)
  int w_group_rows;          // gate|up: 2 I_sub; down: H
  void* out;                 // bf16 [out_rows, n_out]
  long long out_rows;
  float* partial;            // fp32 [max_split][out_rows][2 n_out] (gate|up, max_split > 1)
  int32_t* split_word;
  int max_split;
  int32_t* status;
  uint32_t debug_flags;
  int sm_count;
  int chunk;                 // tokens per item: 64 (decode-sized units) or more (prefill)
};

cudaError_t launch_decode_gemm(const DecodeGemmArgs& a, cudaStream_t s);
bool decode_gemm_supports(int n_out, bool gate_up);

// ---- ffn_decode.cu: gate|up + SwiGLU + down of a decode-sized batch in one kernel
struct DecodeFfnArgs {
  const void* x_perm;        // bf16 [x_rows, H], permuted token rows
  long long x_rows;
  const void* w_gate_up;     // bf16 [E_r, 2 I, H]
  const void* w_down;        // bf16 [E_r, H, I]
  const int32_t* offsets;    // [n_groups + 1]
  int n_groups;
  int H;
  int I;
  void* act;                 // bf16 [rows, I] (scratch)
  void* y;                   // bf16 [rows, H]
  int chunk;                 // tokens per item: 64, or 16 when T <= 16
  int32_t* done;             // per token-chunk counters, zero before the launch
  int32_t* work;             // dynamic-schedule counter, zero before the launch
  int32_t* split_cnt;        // [kFfnPartSlots / 2] split arrivals, zero before the launch
  float* part;               // [kFfnPartSlots][chunk][128] fp32 (split gate|up partial sums)
  long long rows;
  int32_t* status;
  uint32_t debug_flags;
  int sm_count;
  const void* gather_x;      // non-null: gate|up items copy their token rows from
  const int32_t* gather_tok; //   gather_x[gather_tok[r]] (bf16 [gather_rows, H]) instead
  int gather_rows;           //   of reading x_perm
};

cudaError_t launch_decode_ffn(const DecodeFfnArgs& a, cudaStream_t s);
constexpr int kFfnPartSlots = 256;
bool decode_ffn_supports(int H, int I_sub);

// bf16 [rows, cols] row-major tensor map: box of 64 columns x box_rows rows,
// 128-byte swizzle, zero fill out of bounds.
bool make_tmap_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);
bool gemm_supports_f32_router(int E_r);
// Output columns per tile and K splits of the tensor-core router GEMM for T
// tokens: small batches take 64-column tiles, and K is split until about 128
// tiles exist (the split partial sums go to a workspace and the top-k kernel
// adds them in order).
void router_gemm_shape(int T, int H, int E_r, int* bn, int* splits);

}  // namespace moe
