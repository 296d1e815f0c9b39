/*
 * moe.h - C ABI of libmoe.so: one k-aware Mixture-of-Experts layer forward
 * on an NVIDIA GB300 (sm_103a).
 *
 * The layer (MoE-Prism, arXiv 2510.19366, §III-B and §III-C1): every token t
 * carries its own routing budget k_t.  The router scores E_r = n_experts *
 * n_sub routing units (an expert's intermediate neurons split into n_sub equal
 * sub-experts, §III-B1 Eq. (3)); token t runs the k_t best units through a
 * SwiGLU FFN (§III-B1 Eq. (1)) and sums their outputs weighted by the gate
 * (§III-B2, expanded linear gate).
 *
 * Conventions for every call below
 *  - Tensor pointers are DEVICE memory owned by the caller; bf16 tensors are
 *    passed as const void*, row-major, contiguous, 16-byte aligned.  The
 *    library never allocates, frees, or synchronises inside these calls.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream) and returns a moe_status for errors
 *    the host can see (bad arguments, unsupported shapes, launch failures).
 *  - Errors the device finds (k_t out of range, non-finite logits, bad unit
 *    indices, a device wait that gave up) are written to `dev_status`, a
 *    caller-owned int32 in device memory that the caller zeroes; the first
 *    error wins.  Read it with moe_get_device_status (the only call that
 *    synchronises).
 *  - Kernels are launched with programmatic dependent launch: the first
 *    kernel of a call may start while the previous kernel on `stream`
 *    finishes.  It reads the layer's parameters (router_w, expert_bias)
 *    before it waits for that kernel and every other input after; so a
 *    parameter must not be written by a kernel on the same stream that is
 *    still running when the call starts (one that lets its dependents launch
 *    early).  Inputs written by the preceding kernel (x, k_per_token, ...)
 *    are always read after it has finished.
 *  - `workspace` is caller-owned device memory of at least
 *    moe_workspace_size(desc) bytes, 256-byte aligned.  Calls on the same
 *    workspace must not overlap in time.
 *  - Weight layout (routing unit u = e * n_sub + n):
 *      w_gate_up [E_r, 2*I_sub, H]  rows 0..I_sub-1 gate, I_sub..2*I_sub-1 up
 *                                   (out x in, as a linear layer)
 *      w_down    [E_r, H, I_sub]
 *      router_w  [E_r, H]
 *  - Supported shapes: H % 64 == 0, I_sub % 64 == 0, I_shared % 64 == 0,
 *    1 <= E_r <= 256, 1 <= k_max <= min(E_r, 32), T >= 0.  Anything else
 *    returns MOE_ERR_UNSUPPORTED_SHAPE; there is no fallback path.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1,  /* null / misaligned / inconsistent argument       */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above          */
  MOE_ERR_WORKSPACE = 3,         /* workspace pointer null or misaligned           */
  MOE_ERR_CUDA = 4,              /* a CUDA runtime/driver call or launch failed     */
  MOE_ERR_DEVICE_TIMEOUT = 5,    /* device: a bounded wait gave up                  */
  MOE_ERR_NONFINITE = 6,         /* device: a router logit is NaN or infinite       */
  MOE_ERR_K_RANGE = 7,           /* device: some k_t outside [1, k_max]             */
  MOE_ERR_BAD_INDEX = 8          /* device: unit index out of range or repeated     */
} moe_status;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_PREFILL = 1, MOE_PATH_DECODE = 2 } moe_path;

/* debug_flags bits (tests only; 0 in normal use) */
#define MOE_DEBUG_SKIP_FIRST_LOAD 1u /* the FFN producer skips its first load, so the
                                        consumer's bounded wait must give up and report
                                        MOE_ERR_DEVICE_TIMEOUT (about 2 s)            */
#define MOE_DEBUG_FORCE_PAIR 2u      /* grouped prefill-path GEMMs run on the CTA-pair
                                        kernel (tcgen05 cta_group::2), which the library
                                        otherwise keeps for dense GEMMs; same results */

typedef struct {
  int32_t T;          /* tokens                                                  */
  int32_t H;          /* hidden size                                             */
  int32_t n_experts;  /* original experts                                        */
  int32_t n_sub;      /* sub-experts per expert (MoE-Prism's N); E_r = n_experts*n_sub */
  int32_t I_sub;      /* intermediate size of one sub-expert (C / N)             */
  int32_t k_max;      /* upper bound of every k_t; sizes the [T, k_max] outputs   */
  moe_score_fn score; /* softmax over all units, or sigmoid                      */
  int32_t renorm;     /* 1: divide the selected units' scores by their sum        */
  float route_scale;  /* multiplies every gate weight                            */
  const float* expert_bias;       /* nullable fp32 [n_experts], added to the logits
                                     of the expert's n_sub units                  */
  int32_t I_shared;               /* 0: no shared expert                         */
  const void* w_shared_gate_up;   /* bf16 [2*I_shared, H] (gate rows, then up)   */
  const void* w_shared_down;      /* bf16 [H, I_shared]                          */
  moe_path path;                  /* reserved: AUTO/PREFILL/DECODE give the same
                                     result; the library picks launch shapes     */
  uint32_t debug_flags;           /* MOE_DEBUG_* bits, tests only                 */
} moe_layer_desc;

/* Bytes of workspace every call below needs for this desc (0 on a bad desc). */
size_t moe_workspace_size(const moe_layer_desc* desc);

/* Steps 1-3 of the layer: router logits, per-token top-k_t, gate weights.
 * MoE-Prism §III-B2 (expanded linear gate scores every sub-expert and takes
 * the top-k) with the per-request budget k_i of §III-C1.
 *   x            bf16 [T, H]            (ignored when logits_in is given)
 *   router_w     bf16 [E_r, H]          (ignored when logits_in is given)
 *   logits_in    nullable fp32 [T, E_r]: route these logits instead of x.router_w
 *   k_per_token  int32 [T], each in [1, k_max] (else MOE_ERR_K_RANGE on device;
 *                the offending row is clamped into [0, k_max])
 *   logits_out   nullable fp32 [T, E_r]: receives x.router_w^T + bias
 *   topk_idx     int32 [T, k_max]: selected units, best first; -1 after k_t.
 *                Order: logit descending, lower index first on ties, -0 == +0,
 *                NaN last (and MOE_ERR_NONFINITE).
 *   topk_w       fp32 [T, k_max]: gate weight of each selected unit, 0 after k_t.
 *                softmax: exp(L_u - max L) / sum over ALL units; sigmoid:
 *                1/(1+exp(-L_u)); renorm divides by the selected sum; then
 *                times route_scale.
 *   workspace    moe_workspace_size(desc) bytes; unused (may be null) when
 *                logits_in is given. */
moe_status moe_route(const moe_layer_desc* desc, const void* x, const void* router_w,
                     const float* logits_in, const int32_t* k_per_token, float* logits_out,
                     int32_t* topk_idx, float* topk_w, int32_t* dev_status, void* workspace,
                     void* stream);

/* Step 4: group the assignments by routing unit (MoE-Prism §II-D: grouped
 * GEMMs need one unit's rows contiguous).  Deterministic: unit ascending,
 * token ascending inside a unit.
 *   topk_idx, k_per_token  as produced by moe_route
 *   counts        int32 [E_r]       assignments per unit
 *   offsets       int32 [E_r + 1]   exclusive prefix sum of counts
 *   sorted_token  int32 [T * k_max] token of each permuted row (first offsets[E_r] valid)
 *   inv_row       int32 [T, k_max]  permuted row of assignment (t, j); -1 after k_t
 * A unit index outside [0, E_r) or repeated within a token -> MOE_ERR_BAD_INDEX. */
moe_status moe_permute(const moe_layer_desc* desc, const int32_t* topk_idx,
                       const int32_t* k_per_token, int32_t* counts, int32_t* offsets,
                       int32_t* sorted_token, int32_t* inv_row, int32_t* dev_status,
                       void* workspace, void* stream);

/* Step 5a: for every unit u, act[r] = SiLU(x_t Wg_u^T) * (x_t Wu_u^T) for the
 * permuted rows r of u (t = sorted_token[r]).  MoE-Prism §III-B1 Eq. (1).
 *   act  bf16 [T * k_max, I_sub]; rows >= offsets[E_r] are left untouched.
 * Accumulation in fp32 on the tensor cores; act is rounded to bf16. */
moe_status moe_gate_up(const moe_layer_desc* desc, const void* x, const int32_t* sorted_token,
                       const int32_t* offsets, const void* w_gate_up, void* act,
                       int32_t* dev_status, void* workspace, void* stream);

/* Step 5b: y_perm[r] = act[r] Wd_u^T for the permuted rows r of unit u
 * (MoE-Prism §III-B1 Eq. (1), X' = A Wdown).
 *   y_perm  bf16 [T * k_max, H]; rows >= offsets[E_r] untouched. */
moe_status moe_down(const moe_layer_desc* desc, const void* act, const int32_t* offsets,
                    const void* w_down, void* y_perm, int32_t* dev_status, void* workspace,
                    void* stream);

/* Steps 5a + 5b with act kept in the workspace. */
moe_status moe_grouped_ffn(const moe_layer_desc* desc, const void* x,
                           const int32_t* sorted_token, const int32_t* offsets,
                           const void* w_gate_up, const void* w_down, void* y_perm,
                           int32_t* dev_status, void* workspace, void* stream);

/* The always-on shared expert of every token (weight 1, not counted in k):
 * y_shared = SwiGLU_shared(x), bf16 [T, H].  Requires desc->I_shared > 0. */
moe_status moe_shared_ffn(const moe_layer_desc* desc, const void* x, void* y_shared,
                          int32_t* dev_status, void* workspace, void* stream);

/* Step 6: out_t = sum_{j < k_t} topk_w[t,j] * y_perm[inv_row[t,j]] (+ y_shared[t]),
 * accumulated in fp32 in j order, rounded once to bf16 [T, H].
 * MoE-Prism §III-B2: the routed output is sum_j w_j FFN_j(x). */
moe_status moe_combine(const moe_layer_desc* desc, const void* y_perm, const void* y_shared,
                       const int32_t* inv_row, const float* topk_w, const int32_t* k_per_token,
                       void* out, int32_t* dev_status, void* stream);

/* The whole layer: route -> permute -> [shared FFN] -> grouped FFN -> combine,
 * every intermediate in the workspace.  out bf16 [T, H]. */
moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, const void* router_w,
                             const void* w_gate_up, const void* w_down,
                             const int32_t* k_per_token, void* out, int32_t* dev_status,
                             void* workspace, void* stream);

/* moe_layer_forward for callers whose token-side tensors live in host memory
 * (a serving loop that receives activations from the host and returns the
 * layer's output there).  On `stream`: x_host -> x_dev (bf16 [T, H]) and
 * k_host -> k_dev (int32 [T]) host-to-device copies, moe_layer_forward on the
 * device copies, then out_dev -> out_host (bf16 [T, H]).  x_dev, k_dev and
 * out_dev are caller-owned device buffers of those sizes; the weights, the
 * workspace and dev_status are as for moe_layer_forward.  Nothing is
 * allocated.  With pinned (page-locked) host buffers the whole call is
 * asynchronous; pageable ones make the copies synchronise with the host.
 * Host-side argument errors are reported before any copy is enqueued; a
 * failed copy returns MOE_ERR_CUDA.  (A host-memory convenience around the
 * layer of MoE-Prism §III-B; the paper's layer is moe_layer_forward.) */
moe_status moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host,
                                  const int32_t* k_host, void* out_host, void* x_dev,
                                  int32_t* k_dev, void* out_dev, const void* router_w,
                                  const void* w_gate_up, const void* w_down,
                                  int32_t* dev_status, void* workspace, void* stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory where they route (inside a serving loop that must stay out of the
 * allocator, or in a plug-in that owns no buffers of its own).  The published method has no
 * counterpart to this call: it only changes where the scratch lives.
 *   Arguments and results are those of moe_permute, minus `workspace`.
 *   Scratch: a 1 MiB array in device memory that every GPU loading this
 *   library keeps until exit; 2 * E_r * ceil(T/32) * 4 bytes must fit, else
 *   MOE_ERR_UNSUPPORTED_SHAPE (e.g. E_r = 256 allows T <= 16384).
 *   The first call on a device looks up the array's device address (a
 *   runtime call, made once per device).
 *   All calls share the array: calls whose kernels may overlap on the GPU
 *   race and must not be issued.  Nothing in it needs clearing between calls.
 *   Allocates nothing (no cudaMalloc, cudaFree or allocating library call). */
moe_status moe_permute_static(const moe_layer_desc* desc, const int32_t* topk_idx,
                              const int32_t* k_per_token, int32_t* counts, int32_t* offsets,
                              int32_t* sorted_token, int32_t* inv_row, int32_t* dev_status,
                              void* stream);

/* ---------------------------------------------------------------------------
 * Decode expert-pool folding ("ExFold: Unified Expert Folding for Training-Free
 * MoE Prefill-Decode Acceleration", arXiv 2608.24938, "Phase-Specific Routing
 * and Folding").  Decode time follows the distinct units a batch activates;
 * folding keeps a pool of D units and remaps every other route to its pool
 * target tau(u) = argmin_{p in pool} L[u, p] (lower index on ties), its weight
 * scaled by S[u, tau(u)].  Routes of a token that reach one target are merged
 * (fp32 sum in slot order) at the position of their first occurrence, so each
 * target runs once; the token's budget becomes the number of targets.
 * Dynamic pool: the D units with the largest score h_u * sum of their routed
 * weights over the batch (fp32, tokens in blocks of 64 added in order; score
 * descending, lower index on ties).  Static pool: the caller's D units.
 */
typedef struct {
  int32_t D;                  /* pool size, 1..E_r                                      */
  const int32_t* pool;        /* nullable device int32 [D]: a static pool of distinct
                                 units (else MOE_ERR_BAD_INDEX); null: dynamic pool      */
  const float* unit_scale;    /* nullable device fp32 [E_r]: h_u of the dynamic score
                                 (null: 1)                                               */
  const float* S;             /* device fp32 [E_r, E_r]: S[u, v] scales a route folded
                                 from unit u into unit v (calibration data)              */
  const float* L;             /* device fp32 [E_r, E_r]: loss of folding u into v        */
} moe_fold_desc;

/* Rewrites routing (topk_idx, topk_w, k_per_token: as from moe_route) into
 *   topk_idx_out int32 [T, k_max]  targets, first-occurrence order, -1 after k_out[t]
 *   topk_w_out   fp32 [T, k_max]   merged weights, 0 after k_out[t]
 *   k_out        int32 [T]         the new budgets (<= the old ones)
 *   pool_out     nullable int32 [D]: the pool, ascending.
 * The outputs feed moe_permute / moe_combine like moe_route's.  Workspace:
 * moe_workspace_size(desc) bytes. */
moe_status moe_fold_decode(const moe_layer_desc* desc, const moe_fold_desc* fold,
                           const int32_t* topk_idx, const float* topk_w,
                           const int32_t* k_per_token, int32_t* topk_idx_out,
                           float* topk_w_out, int32_t* k_out, int32_t* pool_out,
                           int32_t* dev_status, void* workspace, void* stream);

/* The whole layer with folding: route -> fold -> permute -> [shared FFN] ->
 * grouped FFN -> combine.  out bf16 [T, H].  Workspace: moe_workspace_size. */
moe_status moe_layer_forward_fold(const moe_layer_desc* desc, const moe_fold_desc* fold,
                                  const void* x, const void* router_w, const void* w_gate_up,
                                  const void* w_down, const int32_t* k_per_token, void* out,
                                  int32_t* dev_status, void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * Path-composed execution with source-grouped reuse ("PCoMoE: Shifting MoE
 * Inference from Monolithic Expert Selection to Fine-Grained Path
 * Composition", arXiv 2609.01024, "Source-Grouped Compute Reuse", Fig. 8).
 * A SwiGLU unit splits into an expansion U_u(h) = SiLU(h Wg_u) * (h Wu_u)
 * and a projection D_u(z) = z Wd_u; a path (i, j) is D_j(U_i(h)), and
 *     out_t = sum_{j < n_paths[t]} beta[t,j] * D_{tgt[t,j]}(U_{src[t,j]}(x_t))
 *             (+ the shared expert, weight 1, when desc->I_shared > 0),
 * with U_i evaluated once per distinct source of a token and D_j once per
 * distinct target: D is linear, so the paths of a token into one target j
 * are projected together, D_j(sum_i beta_ij U_i(x_t)) (the weighted sum of
 * their bf16 expansion rows formed in fp32, in slot order, rounded to bf16).
 * Paths are listed in slot order; diagonal paths i == j are the plain layer.
 *   src_idx, tgt_idx  int32 [T, k_max]: units of each path's expansion and
 *                     projection; a token's sources and targets may repeat
 *                     (a repeated (i, j) pair adds its weights)
 *   beta              fp32 [T, k_max]: path weights
 *   n_paths           int32 [T], each in [1, k_max]
 *   out               bf16 [T, H]
 * Unit indices outside [0, E_r) give MOE_ERR_BAD_INDEX.  Path selection (a
 * learned compatibility bias) is the caller's.  Workspace:
 * moe_workspace_size(desc) bytes.  Requires I_sub % 8 == 0. */
moe_status moe_layer_forward_paths(const moe_layer_desc* desc, const void* x,
                                   const void* w_gate_up, const void* w_down,
                                   const int32_t* src_idx, const int32_t* tgt_idx,
                                   const float* beta, const int32_t* n_paths, void* out,
                                   int32_t* dev_status, void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * Quality-tiered batching (host only; MoE-Prism §III-C2 "Temporal Separation
 * via Quality-Tiered Batching", Eq. (5)).  For dispatches that run a whole
 * batch at one budget (the batch maximum), requests are grouped by budget:
 * the queue is sorted by (k, arrival), batches are filled in FIFO order up to
 * M prompt tokens tier by tier, and a residual batch (n_cur tokens at budget
 * k) is promoted to the next tier's budget k_next and merged with the n_next
 * tokens of that tier's leading requests that still fit iff
 *     (n_cur + n_next) / T(n_cur + n_next, k_next) >= n_cur / T(n_cur, k),
 * else it is dispatched at k.  T(n, k) is a table profiled on the deployment
 * GPU at token and budget buckets, interpolated between them.
 */
typedef struct {
  double arrival;     /* arrival time (any unit); FIFO order inside a tier        */
  int32_t n_tokens;   /* prompt tokens, >= 1                                      */
  int32_t k;          /* requested routing budget                                 */
} moe_tier_request;

typedef struct {
  int32_t n_count;            /* token buckets, >= 1                              */
  const int32_t* n_points;    /* host, strictly increasing                        */
  int32_t k_count;            /* budget buckets, >= 1                             */
  const int32_t* k_points;    /* host, strictly increasing                        */
  const double* t_us;         /* host [k_count][n_count]: layer time at each bucket */
} moe_cost_table;

/* T(n, k): linear in n between buckets (end segments extended linearly; one
 * bucket scales proportionally), linear in k between buckets, k clamped to
 * the profiled range.  Returns -1 for a malformed table.  Host only. */
double moe_cost_lookup(const moe_cost_table* table, double n, double k);

/* Schedules n_req host requests under token budget M.  Writes, in dispatch
 * order, batch_of[i] (batch index of request i), and when non-null batch_k[b]
 * (the budget batch b runs at) and batch_tokens[b].  Returns the number of
 * batches, -1 on bad arguments (M < 1, a request with < 1 token, a malformed
 * table), -2 if more than max_batches would be needed.  A request larger than
 * M forms a batch of its own.  Host only: no device memory, no stream. */
int32_t moe_tier_schedule(const moe_tier_request* reqs, int32_t n_req, int32_t M,
                          const moe_cost_table* table, int32_t* batch_of, int32_t* batch_k,
                          int32_t* batch_tokens, int32_t max_batches);

/* ---------------------------------------------------------------------------
 * Training-free proxy router (MoE-Prism §III-B2, "Training-Free Proxy Gating",
 * Fig. 7 left).  The original router scores the n_experts original experts and
 * keeps its native m of them per token (selection, normalisation and scaling
 * as moe_route, with one unit per expert); for each kept expert j and each of
 * its n_sub sub-experts, the proxy score is
 *     s_n = (1/r) sum_{c in G_n} |SiLU(x . Wg[c]) * (x . Wu[c])|
 * over the sub-expert's r gate neurons G_n; the kappa_j best sub-experts of
 * expert j (kappa = row k_t of the allocation table) are routed, each with the
 * expert's weight w_j (no second softmax).  Ties: lower index first.
 */
typedef struct {
  int32_t m;                   /* original experts kept per token, 1..min(n_experts, 32) */
  int32_t r;                   /* gate neurons per sub-expert, 1..I_sub                   */
  const void* router_w_expert; /* bf16 [n_experts, H]: the original router                */
  const void* proxy_w;         /* bf16 [E_r * 2 * r, H], from moe_pack_proxy_rows         */
  const int32_t* kappa;        /* device int32 [k_max + 1, m]: row k allocates a budget k;
                                  a row with entries outside [0, n_sub] or not summing to
                                  k gives MOE_ERR_K_RANGE and no units for that token     */
} moe_cg_router;
/* Requirements beyond moe_layer_desc's: n_sub <= 32, k_max <= m * n_sub,
 * m * n_sub * r <= 2048 (else MOE_ERR_UNSUPPORTED_SHAPE). */

/* Workspace bytes for moe_route_cg and moe_layer_forward_cg (0 on a bad desc).
 * It includes moe_workspace_size(desc) (at its start). */
size_t moe_cg_workspace_size(const moe_layer_desc* desc, const moe_cg_router* cg);

/* Model set-up: gather the gate-neuron rows of every unit into
 *   proxy_w bf16 [E_r * 2 * r, H]: row (u * r + i) * 2 = w_gate_up[u] gate row
 *   gate_neurons[u * r + i], the next row the matching up row.
 *   gate_neurons  device int32 [E_r, r], indices local to the unit (0..I_sub-1);
 *                 an index outside that range -> MOE_ERR_BAD_INDEX, zero rows. */
moe_status moe_pack_proxy_rows(const moe_layer_desc* desc, int32_t r, const void* w_gate_up,
                               const int32_t* gate_neurons, void* proxy_w, int32_t* dev_status,
                               void* stream);

/* Routing with the proxy router.  Outputs as moe_route (topk_idx [T, k_max],
 * best-ranked expert first, inside an expert by proxy score; topk_w [T, k_max]),
 * plus, when non-null,
 *   expert_logits_out  fp32 [T, n_experts]: the original router's logits + bias
 *   proxy_out          fp32 [T, m, n_sub]: the proxy scores the selection used.
 * Workspace: moe_cg_workspace_size bytes. */
moe_status moe_route_cg(const moe_layer_desc* desc, const moe_cg_router* cg, const void* x,
                        const int32_t* k_per_token, float* expert_logits_out, float* proxy_out,
                        int32_t* topk_idx, float* topk_w, int32_t* dev_status, void* workspace,
                        void* stream);

/* The whole layer with the proxy router: route_cg -> permute -> [shared FFN] ->
 * grouped FFN -> combine.  out bf16 [T, H].  Workspace: moe_cg_workspace_size. */
moe_status moe_layer_forward_cg(const moe_layer_desc* desc, const moe_cg_router* cg,
                                const void* x, const void* w_gate_up, const void* w_down,
                                const int32_t* k_per_token, void* out, int32_t* dev_status,
                                void* workspace, void* stream);

/* Synchronises `stream`, then returns the code stored in *dev_status
 * (MOE_OK if zero), or MOE_ERR_CUDA if the synchronisation itself failed. */
moe_status moe_get_device_status(const int32_t* dev_status, void* stream);

/* Static string naming a status code. */
const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
