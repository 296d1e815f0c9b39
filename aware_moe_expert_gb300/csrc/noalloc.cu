// moe_permute_static: the permutation step with its scratch held in a
// file-scope device array instead of a caller-provided workspace.
//
// Who needs it: a caller that may not allocate device memory at the point
// where it routes tokens.  Typical cases are a serving loop that promised
// never to enter the allocator on its hot path (an allocation can
// synchronise the device or fail when memory is fragmented), and a plug-in
// that is handed device pointers for its inputs and outputs but has no way
// to own an extra buffer.  Such a caller still
// passes every input and output; only the scratch comes from here.
//
// The scratch is one array per device that loads this library, kept until
// the process exits.  Its device address is looked up once per device, on
// the first call made with that device current.  Every call shares the
// array, so two calls whose kernels overlap on the GPU (different streams,
// no ordering between them) race on it and must not be issued.  The array
// needs no clearing: each call writes every scratch word it later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

// Membership bitmap plus per-word prefix counts: 2 * E_r * ceil(T / 32) int32.
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_permute_scratch on the current device (host code cannot
// use the symbol itself: in host code it names a host-side stand-in).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" moe_status moe_permute_static(const moe_layer_desc* desc, const int32_t* topk_idx,
                                         const int32_t* k_per_token, int32_t* counts,
                                         int32_t* offsets, int32_t* sorted_token,
                                         int32_t* inv_row, int32_t* dev_status, void* stream) {
  // the same descriptor checks, with the same status, as moe_permute
  const moe_status v = moe::validate_desc(desc);
  if (v != MOE_OK) return v;
  if (!aligned4(counts) || !aligned4(offsets) || !aligned4(dev_status))
    return MOE_ERR_INVALID_ARGUMENT;
  if (desc->T > 0 && (!aligned4(topk_idx) || !aligned4(k_per_token) || !aligned4(sorted_token) ||
                      !aligned4(inv_row)))
    return MOE_ERR_INVALID_ARGUMENT;
  const int E_r = desc->n_experts * desc->n_sub;
  const size_t W = (static_cast<size_t>(desc->T) + 31) / 32;
  const size_t words = static_cast<size_t>(E_r) * W;
  if (2 * words * 4 > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t* bitmap = static_cast<uint32_t*>(base);
  int32_t* wprefix = reinterpret_cast<int32_t*>(bitmap + words);
  const cudaError_t e = moe::launch_permute(topk_idx, k_per_token, desc->T, desc->k_max, E_r,
                                            bitmap, wprefix, counts, offsets, sorted_token,
                                            inv_row, dev_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
