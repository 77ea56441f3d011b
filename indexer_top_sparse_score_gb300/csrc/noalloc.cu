// smla_sparse_mla_prefill_noalloc: the prefill step for callers that cannot
// allocate device memory (no cudaMalloc of their own, no workspace to pass),
// e.g. a plugin that only receives input and output pointers from its host
// framework, or an engine whose device memory is entirely owned by a pool
// that outside code may not draw from. The scratch the prefill needs (status
// word + selected-index list) lives in a fixed array inside this library
// instead of a caller-provided workspace.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per GPU that loads the library
constexpr int kMaxDevices = 64;

// Device-resident scratch shared by every call on a device. In host code this
// name is only a stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first use on that device (which must be current): a host-side reference to
// g_prefill_scratch is not a device address.
int scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr) return SMLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return SMLA_OK;
}

}  // namespace

extern "C" int smla_sparse_mla_prefill_noalloc(const smla_paged_cache* cache, const int32_t* page_table,
                                               int32_t prefix_len, int32_t n_tokens, const void* q,
                                               int32_t n_heads, const void* q_idx, const float* w,
                                               int32_t h_idx, int32_t topk, float sm_scale, void* out,
                                               float* lse, void* stream) {
  if (prefix_len < 0 || n_tokens <= 0 || topk <= 0) return SMLA_ERR_INVALID_ARG;
  // status word + index list must fit; the optional f16 copy of a BF16 cache is
  // used only when it fits in what is left
  if (smla::prefill_min_workspace(n_tokens, topk) > kNoAllocScratchBytes) return SMLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SMLA_OK) return rc;
  // the prefill clears the status word itself and rewrites the whole index list
  return smla_sparse_mla_prefill(cache, page_table, prefix_len, n_tokens, q, n_heads, q_idx, w, h_idx, topk,
                                 sm_scale, out, lse, nullptr, scratch, kNoAllocScratchBytes, stream);
}

// The device-side error report of the calls above: their status word is the
// first word of the scratch array, which only this library can address.
extern "C" int smla_noalloc_read_status(void* stream, uint32_t* bits) {
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SMLA_OK) return rc;
  return smla_read_status(scratch, stream, bits);
}
