// Decode attention for callers that cannot allocate device memory.
//
// kvarn_decode_attention needs a caller-provided workspace for its split partials.  Some
// callers have no way to provide one: plugins inside an inference engine that plans and
// owns all device memory ahead of time, code that must not call cudaMalloc on the decode
// path (it can synchronise the whole device and stall other streams), and embedders with
// no device allocator at hand.  This entry point keeps the partials in a fixed buffer that
// lives inside the library instead.
#include <mutex>

#include "common.cuh"
#include "params.cuh"

namespace {

constexpr size_t kScratchBytes = KVARN_DECODE_NOALLOC_SCRATCH_BYTES;

// The split partials of kvarn_decode_attention_noalloc.  Every GPU that loads the library
// holds this buffer until the process exits.  In host code the name is only a host-side
// stand-in for the symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_lock;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device, looked up once per device and
// kept for the life of the process (cudaDeviceReset would unload the module and leave the kept
// address stale; the header tells callers not to reset a device they use this entry point on).
int scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVARN_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_scratch_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return KVARN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return KVARN_OK;
}

}  // namespace

extern "C" int kvarn_decode_attention_noalloc(const kvarn_desc* desc, int batch, int num_q_heads,
                                              const void* q, const void* page_pool,
                                              int64_t num_pool_pages, const int32_t* block_table,
                                              int max_pages, const int32_t* seq_lens,
                                              const void* partial_k, const void* partial_v,
                                              float softmax_scale, void* out, int32_t* dev_status,
                                              void* stream) {
  // The argument checks of kvarn_decode_attention come first, so that a bad argument gives the
  // same status as there and an empty batch returns without touching the GPU.
  int st = kvarn::decode_args_check(desc, batch, num_q_heads, q, page_pool, num_pool_pages,
                                    block_table, max_pages, seq_lens, partial_k, partial_v,
                                    softmax_scale, out);
  if (st == kvarn::kDecodeNothingToDo) return KVARN_OK;
  if (st != KVARN_OK) return st;
  if (kvarn_decode_workspace_bytes(desc, batch, num_q_heads, max_pages) > kScratchBytes)
    return KVARN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != KVARN_OK) return st;
  // Same kernels as kvarn_decode_attention.  No part of the buffer has to start at zero: every
  // partial the merge reads is written earlier in the same call.
  return kvarn_decode_attention(desc, batch, num_q_heads, q, page_pool, num_pool_pages,
                                block_table, max_pages, seq_lens, partial_k, partial_v,
                                softmax_scale, out, scratch, kScratchBytes, dev_status, stream);
}
