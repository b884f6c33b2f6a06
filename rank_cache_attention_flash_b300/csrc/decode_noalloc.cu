// lrkv_attn_decode_noalloc: the decode entry point for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine at the point
// where they run decode: a host runtime whose memory is carved out once at
// start-up and must not grow, an embedding that forbids allocation on its
// serving path, or code running where the caching allocator of a framework is
// not available. They still own their inputs and outputs, but cannot provide
// the split-partial workspace that lrkv_attn_decode asks for. This file keeps
// that workspace in a fixed-size array in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds LRKV_NOALLOC_SCRATCH_BYTES of it until the process exits. Host
// code cannot use the variable's name as a device address, so on the first
// call on each device (with that device current) the address is resolved
// once with cudaGetSymbolAddress and cached per device. The cache is never
// invalidated: a process that resets a device (cudaDeviceReset) must not call
// this entry point on that device afterwards.
#include <mutex>

#include "lrkv.h"
#include "lrkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[LRKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (resolved on the
// first call on that device, then cached).
lrkv_status scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LRKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LRKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return LRKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return LRKV_OK;
}

}  // namespace

extern "C" lrkv_status lrkv_attn_decode_noalloc(
    const lrkv_config* cfg, const void* q, int32_t num_queries, const int32_t* ctx_q_start,
    int32_t num_ctx, const int32_t* adapter_ids, const int32_t* block_tables, int32_t max_blocks,
    const int32_t* ctx_lens, int32_t max_ctx_len, int32_t max_q_per_ctx, const void* base_pool,
    const void* lr_pool, int64_t num_blocks, const void* B_K, const void* B_V, int32_t n_adapters,
    float scale, void* out, int32_t* dev_status, lrkv_stream_t stream) {
  // Sizes that need more scratch than the fixed array holds are refused
  // before anything else touches the device.
  const size_t need =
      lrkv_decode_workspace_bytes(cfg, num_queries, num_ctx, max_ctx_len, max_q_per_ctx);
  if (need > static_cast<size_t>(LRKV_NOALLOC_SCRATCH_BYTES)) return LRKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  const lrkv_status st = scratch_on_current_device(&scratch);
  if (st != LRKV_OK) return st;
  // The split partials are written before they are read, so nothing in the
  // array has to start at zero; the previous call's contents are harmless.
  return lrkv_attn_decode(cfg, q, num_queries, ctx_q_start, num_ctx, adapter_ids, block_tables,
                          max_blocks, ctx_lens, max_ctx_len, max_q_per_ctx, base_pool, lr_pool,
                          num_blocks, B_K, B_V, n_adapters, scale, out, scratch,
                          static_cast<size_t>(LRKV_NOALLOC_SCRATCH_BYTES), dev_status, stream);
}
