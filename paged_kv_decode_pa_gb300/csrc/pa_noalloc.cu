// pa_decode_noalloc: pa_decode with its scratch in a library-owned device
// array, for callers that cannot allocate device memory when they call (see
// include/pa.h). Nothing here allocates or frees memory.
#include <mutex>

#include "pa_device.cuh"

namespace pa {
size_t workspace_zero_prefix(int32_t batch, int32_t nq, int32_t q_heads, int32_t kv_heads,
                             int32_t max_ctx, int32_t split);
void record_cuda_error(cudaError_t e);
}  // namespace pa

namespace {

// The scratch array. In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_cache* cache, const void* q, void* out,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t batch, int32_t q_heads,
                                       int32_t max_context_len, float scale, const pa_options* opts,
                                       void* stream) {
  if (!cache) return PA_ERR_INVALID_ARG;
  const size_t need = pa_workspace_size(batch, 1, q_heads, cache->kv_heads, cache->head_dim,
                                        max_context_len, opts);
  if (need == 0) return cache->head_dim != pa::kHeadDim ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  if (batch == 0) return PA_OK;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    pa::record_cuda_error(e);
    return PA_ERR_CUDA;
  }
  // The previous call's status word and counters must not leak into this one.
  const int32_t split = (opts && opts->split_tokens > 0) ? opts->split_tokens : PA_DEFAULT_SPLIT_TOKENS;
  const size_t zero = pa::workspace_zero_prefix(batch, 1, q_heads, cache->kv_heads, max_context_len, split);
  e = cudaMemsetAsync(scratch, 0, zero, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    pa::record_cuda_error(e);
    return PA_ERR_CUDA;
  }
  return pa_decode(cache, q, out, block_tables, max_blocks_per_seq, context_lens, batch, q_heads,
                   max_context_len, scale, scratch, need, opts, stream);
}
