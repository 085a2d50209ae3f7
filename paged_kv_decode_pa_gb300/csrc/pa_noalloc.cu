// pa_decode_noalloc: pa_decode with its scratch in a library-owned device
// array, for callers that cannot allocate device memory when they call (see
// include/pa.h). Nothing here allocates or frees memory itself; the array is
// set up by the CUDA runtime when this file's module is first used on a
// device (its first call there).
#include <mutex>

#include "pa_device.cuh"

namespace pa {
pa_status decode_check(const pa_cache* cache, const void* q, const void* out, const int32_t* tables, int32_t mbps,
                       const int32_t* lens, int32_t batch, int32_t q_heads, int32_t max_ctx, float scale,
                       const pa_options* opts);
size_t workspace_zero_prefix(int32_t batch, int32_t nq, int32_t q_heads, int32_t kv_heads,
                             int32_t max_ctx, int32_t split);
void record_cuda_error(cudaError_t e);
}  // namespace pa

namespace {

// The scratch array. In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

void* g_scratch_addr[pa::kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device with that device current. The lookup loads this module on the
// device, which is when the runtime places the array in device memory.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= pa::kMaxDevices) return cudaErrorInvalidDevice;
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
  // pa_decode's own argument checks come first, so a rejected call returns
  // what pa_decode would and touches nothing, not even the shared scratch.
  const pa_status st = pa::decode_check(cache, q, out, block_tables, max_blocks_per_seq, context_lens, batch,
                                        q_heads, max_context_len, scale, opts);
  if (st != PA_OK) return st;
  const size_t need = pa_workspace_size(batch, 1, q_heads, cache->kv_heads, cache->head_dim,
                                        max_context_len, opts);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  if (batch == 0) return PA_OK;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    pa::record_cuda_error(e);
    return PA_ERR_CUDA;
  }
  // The previous call's status word and counters must not leak into this one
  // (their extent does not depend on the split).
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
