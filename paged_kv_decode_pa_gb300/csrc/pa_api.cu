// Host side of libpa: argument checks, workspace layout, TMA descriptors,
// launches, plus the cache-write and validation kernels. See include/pa.h for
// the contract of every entry point.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_device.cuh"

namespace pa {
cudaError_t launch_attn_mma(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                            dim3 grid, cudaStream_t stream);
cudaError_t launch_attn_simt(const AttnParams& p, bool bf16, dim3 grid, cudaStream_t stream);
cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream);
struct Q8Maps {
  CUtensorMap k, v, ks, vs;
};
cudaError_t launch_attn_q8(const Q8Maps& maps, const AttnParams& p, dim3 grid, bool after_append,
                           cudaStream_t stream);
cudaError_t launch_cache_write_q8(const pa_cache* c, const void* k_new, const void* v_new,
                                  const int32_t* slots, int32_t n, uint32_t* status, cudaStream_t stream);
cudaError_t launch_attn_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, dim3 grid,
                                cudaStream_t stream);
cudaError_t launch_attn_prefill_tc(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                                   const AttnParams& p, cudaStream_t stream);
constexpr int kPrefillRows = 128;  // query rows per prefill CTA
}  // namespace pa

namespace {

using namespace pa;

thread_local int g_last_cuda_error = 0;

pa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

size_t elem_size(int32_t dtype) { return dtype == PA_DTYPE_F32 ? 4 : dtype == PA_DTYPE_INT8 ? 1 : 2; }

pa_status check_cache(const pa_cache* c) {
  if (!c || !c->k || !c->v) return PA_ERR_INVALID_ARG;
  if (c->dtype != PA_DTYPE_F32 && c->dtype != PA_DTYPE_BF16 && c->dtype != PA_DTYPE_INT8)
    return PA_ERR_UNSUPPORTED;
  if (c->dtype == PA_DTYPE_INT8 &&
      (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) || !aligned16(c->v_scale)))
    return PA_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (c->kv_heads <= 0 || c->num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (c->kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  // Slot and TMA row coordinates are int32: num_blocks * 16 must fit.
  if (int64_t(c->num_blocks) * kBlockSize > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!aligned16(c->k) || !aligned16(c->v)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// Split for sequences of up to PA_LONG_CONTEXT_TOKENS under the default
// rule, or the caller's split. Without a dtype (workspace sizing) the finer
// of the two defaults is taken, an upper bound on splits.
int32_t split_of(const pa_options* o, int32_t dtype) {
  if (o && o->split_tokens > 0) return o->split_tokens;
  return dtype == PA_DTYPE_INT8 ? PA_DEFAULT_SPLIT_TOKENS_INT8 : PA_DEFAULT_SPLIT_TOKENS;
}

uint32_t wait_limit_of(const pa_options* o) {
  return (o && o->wait_limit_ns > 0) ? o->wait_limit_ns : PA_DEFAULT_WAIT_LIMIT_NS;
}

// Split for sequences longer than PA_LONG_CONTEXT_TOKENS under the default
// rule (0: an explicit split applies to every length). Without a dtype
// (workspace sizing) the finer of the two is taken, an upper bound on splits.
int32_t split_long_of(const pa_options* o, int32_t dtype) {
  if (o && o->split_tokens > 0) return 0;
  if (dtype == PA_DTYPE_INT8 || dtype < 0) return PA_DEFAULT_SPLIT_LONG_INT8;
  return PA_DEFAULT_SPLIT_LONG;
}

// Most splits any sequence of up to max_ctx tokens can have: the split
// count grows with the length under either rule.
int64_t max_splits_of(int32_t max_ctx, int32_t split, int32_t split_long) {
  const int32_t s = (split_long > 0 && max_ctx > PA_LONG_CONTEXT_TOKENS) ? split_long : split;
  return std::max<int64_t>(1, (int64_t(max_ctx) + s - 1) / s);
}

// Workspace: [status word | counters | lse partials | o partials], each
// region 256-byte aligned. Row groups are counted for the 8-row CUDA-core
// kernel, an upper bound for the 16-row tensor-core kernel.
struct WsLayout {
  size_t counters, lse, o, total;
  int64_t units;
  int32_t max_splits;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

bool ws_layout(int32_t batch, int32_t nq, int32_t q_heads, int32_t kv_heads, int32_t max_ctx,
               int32_t split, int32_t split_long, WsLayout* out) {
  if (batch < 0 || nq < 1 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads) return false;
  if (max_ctx < 0 || split <= 0) return false;
  const int64_t rows = int64_t(nq) * (q_heads / kv_heads);
  const int64_t groups = (rows + 7) / 8;
  const int64_t splits = max_splits_of(max_ctx, split, split_long);
  const int64_t units = int64_t(batch) * kv_heads * groups;
  WsLayout L;
  L.max_splits = static_cast<int32_t>(splits);
  L.units = units;
  L.counters = 256;
  L.lse = L.counters + round256(size_t(units) * 4);
  L.o = L.lse + round256(size_t(units * splits * kRowSlots) * 4);
  L.total = L.o + round256(size_t(units * splits * kRowSlots) * kHeadDim * 4);
  *out = L;
  return true;
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// A 3-D view [kv_heads][num_blocks * 16][128] of one bf16 pool; boxes of
// 16 token rows x 64 dims, 128-byte swizzled, zeros outside the tensor.
bool make_pool_map(CUtensorMap* map, void* pool, int32_t kv_heads, int32_t num_blocks) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(num_blocks) * kBlockSize,
                        cuuint64_t(kv_heads)};
  cuuint64_t strides[2] = {cuuint64_t(kHeadDim) * 2, cuuint64_t(num_blocks) * kBlockSize * kHeadDim * 2};
  cuuint32_t box[3] = {64, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same pool as a 4-D view [kv_heads][2 halves][num_blocks * 16][64]
// whose half dimension (128 bytes apart) comes after the rows (256 bytes
// apart): one box of 64 dims x 16 rows x 2 halves lands a whole 16-row tile
// as [half][row][64], the layout two 3-D boxes give.
bool make_pool_map4(CUtensorMap* map, void* pool, int32_t kv_heads, int32_t num_blocks) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, cuuint64_t(num_blocks) * kBlockSize, 2, cuuint64_t(kv_heads)};
  cuuint64_t strides[3] = {cuuint64_t(kHeadDim) * 2, 128, cuuint64_t(num_blocks) * kBlockSize * kHeadDim * 2};
  cuuint32_t box[4] = {64, 16, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query rows of a prefill, [total][q_heads][128] bf16, in boxes of 64 dims x
// `group` heads x `tokens` tokens (128-byte swizzle): a box lands as the rows
// r = token * group + head of one KV head's group. Outside the tensor it
// reads zeros.
bool make_query_map(CUtensorMap* map, const void* q, int32_t total, int32_t q_heads, int32_t group,
                    int32_t tokens) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(q_heads), cuuint64_t(total)};
  cuuint64_t strides[2] = {cuuint64_t(kHeadDim) * 2, cuuint64_t(q_heads) * kHeadDim * 2};
  cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(tokens)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The int8 pool's four views: bytes [kv_heads][num_blocks * 16][128] in
// 16-row x 128-byte boxes (128-byte swizzle), K scales [kv_heads][num_blocks]
// [128] and V scales [kv_heads][num_blocks][16] fp32 in one-block boxes.
// Outside the tensor every view reads zeros.
bool make_q8_maps(Q8Maps* m, const pa_cache* c) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t nb = cuuint64_t(c->num_blocks), hkv = cuuint64_t(c->kv_heads);
  const cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t cdims[3] = {cuuint64_t(kHeadDim), nb * kBlockSize, hkv};
  cuuint64_t cstr[2] = {cuuint64_t(kHeadDim), nb * kBlockSize * kHeadDim};
  cuuint32_t cbox[3] = {cuuint32_t(kHeadDim), cuuint32_t(kBlockSize), 1};
  cuuint64_t kdims[3] = {cuuint64_t(kHeadDim), nb, hkv};
  cuuint64_t kstr[2] = {cuuint64_t(kHeadDim) * 4, nb * kHeadDim * 4};
  cuuint32_t kbox[3] = {cuuint32_t(kHeadDim), 1, 1};
  cuuint64_t vdims[3] = {cuuint64_t(kBlockSize), nb, hkv};
  cuuint64_t vstr[2] = {cuuint64_t(kBlockSize) * 4, nb * kBlockSize * 4};
  cuuint32_t vbox[3] = {cuuint32_t(kBlockSize), 1, 1};
  const auto none = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE;
  return enc(&m->k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c->k, cdims, cstr, cbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             none) == CUDA_SUCCESS &&
         enc(&m->v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c->v, cdims, cstr, cbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             none) == CUDA_SUCCESS &&
         enc(&m->ks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, c->k_scale, kdims, kstr, kbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             none) == CUDA_SUCCESS &&
         enc(&m->vs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, c->v_scale, vdims, vstr, vbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             none) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Cache write: one thread per 16-byte chunk of each new K or V row.

__global__ void cache_write_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc,
                                   const uint4* __restrict__ kn, const uint4* __restrict__ vn,
                                   const int32_t* __restrict__ slots, int32_t n, int32_t kv_heads,
                                   int32_t num_blocks, int32_t chunks_per_row) {
  const int64_t total = int64_t(n) * kv_heads * 2 * chunks_per_row;
  const int64_t num_slots = int64_t(num_blocks) * kBlockSize;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(idx % chunks_per_row);
    int64_t rest = idx / chunks_per_row;
    const int is_v = int(rest & 1);
    rest >>= 1;
    const int h = int(rest % kv_heads);
    const int64_t i = rest / kv_heads;
    const int64_t slot = __ldg(slots + i);
    if (slot < 0 || slot >= num_slots) continue;
    const int64_t src = (i * kv_heads + h) * chunks_per_row + c;
    const int64_t dst = ((int64_t(h) * num_blocks + slot / kBlockSize) * kBlockSize + slot % kBlockSize) *
                            chunks_per_row + c;
    if (is_v)
      vc[dst] = __ldg(vn + src);
    else
      kc[dst] = __ldg(kn + src);
  }
}

// Validation: one CTA per sequence; counts into a 4-word report.
__global__ void validate_kernel(const int32_t* __restrict__ tables, int32_t mbps,
                                const int32_t* __restrict__ lens, int32_t max_ctx, int32_t num_blocks,
                                const int32_t* __restrict__ slots, int32_t nq, uint32_t* report) {
  const int b = blockIdx.x;
  int L = lens[b];
  const int cap = min(max_ctx, mbps * kBlockSize);
  const bool bad_len = L < 0 || L > cap || (nq > 1 && L < nq);
  if (threadIdx.x == 0 && bad_len) {
    atomicAdd(report + 1, 1u);
    atomicOr(report, PA_FLAG_BAD_LENGTH);
  }
  L = max(0, min(L, cap));
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
    const int id = tables[int64_t(b) * mbps + j];
    if (id < 0 || id >= num_blocks) {
      atomicAdd(report + 2, 1u);
      atomicOr(report, PA_FLAG_BAD_BLOCK);
    }
  }
  if (!slots) return;
  for (int i = threadIdx.x; i < nq; i += blockDim.x) {
    const int s = slots[int64_t(b) * nq + i];
    const int pos = L - nq + i;
    int expect = -1;
    if (pos >= 0) {
      const int id = tables[int64_t(b) * mbps + pos / kBlockSize];
      expect = (id >= 0 && id < num_blocks) ? id * kBlockSize + pos % kBlockSize : -2;
    }
    const bool in_range = s >= -1 && int64_t(s) < int64_t(num_blocks) * kBlockSize;
    if (!in_range || s != expect) {
      atomicAdd(report + 3, 1u);
      atomicOr(report, PA_FLAG_BAD_SLOT);
    }
  }
}

// Host-side checks of a decode / verify call, everything but the workspace.
// On PA_OK, *kernel_out is the kernel the call runs (AUTO resolved).
pa_status attend_check(const pa_cache* cache, const void* q, const void* out, const void* k_new,
                       const void* v_new, const int32_t* slots, int32_t nq, const int32_t* tables,
                       int32_t mbps, const int32_t* lens, int32_t batch, int32_t q_heads, int32_t max_ctx,
                       float scale, const pa_options* opts, int32_t* kernel_out) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (batch < 0 || max_ctx < 0 || nq < 1 || q_heads <= 0) return PA_ERR_INVALID_ARG;
  if (q_heads % cache->kv_heads) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  const int32_t split = split_of(opts, cache->dtype);
  if (split % kBlockSize || split > kMaxSplitTokens) return PA_ERR_UNSUPPORTED;
  int32_t kernel = opts ? opts->kernel : PA_KERNEL_AUTO;
  if (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_MMA && kernel != PA_KERNEL_SIMT) return PA_ERR_UNSUPPORTED;
  const bool int8 = cache->dtype == PA_DTYPE_INT8;
  if (int8 && kernel == PA_KERNEL_SIMT) return PA_ERR_UNSUPPORTED;
  const bool bf16 = cache->dtype == PA_DTYPE_BF16 || int8;  // int8: q / out / new rows are bf16
  if (kernel == PA_KERNEL_AUTO) kernel = bf16 ? PA_KERNEL_MMA : PA_KERNEL_SIMT;
  if (kernel == PA_KERNEL_MMA && !bf16) return PA_ERR_UNSUPPORTED;
  *kernel_out = kernel;
  if (batch == 0) return PA_OK;
  if (!q || !out || !tables || !lens || !aligned16(q) || !aligned16(out)) return PA_ERR_INVALID_ARG;
  if (mbps <= 0 || int64_t(max_ctx) > int64_t(mbps) * kBlockSize) return PA_ERR_INVALID_ARG;
  const bool fused = (k_new != nullptr);
  if (fused && (!v_new || !slots || !aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// Shared by pa_decode and pa_verify.
// query_start: null for num_queries (nq) tokens per sequence; otherwise the
// ragged layout ([batch + 1] offsets into total_queries tokens, at most nq per
// sequence).
pa_status attend(const pa_cache* cache, const void* q, void* out, const void* k_new,
                 const void* v_new, const int32_t* slots, int32_t nq, const int32_t* tables,
                 int32_t mbps, const int32_t* lens, int32_t batch, int32_t q_heads,
                 int32_t max_ctx, float scale, void* ws, size_t ws_bytes, const pa_options* opts,
                 void* stream_ptr, const int32_t* query_start = nullptr, int32_t total_queries = 0) {
  int32_t kernel = PA_KERNEL_AUTO;
  const pa_status st = attend_check(cache, q, out, k_new, v_new, slots, nq, tables, mbps, lens, batch, q_heads,
                                    max_ctx, scale, opts, &kernel);
  if (st != PA_OK || batch == 0) return st;
  const int32_t split = split_of(opts, cache->dtype);
  const bool int8 = cache->dtype == PA_DTYPE_INT8;
  const bool bf16 = cache->dtype == PA_DTYPE_BF16 || int8;
  const bool use_mma = kernel == PA_KERNEL_MMA;
  const bool fused = (k_new != nullptr);

  WsLayout L;
  const int32_t split_long = split_long_of(opts, cache->dtype);
  if (!ws_layout(batch, nq, q_heads, cache->kv_heads, max_ctx, split, split_long, &L)) return PA_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return PA_ERR_WORKSPACE;

  AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.k_cache = cache->k;
  p.v_cache = cache->v;
  p.k_cache_w = cache->k;
  p.v_cache_w = cache->v;
  p.k_scale_w = int8 ? cache->k_scale : nullptr;
  p.v_scale_w = int8 ? cache->v_scale : nullptr;
  p.q = q;
  p.out = out;
  p.k_new = k_new;
  p.v_new = v_new;
  p.slot_mapping = slots;
  p.query_start = query_start;
  p.total_queries = query_start ? total_queries : batch * nq;
  p.block_tables = tables;
  p.context_lens = lens;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<uint32_t*>(wsb);
  p.counters = reinterpret_cast<int32_t*>(wsb + L.counters);
  p.part_lse = reinterpret_cast<float*>(wsb + L.lse);
  p.part_o = reinterpret_cast<float*>(wsb + L.o);
  p.kv_heads = cache->kv_heads;
  p.num_blocks = cache->num_blocks;
  p.mbps = mbps;
  p.batch = batch;
  p.q_heads = q_heads;
  p.group = q_heads / cache->kv_heads;
  p.num_queries = nq;
  p.rows = nq * p.group;
  p.rows_per_cta = use_mma ? 16 : 8;
  p.row_groups = (p.rows + p.rows_per_cta - 1) / p.rows_per_cta;
  p.max_context_len = max_ctx;
  p.split_tokens = split;
  p.split_long = split_long;
  p.long_from = PA_LONG_CONTEXT_TOKENS;
  p.max_splits = L.max_splits;
  p.fused_write = fused ? 1 : 0;
  // The CUDA-core kernel merges in its last split; the tensor-core kernels
  // leave the merge to merge_kernel.
  p.merge_in_kernel = kernel == PA_KERNEL_SIMT ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_of(opts);

  const int64_t gz = int64_t(batch) * p.row_groups;
  if (gz > 65535 || L.max_splits > 65535) return PA_ERR_UNSUPPORTED;
  if (int64_t(batch) * cache->kv_heads * p.row_groups * L.max_splits > INT32_MAX) return PA_ERR_UNSUPPORTED;
  // Splits vary slowest: every (sequence, KV head, row group)'s first split
  // is scheduled before any second one, so the later splits of the long
  // sequences fill the slots the short sequences free.
  const dim3 grid(unsigned(cache->kv_heads), unsigned(gz), unsigned(L.max_splits));
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  cudaError_t e;
  if (int8) {
    // With one row group per (sequence, KV head) the CTA that holds a new
    // token's block is its only reader, so it requantises the block itself.
    // With several, the quantised append (which requantises whole blocks)
    // runs first and attention follows as its programmatic dependent. The
    // merge follows if there are splits.
    Q8Maps maps;
    if (!make_q8_maps(&maps, cache)) return cuda_fail(cudaErrorInvalidValue);
    const bool append_first = fused && p.row_groups > 1;
    p.fused_write = (fused && !append_first) ? 1 : 0;
    p.wait_append = append_first ? 1 : 0;
    e = cudaSuccess;
    if (append_first) e = launch_cache_write_q8(cache, k_new, v_new, slots, p.total_queries, p.status, stream);
    if (e == cudaSuccess) e = launch_attn_q8(maps, p, grid, append_first, stream);
    if (e == cudaSuccess && p.max_splits > 1) e = launch_merge(p, stream);
  } else if (kernel == PA_KERNEL_MMA) {
    CUtensorMap tk, tv;
    if (!make_pool_map4(&tk, cache->k, cache->kv_heads, cache->num_blocks) ||
        !make_pool_map4(&tv, cache->v, cache->kv_heads, cache->num_blocks))
      return cuda_fail(cudaErrorInvalidValue);
    e = launch_attn_mma(tk, tv, p, grid, stream);
    if (e == cudaSuccess && p.max_splits > 1) e = launch_merge(p, stream);
  } else {
    e = launch_attn_simt(p, bf16, grid, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return PA_OK;
}

}  // namespace

namespace pa {
// pa_decode's host-side checks without the workspace (pa_decode_noalloc runs
// them before it touches its scratch).
pa_status decode_check(const pa_cache* cache, const void* q, const void* out, const int32_t* tables, int32_t mbps,
                       const int32_t* lens, int32_t batch, int32_t q_heads, int32_t max_ctx, float scale,
                       const pa_options* opts) {
  int32_t kernel = PA_KERNEL_AUTO;
  return attend_check(cache, q, out, nullptr, nullptr, nullptr, 1, tables, mbps, lens, batch, q_heads, max_ctx,
                      scale, opts, &kernel);
}

// Bytes at the start of a workspace that must be zero when a call starts
// (status word and arrival counters); 0 if the sizes are invalid.
size_t workspace_zero_prefix(int32_t batch, int32_t nq, int32_t q_heads, int32_t kv_heads,
                             int32_t max_ctx, int32_t split) {
  WsLayout L;
  return ws_layout(batch, nq, q_heads, kv_heads, max_ctx, split, split_long_of(nullptr, -1), &L) ? L.lse : 0;
}

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }
}  // namespace pa

extern "C" {

pa_status pa_cache_write(const pa_cache* cache, const void* k_new, const void* v_new,
                         const int32_t* slot_mapping, int32_t num_tokens, void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))
    return PA_ERR_INVALID_ARG;
  if (cache->dtype == PA_DTYPE_INT8) {
    const cudaError_t e = launch_cache_write_q8(cache, k_new, v_new, slot_mapping, num_tokens, nullptr,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
  }
  const int32_t cpr = int32_t(kHeadDim * elem_size(cache->dtype) / 16);
  const int64_t total = int64_t(num_tokens) * cache->kv_heads * 2 * cpr;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 152 * 16);
  cache_write_kernel<<<unsigned(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(cache->k), static_cast<uint4*>(cache->v), static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), slot_mapping, num_tokens, cache->kv_heads, cache->num_blocks,
      cpr);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_workspace_size(int32_t batch, int32_t num_queries, int32_t q_heads, int32_t kv_heads,
                         int32_t head_dim, int32_t max_context_len, const pa_options* opts) {
  if (head_dim != kHeadDim) return 0;
  WsLayout L;
  if (!ws_layout(batch, num_queries, q_heads, kv_heads, max_context_len, split_of(opts, -1),
                 split_long_of(opts, -1), &L))
    return 0;
  return L.total;
}

pa_status pa_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace) return PA_ERR_INVALID_ARG;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_workspace_status(void* workspace, uint32_t* host_flags, void* stream) {
  if (!workspace || !host_flags) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  *host_flags = v;
  return PA_OK;
}

pa_status pa_decode(const pa_cache* cache, const void* q, void* out, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                    int32_t q_heads, int32_t max_context_len, float scale, void* workspace,
                    size_t workspace_bytes, const pa_options* opts, void* stream) {
  return attend(cache, q, out, nullptr, nullptr, nullptr, 1, block_tables, max_blocks_per_seq,
                context_lens, batch, q_heads, max_context_len, scale, workspace, workspace_bytes, opts,
                stream);
}

pa_status pa_verify(const pa_cache* cache, const void* q, void* out, const void* k_new,
                    const void* v_new, const int32_t* slot_mapping, int32_t num_queries,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t batch, int32_t q_heads,
                    int32_t max_context_len, float scale, void* workspace, size_t workspace_bytes,
                    const pa_options* opts, void* stream) {
  if (num_queries < 1) return PA_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new || !slot_mapping)) return PA_ERR_INVALID_ARG;
  return attend(cache, q, out, k_new, v_new, slot_mapping, num_queries, block_tables,
                max_blocks_per_seq, context_lens, batch, q_heads, max_context_len, scale, workspace,
                workspace_bytes, opts, stream);
}

pa_status pa_verify_ragged(const pa_cache* cache, const void* q, void* out, const void* k_new,
                           const void* v_new, const int32_t* slot_mapping, const int32_t* query_start,
                           int32_t total_queries, int32_t max_queries, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                           int32_t q_heads, int32_t max_context_len, float scale, void* workspace,
                           size_t workspace_bytes, const pa_options* opts, void* stream) {
  if (total_queries < 0 || max_queries < 1 || batch < 0) return PA_ERR_INVALID_ARG;
  if (batch > 0 && !query_start) return PA_ERR_INVALID_ARG;
  if (batch == 0 || total_queries == 0) return check_cache(cache);
  if (!k_new || !v_new || !slot_mapping) return PA_ERR_INVALID_ARG;
  return attend(cache, q, out, k_new, v_new, slot_mapping, max_queries, block_tables, max_blocks_per_seq,
                context_lens, batch, q_heads, max_context_len, scale, workspace, workspace_bytes, opts,
                stream, query_start, total_queries);
}

pa_status pa_prefill(const pa_cache* cache, const void* q, void* out, const int32_t* query_start,
                     int32_t total_queries, int32_t max_queries, const int32_t* block_tables,
                     int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch, int32_t q_heads,
                     int32_t max_context_len, float scale, void* workspace, size_t workspace_bytes,
                     const pa_options* opts, void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (cache->dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
  const int32_t kernel = opts ? opts->kernel : PA_KERNEL_AUTO;
  if (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_TC && kernel != PA_KERNEL_MMA) return PA_ERR_UNSUPPORTED;
  if (batch < 0 || total_queries < 0 || max_queries < 1 || max_context_len < 0 || q_heads <= 0)
    return PA_ERR_INVALID_ARG;
  if (q_heads % cache->kv_heads || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (batch == 0 || total_queries == 0) return PA_OK;
  if (!q || !out || !query_start || !block_tables || !context_lens || !aligned16(q) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || int64_t(max_context_len) > int64_t(max_blocks_per_seq) * kBlockSize)
    return PA_ERR_INVALID_ARG;
  if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < 256))
    return PA_ERR_WORKSPACE;
  if (batch > 65535) return PA_ERR_UNSUPPORTED;
  const int32_t group = q_heads / cache->kv_heads;
  // The tcgen05 kernel takes whole tokens per CTA (floor(128 / group) of
  // them), so it needs group <= 128; the warp-level kernel takes 128 rows.
  const bool tc = kernel == PA_KERNEL_TC || (kernel == PA_KERNEL_AUTO && group <= kPrefillRows);
  if (tc && group > kPrefillRows) return PA_ERR_UNSUPPORTED;
  const int32_t rows_per_cta = tc ? (kPrefillRows / group) * group : kPrefillRows;
  const int64_t rows = int64_t(max_queries) * group;
  const int64_t tiles = (rows + rows_per_cta - 1) / rows_per_cta;
  if (tiles * cache->kv_heads * batch > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;

  AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.k_cache = cache->k;
  p.v_cache = cache->v;
  p.q = q;
  p.out = out;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.total_queries = total_queries;
  p.status = static_cast<uint32_t*>(workspace);
  p.kv_heads = cache->kv_heads;
  p.num_blocks = cache->num_blocks;
  p.mbps = max_blocks_per_seq;
  p.batch = batch;
  p.q_heads = q_heads;
  p.group = group;
  p.num_queries = max_queries;
  p.rows = int32_t(std::min<int64_t>(rows, INT32_MAX));
  p.rows_per_cta = rows_per_cta;
  p.row_groups = int32_t(tiles);
  p.max_context_len = max_context_len;
  p.split_tokens = kBlockSize;  // unused: a prefill CTA reads its rows' whole visible context
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_of(opts);
  CUtensorMap tk, tv;
  if (!make_pool_map(&tk, cache->k, cache->kv_heads, cache->num_blocks) ||
      !make_pool_map(&tv, cache->v, cache->kv_heads, cache->num_blocks))
    return cuda_fail(cudaErrorInvalidValue);
  const dim3 grid(unsigned(tiles), unsigned(cache->kv_heads), unsigned(batch));
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tc) {
    CUtensorMap tq;
    if (!make_query_map(&tq, q, total_queries, q_heads, group, rows_per_cta / group))
      return cuda_fail(cudaErrorInvalidValue);
    e = launch_attn_prefill_tc(tk, tv, tq, p, cs);  // a persistent grid over the same items
  } else {
    e = launch_attn_prefill(tk, tv, p, grid, cs);
  }
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_validate(const pa_cache* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                      const int32_t* context_lens, int32_t batch, int32_t max_context_len,
                      const int32_t* slot_mapping, int32_t num_queries, uint32_t* report,
                      void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (!report || batch < 0 || num_queries < 1 || max_blocks_per_seq <= 0 || max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (batch > 0 && (!block_tables || !context_lens)) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(report, 0, PA_VALIDATE_WORDS * sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (batch == 0) return PA_OK;
  validate_kernel<<<unsigned(batch), 128, 0, s>>>(block_tables, max_blocks_per_seq, context_lens,
                                                   max_context_len, cache->num_blocks, slot_mapping,
                                                   num_queries, report);
  e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_ERR_UNKNOWN";
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

int pa_version(void) { return 100; }

}  // extern "C"
