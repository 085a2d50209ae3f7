// Device-side building blocks for the paged-attention kernels (sm_103a).
//
// Thin inline-PTX wrappers (mbarrier, TMA tensor loads, ldmatrix, warp-level
// bf16 MMA, movmatrix) plus the parameter block and the split epilogue that
// both attention kernels share. Nothing here allocates or synchronises the
// host.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
constexpr int kRowSlots = 16;         // rows per workspace partial slot (max rows a CTA holds)
constexpr int kMaxSplitTokens = 8192;  // largest split a CTA walks (bounds its block-id buffer)
constexpr int kConsumerWarps = 4;      // warps that attend; they take blocks round-robin
constexpr int kCombineStride = kHeadDim + 4;  // padded fp32 row stride of the cross-warp buffer
constexpr uint32_t kWaitLimitNs = PA_DEFAULT_WAIT_LIMIT_NS;  // bounded waits give up after 1 s
constexpr uint32_t kWaitLimitIters = 1u << 26;

// Everything a CTA needs; passed by value (kernel parameter space).
struct AttnParams {
  const void* k_cache;
  const void* v_cache;
  void* k_cache_w;  // same pools, written by the fused verify
  void* v_cache_w;
  void* k_scale_w;  // int8 pool: K scales [kv_heads, num_blocks, 128] (fused write)
  void* v_scale_w;  // int8 pool: V scales [kv_heads, num_blocks, 16]
  const void* q;  // [batch, num_queries, q_heads, 128]
  void* out;      // same shape
  const void* k_new;  // [batch * num_queries, kv_heads, 128] (fused verify only)
  const void* v_new;
  const int32_t* slot_mapping;  // [batch * num_queries] (fused verify only)
  const int32_t* query_start;   // ragged: [batch + 1] first query token of each sequence; null: uniform
  int32_t total_queries;        // ragged: query tokens in all (rows of q / out / k_new / v_new)
  const int32_t* block_tables;  // [batch, mbps]
  const int32_t* context_lens;  // [batch]
  uint32_t* status;             // workspace status word
  int32_t* counters;            // one per (sequence, kv head, row group)
  float* part_lse;              // [units, max_splits, 16]       (log2 units)
  float* part_o;                // [units, max_splits, 16, 128]
  int32_t kv_heads, num_blocks, mbps, batch, q_heads, group, num_queries;  // ragged: the most of any sequence
  int32_t rows;        // num_queries * group: query rows per (sequence, kv head), at most
  int32_t rows_per_cta;  // 16 (tensor-core kernel) or 8 (CUDA-core kernel)
  int32_t row_groups;  // ceil(rows / rows_per_cta)
  int32_t max_context_len, split_tokens, max_splits;
  int32_t split_long;   // > 0: sequences longer than long_from tokens use this split instead
  int32_t long_from;
  int32_t fused_write;  // 1: new rows come from k_new/v_new and are written to the cache
  int32_t wait_append;  // int8: 1 if a preceding append grid wrote the new tokens' blocks
  int32_t merge_in_kernel;  // 1: the last split to finish merges; 0: merge_kernel does
  float scale_log2;     // scale * log2(e): scores are kept in base-2 units
  uint32_t wait_limit_ns;  // bound on the pipeline waits (drains use kWaitLimitNs)
};

// ---------------------------------------------------------------------------
// Small PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false once limit_ns
// have passed (or after kWaitLimitIters polls). The clock is read every 256
// polls, or on every poll under a limit below 100 us.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  const uint32_t every = limit_ns < 100000u ? 0u : 255u;
  for (uint32_t it = 1; it < kWaitLimitIters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & every) == 0u && global_timer_ns() - t0 > limit_ns) break;
  }
  return false;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled TMA load (x innermost) completing on an mbarrier. Out-of-range
// coordinates read zeros.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar,
                                            uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(cache_policy)
      : "memory");
}

// 4-D tiled TMA load (x innermost) completing on an mbarrier. Out-of-range
// coordinates read zeros.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, int32_t w, uint32_t bar,
                                            uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(cache_policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Keep lines in L2 ahead of others: for tiles that several CTAs read.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Pack two fp32 into bf16x2 (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: let the next kernel on the stream start
// launching, and (in that kernel) wait until this one's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void raise_flag(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// Per-CTA work description

// Tokens per split for a sequence of length L (depends on L alone).
__device__ __forceinline__ int split_for(const AttnParams& p, int L) {
  return (p.split_long > 0 && L > p.long_from) ? p.split_long : p.split_tokens;
}

struct CtaWork {
  int b, h, rg, split;
  int L;          // clamped context length
  int split_size; // tokens per split of this sequence
  int nsplit;     // non-empty splits of this sequence
  int t0, t1;     // token range of this split
  int row0;       // first row of this row group
  int nrows;      // rows of this group (<= rows_per_cta; <= 0: none)
  int unit;       // (b * kv_heads + h) * row_groups + rg
  int nq;         // this sequence's query tokens (new tokens at L - nq .. L - 1)
  int q0;         // flat index of its first query token (q, out, k_new, v_new, slots)
};

// Query tokens of sequence b: uniform (num_queries each) or from query_start
// (clamped to [0, num_queries] and to the flat arrays; an inconsistent entry
// raises PA_FLAG_BAD_LENGTH once). query_range takes the two query_start
// entries already loaded.
__device__ __forceinline__ void query_range(const AttnParams& p, int a, int e, bool report, int* q0, int* nq) {
  int s = max(0, min(a, p.total_queries)), n = max(0, min(e, p.total_queries) - s);
  if (n > p.num_queries || a < 0 || e < a || e > p.total_queries) {
    if (report) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    n = min(n, p.num_queries);
  }
  *q0 = s;
  *nq = n;
}

__device__ __forceinline__ void seq_queries(const AttnParams& p, int b, bool report, int* q0, int* nq) {
  if (!p.query_start) {
    *q0 = b * p.num_queries;
    *nq = p.num_queries;
    return;
  }
  query_range(p, __ldg(p.query_start + b), __ldg(p.query_start + b + 1), report, q0, nq);
}

// The work of CTA (blockIdx.x = KV head, .y = sequence x row group, .z =
// split); L_raw is context_lens[b] if the caller has loaded it already.
__device__ __forceinline__ CtaWork cta_work(const AttnParams& p, int L_raw = -2147483647 - 1) {
  CtaWork w;
  w.split = blockIdx.z;
  w.h = blockIdx.x;
  w.b = blockIdx.y / p.row_groups;
  w.rg = blockIdx.y - w.b * p.row_groups;
  seq_queries(p, w.b, w.split == 0 && w.h == 0 && w.rg == 0, &w.q0, &w.nq);
  int L = L_raw == -2147483647 - 1 ? __ldg(p.context_lens + w.b) : L_raw;
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  if (L < 0 || L > cap) {
    if (w.split == 0 && w.h == 0 && w.rg == 0) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    L = L < 0 ? 0 : cap;
  }
  w.L = L;
  w.split_size = split_for(p, L);
  w.nsplit = (L + w.split_size - 1) / w.split_size;
  w.t0 = w.split * w.split_size;
  w.t1 = min(L, w.t0 + w.split_size);
  w.row0 = w.rg * p.rows_per_cta;
  w.nrows = min(p.rows_per_cta, w.nq * p.group - w.row0);
  w.unit = (w.b * p.kv_heads + w.h) * p.row_groups + w.rg;
  return w;
}

// Element offset of query row r (r = i * group + g) of kv head h, for the
// sequence whose first query token is q0.
__device__ __forceinline__ int64_t row_offset(const AttnParams& p, int64_t q0, int h, int r) {
  const int i = r / p.group;
  const int g = r - i * p.group;
  return ((q0 + i) * p.q_heads + h * p.group + g) * kHeadDim;
}

// Last position query row r may attend to (causal among the sequence's nq new tokens).
__device__ __forceinline__ int row_limit(const AttnParams& p, int L, int nq, int r) {
  return L - nq + r / p.group;
}

template <typename T>
__device__ __forceinline__ void store8(T* dst, const float* v);

template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* v) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

template <>
__device__ __forceinline__ void store8<uint16_t>(uint16_t* dst, const float* v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = u;
}

// A CTA whose sequence has no context (L = 0) writes zeros for its rows.
template <typename T>
__device__ void write_zero_rows(const AttnParams& p, const CtaWork& w) {
  const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int e = threadIdx.x; e < w.nrows * (kHeadDim / 8); e += blockDim.x) {
    const int r = e / (kHeadDim / 8), c = e % (kHeadDim / 8);
    T* dst = static_cast<T*>(p.out) + row_offset(p, w.q0, w.h, w.row0 + r) + c * 8;
    store8<T>(dst, z);
  }
}

// ---------------------------------------------------------------------------
// Split epilogue, shared by both attention kernels.
//
// On entry every consumer warp has written its running state to shared memory:
//   cbuf[w][r][d]  un-normalised accumulator (row stride kCombineStride),
//   mbuf[w][r], lbuf[w][r]  running max (base-2 units) and sum.
// The warps are combined in a fixed order. With a single split the CTA
// normalises and writes the output. Otherwise it stores its normalised
// partial and log-sum-exp, and the last CTA of the (sequence, kv head, row
// group) to arrive merges all partials in split order. The arrival counter
// is reset by that CTA, so the workspace is ready for the next call.
template <typename T>
__device__ void split_epilogue(const AttnParams& p, const CtaWork& w, const float* cbuf,
                               const float* mbuf, const float* lbuf, int nwarps, int* s_flag) {
  const int chunks = kHeadDim / 8;
  const int items = w.nrows * chunks;
  const bool single = (w.nsplit <= 1);
  const size_t slot = size_t(w.unit) * p.max_splits + w.split;

  for (int e = threadIdx.x; e < items; e += blockDim.x) {
    const int r = e / chunks, c = e % chunks;
    float M = -INFINITY;
    for (int k = 0; k < nwarps; ++k) M = fmaxf(M, mbuf[k * kRowSlots + r]);
    float l = 0.f, acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (M != -INFINITY) {
      for (int k = 0; k < nwarps; ++k) {
        const float f = fast_exp2(mbuf[k * kRowSlots + r] - M);
        l += f * lbuf[k * kRowSlots + r];
        const float* src = cbuf + (k * kRowSlots + r) * kCombineStride + c * 8;
#pragma unroll
        for (int d = 0; d < 8; ++d) acc[d] += f * src[d];
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[d] *= inv;
    if (single) {
      T* dst = static_cast<T*>(p.out) + row_offset(p, w.q0, w.h, w.row0 + r) + c * 8;
      store8<T>(dst, acc);
    } else {
      float* dst = p.part_o + (slot * kRowSlots + r) * kHeadDim + c * 8;
      store8<float>(dst, acc);
      if (c == 0) p.part_lse[slot * kRowSlots + r] = l > 0.f ? M + __log2f(l) : -INFINITY;
    }
  }
  if (single || !p.merge_in_kernel) return;

  // Publish this split, then count arrivals; the last arrival merges.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(p.counters + w.unit, 1);
    *s_flag = (prev == w.nsplit - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*s_flag == 0) return;
  __threadfence();

  const size_t base = size_t(w.unit) * p.max_splits;
  for (int e = threadIdx.x; e < items; e += blockDim.x) {
    const int r = e / chunks, c = e % chunks;
    float M = -INFINITY;
    for (int s = 0; s < w.nsplit; ++s) M = fmaxf(M, __ldcg(p.part_lse + (base + s) * kRowSlots + r));
    float den = 0.f, acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (M != -INFINITY) {
      for (int s = 0; s < w.nsplit; ++s) {
        const float lse = __ldcg(p.part_lse + (base + s) * kRowSlots + r);
        const float wgt = fast_exp2(lse - M);
        den += wgt;
        const float4* src =
            reinterpret_cast<const float4*>(p.part_o + ((base + s) * kRowSlots + r) * kHeadDim + c * 8);
        const float4 a = __ldcg(src), bq = __ldcg(src + 1);
        acc[0] += wgt * a.x;
        acc[1] += wgt * a.y;
        acc[2] += wgt * a.z;
        acc[3] += wgt * a.w;
        acc[4] += wgt * bq.x;
        acc[5] += wgt * bq.y;
        acc[6] += wgt * bq.z;
        acc[7] += wgt * bq.w;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[d] *= inv;
    T* dst = static_cast<T*>(p.out) + row_offset(p, w.q0, w.h, w.row0 + r) + c * 8;
    store8<T>(dst, acc);
  }
  if (threadIdx.x == 0) p.counters[w.unit] = 0;
}

// ---------------------------------------------------------------------------
// Host: one-time set-up per device (kernel attributes), safe when several host
// threads launch at once. run() calls set_up() once for the current device
// ordinal; later calls return that first result.
constexpr int kMaxDevices = 64;
struct PerDeviceOnce {
  std::once_flag flag[kMaxDevices];
  cudaError_t result[kMaxDevices] = {};
  template <typename F>
  cudaError_t run(F&& set_up) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { result[dev] = set_up(dev); });
    return result[dev];
  }
};

}  // namespace pa
