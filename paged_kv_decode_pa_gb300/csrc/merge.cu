// Log-sum-exp merge of split partials (flash-decoding's second pass). The
// tensor-core kernels write, for every split of a (sequence, KV head, row
// group) with more than one split, the split's normalised output and its
// log-sum-exp in base-2 units; this kernel combines them:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s.
// A split with no visible key has lse = -inf and weight 0.
#include "pa_device.cuh"

namespace pa {

constexpr int kMergeWarps = 8;

// CTA c takes (unit, row) pairs c, c + grid, ...; units with a single split
// were written by the attention kernel and are skipped. Warp w takes splits w, w+8, ...; a lane holds 4 dims; the warps'
// sums are added in warp order. Launched as a programmatic dependent of the
// attention kernel: it waits for that grid before reading anything it wrote.
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const AttnParams p) {
  pdl_wait_primary();
  __shared__ float s_max[kMergeWarps], s_den[kMergeWarps];
  __shared__ __align__(16) float s_acc[kMergeWarps][kHeadDim];
  __shared__ int s_pairs[kMergeWarps * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = min(p.rows_per_cta, p.rows);  // rows of the largest row group
  const int units = p.batch * p.kv_heads * p.row_groups;
  const int total = units * rows;
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  // CTA c owns pairs c, c + grid, c + 2 grid, ... One thread per owned pair
  // checks, in parallel, whether it needs a merge (several splits, a real
  // row); the CTA then merges the pairs found, in order.
  const int stride = gridDim.x;
  for (int first = 0; blockIdx.x + first * stride < total; first += blockDim.x) {
    const int mine = blockIdx.x + (first + threadIdx.x) * stride;
    bool need = false;
    if (mine < total) {
      const int unit = mine / rows, r = mine - unit * rows;
      const int rg = unit % p.row_groups;
      const int b = unit / p.row_groups / p.kv_heads;
      int L = __ldg(p.context_lens + b);
      L = L < 0 ? 0 : min(L, cap);
      need = r < min(p.rows_per_cta, p.rows - rg * p.rows_per_cta) &&
             (L + p.split_tokens - 1) / p.split_tokens > 1;
    }
    // Compact the pairs that need work, keeping their order.
    const unsigned ballot = __ballot_sync(0xffffffffu, need);
    if (lane == 0) s_pairs[warp] = __popc(ballot);  // per-warp counts first
    __syncthreads();
    int before = 0, found = 0;
    for (int w = 0; w < kMergeWarps; ++w) {
      if (w < warp) before += s_pairs[w];
      found += s_pairs[w];
    }
    __syncthreads();
    if (need) s_pairs[before + __popc(ballot & ((1u << lane) - 1u))] = mine;
    __syncthreads();
    for (int k = 0; k < found; ++k) {
      const int pair = s_pairs[k];
      const int unit = pair / rows, r = pair - unit * rows;
      const int rg = unit % p.row_groups;
      const int bh = unit / p.row_groups;
      const int h = bh % p.kv_heads, b = bh / p.kv_heads;
      const int row0 = rg * p.rows_per_cta;
      int L = __ldg(p.context_lens + b);
      L = L < 0 ? 0 : min(L, cap);
      const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
      const size_t base = size_t(unit) * p.max_splits;

      float mx = -INFINITY;
      for (int s = warp; s < nsplit; s += kMergeWarps)
        mx = fmaxf(mx, __ldcg(p.part_lse + (base + s) * kRowSlots + r));
      if (lane == 0) s_max[warp] = mx;
      __syncthreads();
      float M = -INFINITY;
  #pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, s_max[w]);

      float den = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (M != -INFINITY) {
  #pragma unroll 4
        for (int s = warp; s < nsplit; s += kMergeWarps) {
          const float lse = __ldcg(p.part_lse + (base + s) * kRowSlots + r);
          const float4 v =
              __ldcg(reinterpret_cast<const float4*>(p.part_o + ((base + s) * kRowSlots + r) * kHeadDim) + lane);
          const float wgt = fast_exp2(lse - M);
          den += wgt;
          acc[0] += wgt * v.x;
          acc[1] += wgt * v.y;
          acc[2] += wgt * v.z;
          acc[3] += wgt * v.w;
        }
      }
      if (lane == 0) s_den[warp] = den;
      *reinterpret_cast<float4*>(&s_acc[warp][lane * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      __syncthreads();
      if (warp == 0) {
        float d = 0.f, v[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
          d += s_den[w];
  #pragma unroll
          for (int e = 0; e < 4; ++e) v[e] += s_acc[w][lane * 4 + e];
        }
        const float iv = d > 0.f ? 1.f / d : 0.f;
        uint16_t* dst = static_cast<uint16_t*>(p.out) + row_offset(p, b, h, row0 + r) + lane * 4;
        uint2 u;
        u.x = pack_bf16x2(v[0] * iv, v[1] * iv);
        u.y = pack_bf16x2(v[2] * iv, v[3] * iv);
        *reinterpret_cast<uint2*>(dst) = u;
      }
      __syncthreads();  // the shared buffers are reused by the next pair
    }
  }
}

// Launched right after an attention kernel on the same stream, as its
// programmatic dependent: the launch overlaps the attention kernel's tail and
// griddepcontrol.wait orders every read after that kernel's writes.
cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream) {
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sms[dev]) {
    e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int64_t rows = p.rows < p.rows_per_cta ? p.rows : p.rows_per_cta;
  const int64_t pairs = int64_t(p.batch) * p.kv_heads * p.row_groups * rows;
  // One CTA per SM at most: that many fit beside a running attention kernel,
  // so the whole grid is resident and waiting when the attention kernel ends.
  const int64_t wave = int64_t(sms[dev]);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(pairs < wave ? pairs : wave), 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

}  // namespace pa
