// Log-sum-exp merge of split partials (flash-decoding's second pass). The
// tensor-core kernels write, for every split of a (sequence, KV head, row
// group) with more than one split, the split's normalised output and its
// log-sum-exp in base-2 units; this kernel combines them:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s.
// A split with no visible key has lse = -inf and weight 0.
#include "pa_device.cuh"

namespace pa {

constexpr int kMergeWarps = 8;

// WP warps per (unit, row) pair: with few splits one warp takes a pair; with
// many, a whole CTA does (more loads in flight per pair). Warp part takes the
// pair's splits part, part + WP, ...: lane k of a 32-split chunk reads that
// split's log-sum-exp, the warp reduces max and sum with shuffles, and each
// lane accumulates 4 output dims over the chunk in split order; the warps'
// sums are combined in warp order. The length is read before waiting for the
// attention grid (it is an input, not written there), so pairs with a single
// split leave at once and the rest wait with their length in hand.
template <int WP>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const AttnParams p) {
  static_assert(WP == 1 || WP == kMergeWarps, "a pair takes one warp or the whole CTA");
  __shared__ float s_m[WP], s_d[WP];
  __shared__ __align__(16) float4 s_acc[WP][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = warp % WP;
  const int rows = min(p.rows_per_cta, p.rows);  // rows of the largest row group
  const int64_t units = int64_t(p.batch) * p.kv_heads * p.row_groups;
  const int64_t pair = (int64_t(blockIdx.x) * kMergeWarps + warp) / WP;
  // Every exit below depends on the pair only, so with WP > 1 the whole CTA
  // leaves together and the __syncthreads at the end is reached by all.
  if (pair >= units * rows) return;
  const int unit = int(pair / rows), r = int(pair - int64_t(unit) * rows);
  const int rg = unit % p.row_groups;
  const int bh = unit / p.row_groups;
  const int h = bh % p.kv_heads, b = bh / p.kv_heads;
  const int row0 = rg * p.rows_per_cta;
  int q0, nq;
  seq_queries(p, b, false, &q0, &nq);
  if (r >= min(p.rows_per_cta, nq * p.group - row0)) return;
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  int L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : min(L, cap);
  const int split = split_for(p, L);
  const int nsplit = (L + split - 1) / split;
  if (nsplit <= 1) return;  // written by the attention kernel itself

  pdl_wait_primary();
  const size_t base = size_t(unit) * p.max_splits;
  const float* lse = p.part_lse + base * kRowSlots + r;  // split s at lse[s * kRowSlots]
  const float4* po = reinterpret_cast<const float4*>(p.part_o + (base * kRowSlots + r) * kHeadDim) + lane;
  constexpr int kSplitStride4 = kRowSlots * kHeadDim / 4;  // float4s between splits
  constexpr int kChunk = 32 * WP;                          // splits per chunk (all warps)

  const int s_first = part + WP * lane;
  const float first = s_first < nsplit ? __ldcg(lse + size_t(s_first) * kRowSlots) : -INFINITY;
  // When this warp has at most kPre splits, their partial rows are loaded
  // together with the log-sum-exps instead of after the maximum: one memory
  // round trip instead of two. The sums run in the same order either way.
  constexpr int kPre = 8;
  const int n_w = nsplit > part ? (nsplit - part + WP - 1) / WP : 0;
  const bool pre = n_w <= kPre;
  float4 v[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k)
    v[k] = pre && k < n_w ? __ldcg(po + size_t(part + WP * k) * kSplitStride4) : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = first;
  for (int s = s_first + kChunk; s < nsplit; s += kChunk) M = fmaxf(M, __ldcg(lse + size_t(s) * kRowSlots));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY && pre) {
    // Weights and products are summed in split order, the order the CTA-wide
    // form combines its warps in: a pair of up to 8 splits gets the same bits
    // whichever form the launch takes (it depends on the batch's longest
    // sequence).
    const float wgt = s_first < nsplit ? fast_exp2(first - M) : 0.f;
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      if (k < n_w) {
        const float wk = __shfl_sync(0xffffffffu, wgt, k);
        den += wk;
        acc.x += wk * v[k].x;
        acc.y += wk * v[k].y;
        acc.z += wk * v[k].z;
        acc.w += wk * v[k].w;
      }
    }
  } else if (M != -INFINITY) {
    for (int s0 = part; s0 < nsplit; s0 += kChunk) {
      const int s = s0 + WP * lane;
      const float ls = s0 == part ? first : (s < nsplit ? __ldcg(lse + size_t(s) * kRowSlots) : -INFINITY);
      const float wgt = s < nsplit ? fast_exp2(ls - M) : 0.f;
      den += wgt;
      const int n = min(32, (nsplit - s0 + WP - 1) / WP);
#pragma unroll 8
      for (int k = 0; k < n; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wgt, k);
        const float4 v = __ldcg(po + size_t(s0 + WP * k) * kSplitStride4);
        acc.x += wk * v.x;
        acc.y += wk * v.y;
        acc.z += wk * v.z;
        acc.w += wk * v.w;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  }
  if constexpr (WP > 1) {
    // Rescale each warp's sums to the pair's maximum and add them in warp order.
    if (lane == 0) {
      s_m[warp] = M;
      s_d[warp] = den;
    }
    s_acc[warp][lane] = acc;
    __syncthreads();
    if (warp != 0) return;
    float Mall = -INFINITY;
#pragma unroll
    for (int k = 0; k < WP; ++k) Mall = fmaxf(Mall, s_m[k]);
    den = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mall != -INFINITY) {
#pragma unroll
      for (int k = 0; k < WP; ++k) {
        const float f = s_m[k] == -INFINITY ? 0.f : fast_exp2(s_m[k] - Mall);
        const float4 a = s_acc[k][lane];
        den += f * s_d[k];
        acc.x += f * a.x;
        acc.y += f * a.y;
        acc.z += f * a.z;
        acc.w += f * a.w;
      }
    }
  }
  const float iv = den > 0.f ? 1.f / den : 0.f;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + row_offset(p, q0, h, row0 + r) + lane * 4;
  uint2 u;
  u.x = pack_bf16x2(acc.x * iv, acc.y * iv);
  u.y = pack_bf16x2(acc.z * iv, acc.w * iv);
  *reinterpret_cast<uint2*>(dst) = u;
}

// Launched right after an attention kernel on the same stream, as its
// programmatic dependent: the launch overlaps the attention kernel's tail and
// griddepcontrol.wait orders every read after that kernel's writes.
cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream) {
  const int64_t rows = p.rows < p.rows_per_cta ? p.rows : p.rows_per_cta;
  const int64_t pairs = int64_t(p.batch) * p.kv_heads * p.row_groups * rows;
  cudaLaunchConfig_t cfg = {};
  // Up to 8 splits a warp per pair; beyond that a CTA per pair.
  const bool wide = p.max_splits > kMergeWarps;
  cfg.gridDim = dim3(unsigned(wide ? pairs : (pairs + kMergeWarps - 1) / kMergeWarps), 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return wide ? cudaLaunchKernelEx(&cfg, merge_kernel<kMergeWarps>, p)
              : cudaLaunchKernelEx(&cfg, merge_kernel<1>, p);
}

}  // namespace pa
