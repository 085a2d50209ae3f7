// Quantised append into the int8 KV pool ("A Rust inference server for Qwen2
// on Apple Silicon", Day 4, "Partial blocks").
//
// A per-channel K scale spans all 16 rows of a block, so a write requantises
// the whole block: dequantise its K rows, overwrite the incoming rows,
// recompute each channel's scale, requantise every row. Every incoming V row
// is quantised on its own scale. All rows one call writes into a block are
// applied together (the later token wins for a repeated slot), then the block
// is requantised once. The fp32 steps use IEEE division and multiplication
// with no contraction, so bytes and scales are reproducible exactly.
//
// One CTA per (token, KV head), one thread per channel. The CTA of the first
// token of the call that lands in a block (in token order) handles that block
// for its head; the CTAs of later tokens in the same block return at once.
#include "q8.cuh"

namespace pa {

__global__ void __launch_bounds__(kHeadDim)
    cache_write_q8_kernel(uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, float* __restrict__ ks,
                          float* __restrict__ vs, const uint16_t* __restrict__ kn,
                          const uint16_t* __restrict__ vn, const int32_t* __restrict__ slots,
                          int32_t n, int32_t kv_heads, int32_t num_blocks, uint32_t* status) {
  pdl_launch_dependents();  // a dependent attention grid may start its prologue
  __shared__ int s_last[kBlockSize];
  __shared__ float s_red[kHeadDim / 32];
  const int i = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int warp = d >> 5, lane = d & 31;
  const int64_t num_slots = int64_t(num_blocks) * kBlockSize;
  // One round trip for what does not depend on the block: this token's slot,
  // the nearest earlier and later tokens' slots (one per thread), and this
  // token's own new K and V channel (the row it nearly always writes).
  const int64_t slot = __ldg(slots + i);
  const int jb = i - 1 - d, jf = i + d;
  const int64_t sb = jb >= 0 ? __ldg(slots + jb) : -1;
  const int64_t sf = jf < n ? __ldg(slots + jf) : -1;
  const float k_own = bf16_lo(uint32_t(__ldg(kn + (int64_t(i) * kv_heads + h) * kHeadDim + d)));
  const float v_own = bf16_lo(uint32_t(__ldg(vn + (int64_t(i) * kv_heads + h) * kHeadDim + d)));
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (d == 0 && h == 0) raise_flag(status, PA_FLAG_BAD_SLOT);
    return;
  }
  const int64_t block = slot / kBlockSize;
  // The block's K codes and scale of this thread's channel, requested before
  // the scans below so that their latency overlaps them.
  const int64_t blk = int64_t(h) * num_blocks + block;
  uint8_t* kb = kc + blk * kBlockSize * kHeadDim;
  const float s_old = ks[blk * kHeadDim + d];
  uint8_t code[kBlockSize];
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r) code[r] = kb[r * kHeadDim + d];

  // Leave the block to an earlier token of this call that lands in it.
  // Scanning backwards finds the usual case (the previous token) at once.
  if (__syncthreads_or(sb >= 0 && sb < num_slots && sb / kBlockSize == block)) return;
  for (int j0 = i - 1 - kHeadDim; j0 >= 0; j0 -= kHeadDim) {
    const int j = j0 - d;
    bool hit = false;
    if (j >= 0) {
      const int64_t sj = __ldg(slots + j);
      hit = sj >= 0 && sj < num_slots && sj / kBlockSize == block;
    }
    if (__syncthreads_or(hit)) return;
  }

  // The last token of the call (in token order) for each row of the block.
  if (d < kBlockSize) s_last[d] = -1;
  __syncthreads();
  if (sf >= 0 && sf < num_slots && sf / kBlockSize == block) atomicMax(&s_last[sf % kBlockSize], jf);
  for (int j = jf + kHeadDim; j < n; j += kHeadDim) {
    const int64_t sj = __ldg(slots + j);
    if (sj >= 0 && sj < num_slots && sj / kBlockSize == block) atomicMax(&s_last[sj % kBlockSize], j);
  }
  __syncthreads();

  // K: this thread's channel over the block's rows.
  float x[kBlockSize];
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r) {
    const int t = s_last[r];
    x[r] = t < 0    ? q8_value(code[r], s_old)
           : t == i ? k_own
                    : bf16_lo(uint32_t(__ldg(kn + (int64_t(t) * kv_heads + h) * kHeadDim + d)));
  }
  float m = 0.f;
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r) m = fmaxf(m, fabsf(x[r]));
  const float inv = q8_inverse(m);
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r) kb[r * kHeadDim + d] = uint8_t(q8_code(x[r], inv));
  ks[blk * kHeadDim + d] = q8_scale(m);

  // V: each incoming row on its own scale (the loop condition is uniform).
  for (int r = 0; r < kBlockSize; ++r) {
    const int t = s_last[r];
    if (t < 0) continue;
    const float v = t == i ? v_own : bf16_lo(uint32_t(__ldg(vn + (int64_t(t) * kv_heads + h) * kHeadDim + d)));
    float a = fabsf(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (lane == 0) s_red[warp] = a;
    __syncthreads();
    float mv = 0.f;
#pragma unroll
    for (int k = 0; k < kHeadDim / 32; ++k) mv = fmaxf(mv, s_red[k]);
    vc[(blk * kBlockSize + r) * kHeadDim + d] = uint8_t(q8_code(v, q8_inverse(mv)));
    if (d == 0) vs[blk * kBlockSize + r] = q8_scale(mv);
    __syncthreads();  // s_red is reused by the next row
  }
}

// status may be null (plain pa_cache_write has no workspace).
cudaError_t launch_cache_write_q8(const pa_cache* c, const void* k_new, const void* v_new,
                                  const int32_t* slots, int32_t n, uint32_t* status, cudaStream_t stream) {
  const dim3 grid(unsigned(n), unsigned(c->kv_heads), 1);
  cache_write_q8_kernel<<<grid, kHeadDim, 0, stream>>>(
      static_cast<uint8_t*>(c->k), static_cast<uint8_t*>(c->v), static_cast<float*>(c->k_scale),
      static_cast<float*>(c->v_scale), static_cast<const uint16_t*>(k_new),
      static_cast<const uint16_t*>(v_new), slots, n, c->kv_heads, c->num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pa
