// Paged decode / verify attention on CUDA cores (fp32 arithmetic), fp32 or
// bf16 caches.
//
// Same work split as the tensor-core kernel: one CTA per (context split, KV
// head, sequence x row group), up to 8 query rows per CTA, four warps taking
// the split's 16-token blocks round-robin, then the shared split epilogue. A
// lane owns four consecutive dims of head_dim 128; each score is a warp
// butterfly sum. The softmax is the online form of "From 183 ms to 19 ms per
// decode step", section "3. A Triton paged-decode kernel", updated per token
// with exp2f. This kernel serves the fp32 cache and is the CUDA-core arm the
// tensor-core kernel is compared against.
#include "pa_device.cuh"

namespace pa {

constexpr int kSimtRows = 8;
constexpr int kSimtThreads = kConsumerWarps * 32;

template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  static __device__ __forceinline__ void load(const float* src, float (&v)[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  static __device__ __forceinline__ void load_plain(const float* src, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  static __device__ __forceinline__ void copy(float* dst, const float* src) {
    *reinterpret_cast<float4*>(dst) = __ldg(reinterpret_cast<const float4*>(src));
  }
};
template <>
struct Vec4<uint16_t> {
  static __device__ __forceinline__ void unpack(uint2 x, float (&v)[4]) {
    v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
  }
  static __device__ __forceinline__ void load(const uint16_t* src, float (&v)[4]) {
    unpack(__ldg(reinterpret_cast<const uint2*>(src)), v);
  }
  static __device__ __forceinline__ void load_plain(const uint16_t* src, float (&v)[4]) {
    unpack(*reinterpret_cast<const uint2*>(src), v);
  }
  static __device__ __forceinline__ void copy(uint16_t* dst, const uint16_t* src) {
    *reinterpret_cast<uint2*>(dst) = __ldg(reinterpret_cast<const uint2*>(src));
  }
};

template <typename T>
__global__ void __launch_bounds__(kSimtThreads) attn_simt_kernel(const AttnParams p) {
  __shared__ __align__(16) float cbuf[kConsumerWarps * kRowSlots * kCombineStride];
  __shared__ float s_m[kConsumerWarps * kRowSlots], s_l[kConsumerWarps * kRowSlots];
  __shared__ int s_flag[4];

  const CtaWork w = cta_work(p);
  if (w.nrows <= 0) return;  // a ragged sequence with fewer query rows than this group
  if (w.split >= w.nsplit) {
    if (w.L == 0 && w.split == 0) write_zero_rows<T>(p, w);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d0 = lane * 4;
  const int nblk = (w.t1 - w.t0 + kBlockSize - 1) / kBlockSize;
  const int new0 = w.L - w.nq;
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);

  float q[kSimtRows][4], acc[kSimtRows][4], m[kSimtRows], l[kSimtRows];
  int limit[kSimtRows];
#pragma unroll
  for (int r = 0; r < kSimtRows; ++r) {
    if (r < w.nrows) {
      Vec4<T>::load(static_cast<const T*>(p.q) + row_offset(p, w.q0, w.h, w.row0 + r) + d0, q[r]);
      limit[r] = row_limit(p, w.L, w.nq, w.row0 + r);
    } else {
      q[r][0] = q[r][1] = q[r][2] = q[r][3] = 0.f;
      limit[r] = -1;
    }
    acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
    m[r] = -INFINITY;
    l[r] = 0.f;
  }

  for (int j = warp; j < nblk; j += kConsumerWarps) {
    const int tok0 = w.t0 + j * kBlockSize;
    int id = __ldg(p.block_tables + int64_t(w.b) * p.mbps + tok0 / kBlockSize);
    const bool id_ok = id >= 0 && id < p.num_blocks;
    if (!id_ok && lane == 0) raise_flag(p.status, PA_FLAG_BAD_BLOCK);
    const int ntok = min(kBlockSize, w.t1 - tok0);
    for (int t = 0; t < ntok; ++t) {
      const int pos = tok0 + t;
      float k[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
      const int slot = (p.fused_write && pos >= new0) ? __ldg(p.slot_mapping + w.q0 + (pos - new0)) : -1;
      if (p.fused_write && pos >= new0) {
        // A new (verify) token: read from the inputs when its slot is the
        // table slot of its position, else from the pool (a negative slot is
        // not written); row group 0 writes every in-pool slot.
        const int i = pos - new0;
        const int64_t src = (int64_t(w.q0 + i) * p.kv_heads + w.h) * kHeadDim + d0;
        if (id_ok && slot == id * kBlockSize + t) {
          Vec4<T>::load(static_cast<const T*>(p.k_new) + src, k);
          Vec4<T>::load(static_cast<const T*>(p.v_new) + src, v);
        } else if (id_ok) {
          const int64_t off = ((int64_t(w.h) * p.num_blocks + id) * kBlockSize + t) * kHeadDim + d0;
          Vec4<T>::load_plain(kc + off, k);
          Vec4<T>::load_plain(vc + off, v);
        }
        if (w.rg == 0) {
          if (slot >= 0 && slot < p.num_blocks * kBlockSize) {
            const int64_t dst =
                ((int64_t(w.h) * p.num_blocks + slot / kBlockSize) * kBlockSize + slot % kBlockSize) *
                    kHeadDim + d0;
            Vec4<T>::copy(static_cast<T*>(p.k_cache_w) + dst, static_cast<const T*>(p.k_new) + src);
            Vec4<T>::copy(static_cast<T*>(p.v_cache_w) + dst, static_cast<const T*>(p.v_new) + src);
          } else if (slot >= 0 && lane == 0) {
            raise_flag(p.status, PA_FLAG_BAD_SLOT);
          }
        }
      } else if (id_ok) {
        const int64_t off = ((int64_t(w.h) * p.num_blocks + id) * kBlockSize + t) * kHeadDim + d0;
        // Plain loads: with a fused verify another CTA may write this pool.
        Vec4<T>::load_plain(kc + off, k);
        Vec4<T>::load_plain(vc + off, v);
      }
#pragma unroll
      for (int r = 0; r < kSimtRows; ++r) {
        if (pos > limit[r]) continue;  // warp-uniform
        float dot = q[r][0] * k[0] + q[r][1] * k[1] + q[r][2] * k[2] + q[r][3] * k[3];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float s = dot * p.scale_log2;
        const float m_new = fmaxf(m[r], s);
        const float alpha = exp2f(m[r] - m_new);
        const float pw = exp2f(s - m_new);
        m[r] = m_new;
        l[r] = l[r] * alpha + pw;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = acc[r][e] * alpha + pw * v[e];
      }
    }
  }

  float* mine = cbuf + warp * kRowSlots * kCombineStride;
#pragma unroll
  for (int r = 0; r < kSimtRows; ++r) {
    *reinterpret_cast<float4*>(mine + r * kCombineStride + d0) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    if (lane == 0) {
      s_m[warp * kRowSlots + r] = m[r];
      s_l[warp * kRowSlots + r] = l[r];
    }
  }
  __syncthreads();
  split_epilogue<T>(p, w, cbuf, s_m, s_l, kConsumerWarps, s_flag);
}

cudaError_t launch_attn_simt(const AttnParams& p, bool bf16, dim3 grid, cudaStream_t stream) {
  if (bf16)
    attn_simt_kernel<uint16_t><<<grid, kSimtThreads, 0, stream>>>(p);
  else
    attn_simt_kernel<float><<<grid, kSimtThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
