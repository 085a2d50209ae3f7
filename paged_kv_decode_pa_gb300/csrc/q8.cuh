// The int8 KV pool: quantiser steps and one warp's attention step over a
// 16-token block of int8 codes (sm_103a).
//
// Pool format ("A Rust inference server for Qwen2 on Apple Silicon", Day 4,
// "int8 KV", "Grouping is the whole question", "Partial blocks"): symmetric
// codes q in [-127, 127] stored as bytes q + 128; K has one fp32 scale per
// (head, block, channel), spanning the block's 16 rows; V one per (head,
// block, row). Quantising stores s = max|x| / 127 and takes q = x * (127 /
// max|x|) rounded to nearest, ties to even: one IEEE fp32 division per group
// and one multiply per element, so the bytes are reproducible exactly. An
// all-zero group has s = 0 and bytes 128. A value is (byte - 128) * s.
//
// Attention step. The bytes stay exact in f16: a byte c placed as the low
// mantissa byte of the f16 pattern 0x64cc is 1024 + c, and subtracting 1152
// leaves c - 128 with no rounding. Scores are a sum over channels of
// K code x (K scale x q), so K's per-channel scales multiply the query once
// per block, in fp32, and the product enters the MMA as two f16 parts (hi +
// lo, about 22 bits): a single f16 rounding (2^-11 of each term) would put
// an error of that relative size on every score, which the exponential turns
// into percent-level weight errors once scores are large (sharply peaked
// rows). V's per-row scales fold into the softmax weights (P' = p * s_row,
// one f16 rounding: 2^-12 of the weight, well inside the output tolerance).
// Both products run on m16n8k16 f16 tensor-core MMAs with fp32
// accumulation. The accumulator is rescaled only when some row's running
// maximum grew in the block (otherwise the factor is exactly 1). A product
// q x (K scale) beyond the f16 range (|x| > 65504) is not supported.
//
// Fragments straight from the byte tiles. ldmatrix of a 16-row x 128-byte
// tile in 16-bit units gives each lane 4 consecutive bytes of a row. A dot
// product does not care in which order its terms are summed, so for
// S^T = K Q^T a lane's bytes for dims 4c..4c+3 serve as the MMA's k slots
// 2c, 2c+1, 2c+8, 2c+9, and Q^T is loaded with the same assignment. For
// O^T = V^T P^T, ldmatrix.trans gives a lane (token 2c, 2c+1) x (dim 2g,
// 2g+1); the MMA's rows g and g+8 are taken as dims 2g and 2g+1, so the
// accumulator of tile m holds dims 16m + 2g (elements 0, 1) and 16m + 2g + 1
// (elements 2, 3).
#pragma once

#include "mma_tile.cuh"

namespace pa {

// ---- quantiser steps (shared by the append kernel and nothing else) -----

__device__ __forceinline__ float q8_scale(float maxabs) { return __fdiv_rn(maxabs, 127.0f); }

// Inverse scale of a group (0 for an all-zero group).
__device__ __forceinline__ float q8_inverse(float maxabs) {
  return maxabs == 0.0f ? 0.0f : __fdiv_rn(127.0f, maxabs);
}

__device__ __forceinline__ uint32_t q8_code(float x, float inv) {
  if (inv == 0.0f) return 128u;
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return uint32_t(int(r) + 128);
}

__device__ __forceinline__ float q8_value(uint32_t byte, float s) {
  return __fmul_rn(float(int(byte) - 128), s);
}

// ---- f16 fragments -------------------------------------------------------

constexpr int kQ8TileBytes = 16 * 128;   // one 16-row tile of bytes
constexpr int kQ8KScaleBytes = 128 * 4;  // K scales of one block
constexpr int kQ8VScaleBytes = 16 * 4;   // V scales of one block
// Stage layout: K bytes | V bytes | K scales | V scales, 1024-byte stride so
// the swizzled tiles keep their alignment.
constexpr int kQ8KOff = 0;
constexpr int kQ8VOff = kQ8TileBytes;
constexpr int kQ8KsOff = 2 * kQ8TileBytes;
constexpr int kQ8VsOff = kQ8KsOff + kQ8KScaleBytes;
constexpr int kQ8BlockBytes = kQ8VsOff + kQ8VScaleBytes;  // bytes a block brings in (4672)
constexpr int kQ8StageBytes = 5 * 1024;

// Byte offset of (row t, 16-byte chunk c of 8) in a 128-byte-swizzled byte tile.
__device__ __forceinline__ uint32_t q8_off(int t, int c) {
  return uint32_t(t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Two bytes of x (selected by sel, see q8_pair_*) as f16 (c - 128) values.
__device__ __forceinline__ uint32_t q8_pair(uint32_t x, uint32_t sel) {
  const uint32_t biased = __byte_perm(x, 0x6464u, sel);  // f16 1024 + c in each half
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x64806480u));  // - 1152
  return r;
}
constexpr uint32_t kSelB01 = 0x5140u;  // bytes 0, 1
constexpr uint32_t kSelB23 = 0x5342u;  // bytes 2, 3
constexpr uint32_t kSelB02 = 0x5240u;  // bytes 0, 2
constexpr uint32_t kSelB13 = 0x5341u;  // bytes 1, 3

// Pack two fp32 into f16x2 (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// q (a bf16 pair) times two fp32 scales as two f16x2 parts, hi + lo: the
// products in packed fp32, hi = the top 11 significant bits (exact in f16),
// lo = p - hi exactly, then rounded to f16.
__device__ __forceinline__ void split_qs(uint32_t q2, float s0, float s1, uint32_t& h, uint32_t& l) {
  uint64_t p, s, a;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(bf16_lo(q2)), "f"(bf16_hi(q2)));
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(p), "l"(s));
  a = p & 0xffffe000ffffe000ull;
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(p), "l"(a));
  float a0, a1, d0, d1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
  h = pack_f16x2(a0, a1);
  l = pack_f16x2(d0, d1);
}

// D (16x8 fp32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Q^T in the permuted k order, as the query's own bf16 pairs: qb[kk][nt][0]
// = dims 16kk + 4c, +1 of row nt*8 + g; [1] = dims 16kk + 4c + 2, +3. Rows
// past the group are zero. Each block multiplies them by its K scales.
template <int NT>
__device__ __forceinline__ void q8_load_q(const uint16_t* q_rows, const int64_t (&row_off)[NT],
                                          const bool (&live)[NT], int c, uint32_t (&qb)[8][NT][2]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint2 v = make_uint2(0u, 0u);
      if (live[nt]) v = __ldg(reinterpret_cast<const uint2*>(q_rows + row_off[nt] + kk * 16 + 4 * c));
      qb[kk][nt][0] = v.x;
      qb[kk][nt][1] = v.y;
    }
}

// NB consecutive blocks (1 or 2) in one online-softmax step: S^T = K Q^T for
// each, mask, one running-max update over all NB x 16 tokens, O^T += V^T P'^T.
// Two blocks give the warp two independent chains of byte conversions and
// MMAs to interleave, and halve the softmax bookkeeping per token.
// stage[b]: shared address of block b's stage; kst / vst: generic pointers to
// its K and V scales; tok0: position of the first block's first token.
// limit[nt][e]: last visible position of row nt*8+2c+e.
template <int NT, int NB>
__device__ __forceinline__ void attend_blocks_q8(const uint32_t (&stage)[NB], const float* const (&kst)[NB],
                                                 const float* const (&vst)[NB],
                                                 const uint32_t (&qb)[8][NT][2], const int (&limit)[NT][2],
                                                 int tok0, float scale_log2, const Lanes& ln,
                                                 RowState<NT>& st) {
  // S^T per block, as two accumulation chains (even / odd 16-dim slices).
  float sc[NB][NT][4], sc_odd[NB][NT][4];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[b][nt][e] = sc_odd[b][nt][e] = 0.f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {  // 32 dims per ldmatrix.x4
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint32_t r0, r1, r2, r3;  // rows g / g+8, dims 32s + 4c.. and 32s + 16 + 4c..
      ldsm_x4(stage[b] + kQ8KOff + q8_off(ln.k_tok, 2 * s + ln.k_chunk), r0, r1, r2, r3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = 2 * s + h;
        const float4 ks = *reinterpret_cast<const float4*>(kst[b] + kk * 16 + 4 * ln.c);  // channel scales
        const uint32_t lo = h ? r2 : r0, hi = h ? r3 : r1;
        uint32_t a[4];
        a[0] = q8_pair(lo, kSelB01);
        a[1] = q8_pair(hi, kSelB01);
        a[2] = q8_pair(lo, kSelB23);
        a[3] = q8_pair(hi, kSelB23);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t h01, h23, l01, l23;
          split_qs(qb[kk][nt][0], ks.x, ks.y, h01, l01);
          split_qs(qb[kk][nt][1], ks.z, ks.w, h23, l23);
          mma_f16_16816(h ? sc_odd[b][nt] : sc[b][nt], a, h01, h23);
          mma_f16_16816(h ? sc_odd[b][nt] : sc[b][nt], a, l01, l23);
        }
      }
    }
  }

  // Scale to base-2 units and mask: sc[b][nt][0/1] token 16b + g, rows
  // 2c/2c+1; sc[b][nt][2/3] token 16b + g + 8.
  float bmax[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) bmax[nt][e] = -INFINITY;
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int lim = limit[nt][e], t = tok0 + 16 * b + ln.g;
        const float s0 = (t <= lim) ? (sc[b][nt][e] + sc_odd[b][nt][e]) * scale_log2 : -INFINITY;
        const float s1 = (t + 8 <= lim) ? (sc[b][nt][e + 2] + sc_odd[b][nt][e + 2]) * scale_log2 : -INFINITY;
        sc[b][nt][e] = s0;
        sc[b][nt][e + 2] = s1;
        bmax[nt][e] = fmaxf(bmax[nt][e], fmaxf(s0, s1));
      }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        bmax[nt][e] = fmaxf(bmax[nt][e], __shfl_xor_sync(0xffffffffu, bmax[nt][e], off));

  bool grew = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) grew |= bmax[nt][e] > st.m[nt][e];
  grew = __any_sync(0xffffffffu, grew);

  // Weights. Row scales of this lane's tokens (NaN-safe: masked tokens get 0).
  uint32_t pb[NB][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float alpha[2] = {1.f, 1.f}, m_use[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m_new = fmaxf(st.m[nt][e], bmax[nt][e]);
      m_use[e] = (m_new == -INFINITY) ? 0.f : m_new;
      if (grew) alpha[e] = fast_exp2(st.m[nt][e] - m_use[e]);
      st.m[nt][e] = m_new;
      st.l[nt][e] *= alpha[e];
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sv0 = vst[b][ln.g], sv1 = vst[b][ln.g + 8];
      float pr[4], pw[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pr[e] = fast_exp2(sc[b][nt][e] - m_use[e]);
        pr[e + 2] = fast_exp2(sc[b][nt][e + 2] - m_use[e]);
        pw[e] = sc[b][nt][e] == -INFINITY ? 0.f : pr[e] * sv0;
        pw[e + 2] = sc[b][nt][e + 2] == -INFINITY ? 0.f : pr[e + 2] * sv1;
      }
      st.l[nt][0] += pr[0] + pr[2];
      st.l[nt][1] += pr[1] + pr[3];
      pb[b][nt][0] = movmatrix_trans(pack_f16x2(pw[0], pw[1]));  // tokens 2c, 2c+1 of row g
      pb[b][nt][1] = movmatrix_trans(pack_f16x2(pw[2], pw[3]));  // tokens 8+2c, 9+2c of row g
    }
    if (grew) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.o[mt][nt][0] *= alpha[0];
        st.o[mt][nt][1] *= alpha[1];
        st.o[mt][nt][2] *= alpha[0];
        st.o[mt][nt][3] *= alpha[1];
      }
    }
  }

  // O^T += V^T P'^T: tile m = 2s + h holds dims 16m + 2g (+1).
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint32_t r0, r1, r2, r3;  // (tokens 2c, 2c+1 | 8+2c, 9+2c) x (dims 2g, 2g+1) of chunks 2s, 2s+1
      ldsm_x4_trans(stage[b] + kQ8VOff + q8_off(ln.k_tok, 2 * s + ln.k_chunk), r0, r1, r2, r3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lo = h ? r2 : r0, hi = h ? r3 : r1;
        uint32_t a[4];
        a[0] = q8_pair(lo, kSelB02);  // dim 2g,   tokens 2c, 2c+1
        a[1] = q8_pair(lo, kSelB13);  // dim 2g+1, tokens 2c, 2c+1
        a[2] = q8_pair(hi, kSelB02);  // dim 2g,   tokens 8+2c, 9+2c
        a[3] = q8_pair(hi, kSelB13);  // dim 2g+1
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(st.o[2 * s + h][nt], a, pb[b][nt][0], pb[b][nt][1]);
      }
    }
  }
}

}  // namespace pa
