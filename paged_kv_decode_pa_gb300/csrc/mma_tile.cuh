// One warp's attention step over a 16-token K/V block held in shared memory,
// with bf16 tensor-core products (m16n8k16) and an fp32 online softmax. Used
// by both tensor-core kernels (TMA-staged and load-staged).
//
// Tile layout in shared memory (8 KiB per block): K then V, each 16 token
// rows x 128 dims bf16, stored as two 2 KiB halves (dims 0..63, 64..127) of
// 128-byte rows whose 16-byte chunks are XOR-swizzled by (row & 7). This is
// the layout a 128-byte-swizzled TMA box produces, and it makes every
// ldmatrix below bank-conflict free.
//
// Per block a warp computes S^T = K Q^T (16 tokens x 8*NT query rows), masks
// positions past each row's limit, runs the online softmax update (running
// max and sum, rescaled per block: "From 183 ms to 19 ms per decode step",
// section "3. A Triton paged-decode kernel"), turns P^T into the B operand in
// registers with movmatrix, and accumulates O^T += V^T P^T.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kTileBytes = 16 * 128 * 2;   // one 16-token bf16 tile of K or V
constexpr int kHalfTile = kTileBytes / 2;  // 16 rows x 64 dims
constexpr int kBlockBytes = 2 * kTileBytes;  // K + V

// Byte offset of (token row t, 16-byte chunk c of 16) inside a K or V tile.
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
  return uint32_t((c >> 3) * kHalfTile + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Per-lane roles in the MMA fragments and ldmatrix address patterns.
struct Lanes {
  int g, c;             // fragment group id (lane / 4) and thread in group (lane % 4)
  int k_tok, k_chunk;   // K as the A operand of S^T = K Q^T (tokens x dims)
  int v_tok, v_chunk;   // V^T as the A operand of O^T = V^T P^T, via ldmatrix.trans
  __device__ __forceinline__ explicit Lanes(int lane) {
    g = lane >> 2;
    c = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    k_tok = (mi & 1) * 8 + rr;
    k_chunk = mi >> 1;
    v_tok = (mi >> 1) * 8 + rr;
    v_chunk = mi & 1;
  }
};

// Running state of one warp for up to 8*NT query rows. o holds O^T fragments:
// o[mt][nt][0/1] = (dim 16mt + g, rows nt*8 + 2c, +1), [2/3] = dim + 8.
template <int NT>
struct RowState {
  float o[8][NT][4];
  float m[NT][2], l[NT][2];  // rows nt*8 + 2c + e; l is a per-lane partial sum
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m[nt][e] = -INFINITY;
        l[nt][e] = 0.f;
      }
  }
  // Sum each row's partial l over the 8 lanes that share it.
  __device__ __forceinline__ void reduce_l() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], off);
  }
};

// S^T = K . Q^T, masking, online softmax, O^T += V^T . P^T for one block.
// kt / vt: shared addresses of the block's K and V tiles. qb: Q^T B-operand
// fragments (qb[kk][nt][0] = row nt*8+g, dims 16kk+2c,+1; [1] = dims +8).
// limit[nt][e]: last visible position of row nt*8+2c+e (-1: row unused).
template <int NT>
__device__ __forceinline__ void attend_block(uint32_t kt, uint32_t vt, const uint32_t (&qb)[8][NT][2],
                                             const int (&limit)[NT][2], int tok0, float scale_log2,
                                             const Lanes& ln, RowState<NT>& st) {
  // S^T (16 tokens x 8*NT rows) = K (16 x 128) . Q^T (128 x 8*NT)
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t a[4];
    ldsm_x4(kt + tile_off(ln.k_tok, 2 * kk + ln.k_chunk), a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
  }

  // Scale to base-2 units and mask. sc[nt][0/1]: token g, rows 2c/2c+1;
  // sc[nt][2/3]: token g+8, same rows.
  float bmax[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int lim = limit[nt][e];
      const float s0 = (tok0 + ln.g <= lim) ? sc[nt][e] * scale_log2 : -INFINITY;
      const float s1 = (tok0 + ln.g + 8 <= lim) ? sc[nt][e + 2] * scale_log2 : -INFINITY;
      sc[nt][e] = s0;
      sc[nt][e + 2] = s1;
      bmax[nt][e] = fmaxf(s0, s1);
    }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        bmax[nt][e] = fmaxf(bmax[nt][e], __shfl_xor_sync(0xffffffffu, bmax[nt][e], off));

  // Online softmax update. P enters the MMA as a sum of two bf16 parts,
  // p = hi + lo (hi = bf16(p), lo = bf16(p - hi)), so the weights carry about
  // 16 mantissa bits: a single bf16 rounding of p (2^-9 relative) can cost
  // more than the output tolerance when a short context's weighted V rows
  // cancel.
  uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float alpha[2], pr[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m_new = fmaxf(st.m[nt][e], bmax[nt][e]);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[e] = fast_exp2(st.m[nt][e] - m_use);
      st.m[nt][e] = m_new;
      pr[e] = fast_exp2(sc[nt][e] - m_use);
      pr[e + 2] = fast_exp2(sc[nt][e + 2] - m_use);
    }
    const uint32_t x0 = pack_bf16x2(pr[0], pr[1]);  // token g,   rows 2c, 2c+1
    const uint32_t x1 = pack_bf16x2(pr[2], pr[3]);  // token g+8, rows 2c, 2c+1
    const uint32_t y0 = pack_bf16x2(pr[0] - bf16_lo(x0), pr[1] - bf16_hi(x0));
    const uint32_t y1 = pack_bf16x2(pr[2] - bf16_lo(x1), pr[3] - bf16_hi(x1));
    st.l[nt][0] = alpha[0] * st.l[nt][0] + (pr[0] + pr[2]);
    st.l[nt][1] = alpha[1] * st.l[nt][1] + (pr[1] + pr[3]);
    pb[nt][0] = movmatrix_trans(x0);  // P^T (hi): tokens 2c, 2c+1 of row g
    pb[nt][1] = movmatrix_trans(x1);  // P^T (hi): tokens 8+2c, 9+2c of row g
    pl[nt][0] = movmatrix_trans(y0);  // P^T (lo)
    pl[nt][1] = movmatrix_trans(y1);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.o[mt][nt][0] *= alpha[0];
      st.o[mt][nt][1] *= alpha[1];
      st.o[mt][nt][2] *= alpha[0];
      st.o[mt][nt][3] *= alpha[1];
    }
  }

  // O^T (128 dims x 8*NT rows) += V^T (128 x 16 tokens) . P^T (16 x 8*NT)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(vt + tile_off(ln.v_tok, 2 * mt + ln.v_chunk), a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_bf16_16816(st.o[mt][nt], a, pb[nt][0], pb[nt][1]);
      mma_bf16_16816(st.o[mt][nt], a, pl[nt][0], pl[nt][1]);
    }
  }
}

}  // namespace pa
