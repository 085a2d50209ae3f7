// Paged decode / verify attention over an int8 KV pool, dequantisation fused
// (sm_103a).
//
// The int8 pool stores symmetric codes as bytes with one fp32 scale per
// (head, block, channel) for K and per (head, block, row) for V ("A Rust
// inference server for Qwen2 on Apple Silicon", Day 4). The page's own
// measurement lost throughput because it dequantised on the gather; its
// stated fix is to dequantise inside the attention kernel, which this kernel
// does: the bytes and scales are staged in shared memory and turned into
// tensor-core fragments in registers (csrc/q8.cuh), so HBM carries 4,672
// bytes per 16-token block and head instead of bf16's 8,192.
//
// Work split and warp roles as in the bf16 kernel: one CTA per (context
// split, KV head, sequence x row group) with the whole query-head group
// ("From 183 ms to 19 ms per decode step", sections "1. Grouped attention"
// and "3. A Triton paged-decode kernel"); warp 2 is the producer, issuing
// four TMA loads per block (K bytes, V bytes, K scales, V scales) into an
// mbarrier ring; warps 0..1 consume blocks round-robin.
//
// Verify. A block that receives a new row is requantised as a whole (its K
// scales span the block), so its reader must see the rewritten block. With
// one row group per (sequence, KV head) this CTA is that block's only reader:
// once the block has landed, the producer warp dequantises its K rows,
// inserts the new rows, requantises, quantises the new V rows and writes the
// block back to the pool (q8_fuse_new_rows); the consumer that owns the block
// attends over it after that. With several row groups,
// pa_verify runs the quantised append first and this kernel as its
// programmatic dependent; the producer then streams the blocks before the new
// tokens at once and waits for the append grid only before the first block
// that holds one.
#include "q8.cuh"

namespace pa {

constexpr int kQ8Consumers = 2;
constexpr int kQ8Stages = 8;
constexpr int kQ8Threads = (kQ8Consumers + 1) * 32;
static_assert(kQ8Stages % (2 * kQ8Consumers) == 0,
              "every phase of a stage must go to one warp: stages must be a multiple of 2 x consumers");

struct Q8Smem {
  static constexpr int stages = 0;
  static constexpr int bars = kQ8Stages * kQ8StageBytes;  // full[S], empty[S], fixed[2]
  static constexpr int ids = bars + (2 * kQ8Stages + 2) * 8;
  static constexpr int ml = ids + (kMaxSplitTokens / kBlockSize) * 4;
  static constexpr int flag = ml + 2 * kQ8Consumers * kRowSlots * 4;
  static constexpr int total = flag + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(kQ8Consumers * kRowSlots * kCombineStride * 4 <= kQ8Stages * kQ8StageBytes,
              "cross-warp buffer must fit in the stage ring");

struct Q8Maps {
  CUtensorMap k, v, ks, vs;
};

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}

// Requantise, in a stage and in the pool, the block at position tok0 for the
// new tokens it holds (this sequence's tokens at positions >= new0), exactly
// as the quantised append does; run by the whole producer warp. Lane l owns
// channels 4l..4l+3; lane t < 16 brings the slot of position tok0 + t (any
// value where that position holds no new token). A token whose slot is
// negative is not written (as in the append); a slot that is not the table
// slot of its position is a caller error: it raises PA_FLAG_BAD_SLOT and the
// token is not written.
//
// This runs once per launch in a few CTAs, late, while the other CTAs stream
// at the full memory rate, so nearly all of its time goes to first touches:
// its own instructions and the new rows. It is therefore written as short
// rolled loops (a 16-way unrolled form measured 15 us on a 32k-context step,
// of which 12 us disappeared when the same call was repeated), and the
// producer loads the slots and prefetches the new rows into L1 when the CTA
// starts. Out of line: its registers stay out of the consumers' budget.
__device__ __noinline__ void q8_fuse_new_rows(const AttnParams& p, const CtaWork& w, uint8_t* stp, int id,
                                              int tok0, int slot_in, int lane) {
  const int new0 = w.L - w.nq;
  const int lo = max(tok0, new0), hi = min(tok0 + kBlockSize, w.L);
  const bool in_pool = id >= 0 && id < p.num_blocks;
  // Row t of this block is new token (tok0 + t - new0); only rows in [lo, hi)
  // are ever read.
  const int64_t row_step = int64_t(p.kv_heads) * kHeadDim;
  const int64_t first = (int64_t(w.q0) + (tok0 - new0)) * row_step + int64_t(w.h) * kHeadDim;
  const uint16_t* knew = static_cast<const uint16_t*>(p.k_new) + first;
  const uint16_t* vnew = static_cast<const uint16_t*>(p.v_new) + first;

  const int pos = tok0 + lane;
  const bool is_new = lane < kBlockSize && pos >= lo && pos < hi;
  const int slot = is_new ? slot_in : -1;
  const bool ok = is_new && slot >= 0 && in_pool && slot == id * kBlockSize + lane;
  const uint32_t rows = __ballot_sync(0xffffffffu, ok);
  if (__any_sync(0xffffffffu, is_new && slot >= 0 && !ok) && lane == 0) raise_flag(p.status, PA_FLAG_BAD_SLOT);
  if (rows == 0) return;

  const int chunk = lane >> 2, within = (lane & 3) * 4;
  float* ks = reinterpret_cast<float*>(stp + kQ8KsOff);
  float* vs = reinterpret_cast<float*>(stp + kQ8VsOff);
  const int64_t blk = int64_t(w.h) * p.num_blocks + id;
  uint8_t* kpool = static_cast<uint8_t*>(p.k_cache_w) + blk * kQ8TileBytes;
  uint8_t* vpool = static_cast<uint8_t*>(p.v_cache_w) + blk * kQ8TileBytes;
  float* kspool = static_cast<float*>(p.k_scale_w) + blk * kHeadDim;
  float* vspool = static_cast<float*>(p.v_scale_w) + blk * kBlockSize;
  const uint16_t* kmine = knew + 4 * lane;
  const uint16_t* vmine = vnew + 4 * lane;

  // K: this lane's 4 channels of row t, a new row or an old one dequantised
  // from the stage.
  const float4 s_old = *reinterpret_cast<const float4*>(ks + 4 * lane);
  const float so[4] = {s_old.x, s_old.y, s_old.z, s_old.w};
  auto k_row = [&](int t, float x[4]) {
    if (rows >> t & 1u) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(kmine + t * row_step));
      x[0] = bf16_lo(u.x);
      x[1] = bf16_hi(u.x);
      x[2] = bf16_lo(u.y);
      x[3] = bf16_hi(u.y);
    } else {
      const uint32_t b4 = *reinterpret_cast<const uint32_t*>(stp + kQ8KOff + q8_off(t, chunk) + within);
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = q8_value(b4 >> (8 * k) & 0xffu, so[k]);
    }
  };
  // Per-channel maxima over the block, then every row's codes at the new
  // scales (a lane rewrites only the 4 bytes of each row that it read).
  float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int t = 0; t < kBlockSize; ++t) {
    float x[4];
    k_row(t, x);
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], fabsf(x[k]));
  }
  float sn[4], inv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    sn[k] = q8_scale(m[k]);
    inv[k] = q8_inverse(m[k]);
  }
#pragma unroll 4
  for (int t = 0; t < kBlockSize; ++t) {
    float x[4];
    k_row(t, x);
    uint32_t bytes = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) bytes |= q8_code(x[k], inv[k]) << (8 * k);
    *reinterpret_cast<uint32_t*>(stp + kQ8KOff + q8_off(t, chunk) + within) = bytes;
    *reinterpret_cast<uint32_t*>(kpool + t * kHeadDim + 4 * lane) = bytes;
  }
  *reinterpret_cast<float4*>(ks + 4 * lane) = make_float4(sn[0], sn[1], sn[2], sn[3]);
  *reinterpret_cast<float4*>(kspool + 4 * lane) = make_float4(sn[0], sn[1], sn[2], sn[3]);

  // V: each new row on its own scale.
  for (uint32_t r = rows; r != 0u; r &= r - 1u) {
    const int t = __ffs(r) - 1;
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(vmine + t * row_step));
    const float v[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
    float mv = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    const float sc = q8_scale(mv), iv = q8_inverse(mv);
    uint32_t bytes = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) bytes |= q8_code(v[k], iv) << (8 * k);
    *reinterpret_cast<uint32_t*>(stp + kQ8VOff + q8_off(t, chunk) + within) = bytes;
    *reinterpret_cast<uint32_t*>(vpool + t * kHeadDim + 4 * lane) = bytes;
    if (lane == 0) {
      vs[t] = sc;
      vspool[t] = sc;
    }
  }
  __syncwarp();
}

// Register budget, by measurement on GB300: at 142 registers the 8-row
// instance ran a 32k-context call at 52 us against 36 us at 128 (the bound
// below; a few bytes of spill, in the out-of-line requantisation), and the
// 16-row instance ran verify at 62 us at 195 registers against 48.5 us at 168.
template <int NT>
__global__ void __launch_bounds__(kQ8Threads, NT == 1 ? 5 : 3)
    attn_q8_kernel(const __grid_constant__ Q8Maps maps, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  int32_t* s_ids = reinterpret_cast<int32_t*>(sbase + Q8Smem::ids);
  float* s_m = reinterpret_cast<float*>(sbase + Q8Smem::ml);
  float* s_l = s_m + kQ8Consumers * kRowSlots;
  int* s_flag = reinterpret_cast<int*>(sbase + Q8Smem::flag);
  const uint32_t bar_full = base + Q8Smem::bars;
  const uint32_t bar_empty = bar_full + kQ8Stages * 8;
  const uint32_t bar_fixed = bar_empty + kQ8Stages * 8;  // fused blocks requantised by the producer warp

  if (threadIdx.x == kQ8Consumers * 32) {
    prefetch_tensormap(&maps.k);
    prefetch_tensormap(&maps.v);
    prefetch_tensormap(&maps.ks);
    prefetch_tensormap(&maps.vs);
  }
  int L_raw;
  {
    const int b = blockIdx.y / p.row_groups;
    const int per = p.split_tokens / kBlockSize;
    const int j0 = blockIdx.z * per;
    const int jn = min(per, p.mbps - j0);
    L_raw = __ldg(p.context_lens + b);
    for (int j = threadIdx.x; j < jn; j += blockDim.x)
      s_ids[j] = __ldg(p.block_tables + int64_t(b) * p.mbps + j0 + j);
  }
  const CtaWork w = cta_work(p, L_raw);
  if (w.nrows <= 0) return;  // a ragged sequence with fewer query rows than this group
  if (w.split_size != p.split_tokens) {
    // A long sequence with its own split size: its entries start elsewhere.
    // Each thread rewrites the indices it wrote above, so no barrier is needed.
    const int b = blockIdx.y / p.row_groups;
    const int j0 = w.t0 / kBlockSize;
    const int jn = min(w.split_size / kBlockSize, p.mbps - j0);
    for (int j = threadIdx.x; j < jn; j += blockDim.x)
      s_ids[j] = __ldg(p.block_tables + int64_t(b) * p.mbps + j0 + j);
  }
  if (w.split >= w.nsplit) {
    if (w.L == 0 && w.split == 0) write_zero_rows<uint16_t>(p, w);
    return;
  }
  const int nblk = (w.t1 - w.t0 + kBlockSize - 1) / kBlockSize;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_flag[0] = s_flag[1] = s_flag[2] = s_flag[3] = 0;
    for (int s = 0; s < kQ8Stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_fixed, 1);
    mbar_init(bar_fixed + 8, 1);
    fence_mbar_init();
  }
  __syncthreads();

  RowState<NT> st;
  st.reset();
  const Lanes ln(lane);
  const int g = ln.g, c = ln.c;
  // With a fused write, the trailing blocks that hold new tokens (at most two,
  // since a single row group has at most 16 query tokens) are requantised by
  // the producer warp before their consumer attends over them.
  const int nmain =
      p.fused_write ? min(nblk, max(0, (w.L - w.nq - w.t0) / kBlockSize)) : nblk;

  if (warp == kQ8Consumers) {
    // ---------------- producer ----------------
    // The new tokens' slots and rows are needed only at the end of the split:
    // lane l loads the slot of position f0 + l (the fused blocks span at most
    // 32 positions) and brings that token's K and V rows into L1 now.
    const int f0 = w.t0 + nmain * kBlockSize;
    int fused_slot = -1;
    if (nmain < nblk) {
      const int new0 = w.L - w.nq, pos = f0 + lane;
      if (pos >= new0 && pos < w.t1) {
        fused_slot = __ldg(p.slot_mapping + w.q0 + (pos - new0));
        const int64_t row = (int64_t(w.q0 + pos - new0) * p.kv_heads + w.h) * kHeadDim;
        const uint16_t* kr = static_cast<const uint16_t*>(p.k_new) + row;
        const uint16_t* vr = static_cast<const uint16_t*>(p.v_new) + row;
        prefetch_l1(kr);
        prefetch_l1(kr + 64);
        prefetch_l1(vr);
        prefetch_l1(vr + 64);
      }
    }
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      const int new0 = w.L - w.nq;  // first position the append may have rewritten
      bool waited = !p.wait_append;
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kQ8Stages, n = j / kQ8Stages;
        if (n > 0 && !mbar_wait(bar_empty + 8 * s, (n - 1) & 1, p.wait_limit_ns)) {
          raise_flag(p.status, PA_FLAG_TIMEOUT);
          s_flag[2] = 1;
          break;
        }
        if (!waited && w.t0 + (j + 1) * kBlockSize > new0) {
          pdl_wait_primary();  // the append grid's writes to this block are visible after this
          waited = true;
        }
        const uint32_t stg = base + Q8Smem::stages + s * kQ8StageBytes;
        const uint32_t fb = bar_full + 8 * s;
        int id = s_ids[j];
        if (id < 0 || id >= p.num_blocks) {  // outside the pool: TMA reads zeros (scales 0)
          raise_flag(p.status, PA_FLAG_BAD_BLOCK);
          id = -1;
        }
        mbar_arrive_expect_tx(fb, kQ8BlockBytes);
        tma_load_3d(stg + kQ8KOff, &maps.k, 0, id >= 0 ? id * kBlockSize : -kBlockSize, w.h, fb, policy);
        tma_load_3d(stg + kQ8VOff, &maps.v, 0, id >= 0 ? id * kBlockSize : -kBlockSize, w.h, fb, policy);
        tma_load_3d(stg + kQ8KsOff, &maps.ks, 0, id, w.h, fb, policy);
        tma_load_3d(stg + kQ8VsOff, &maps.vs, 0, id, w.h, fb, policy);
        issued = j + 1;
      }
      s_flag[1] = issued;
    }
    __syncwarp();
    if (s_flag[1] == nblk) {
      for (int j = nmain; j < nblk; ++j) {
        const int s = j % kQ8Stages;
        // Every lane waits (each then sees the landed bytes); the warp goes on
        // only if all of them saw the phase complete.
        if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (j / kQ8Stages) & 1, p.wait_limit_ns))) {
          if (lane == 0) {
            raise_flag(p.status, PA_FLAG_TIMEOUT);
            s_flag[2] = 1;
          }
          break;
        }
        const int slot = __shfl_sync(0xffffffffu, fused_slot, (j - nmain) * kBlockSize + (lane & (kBlockSize - 1)));
        q8_fuse_new_rows(p, w, sbase + Q8Smem::stages + s * kQ8StageBytes, s_ids[j], w.t0 + j * kBlockSize,
                         slot, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_fixed + 8 * (j - nmain));
      }
    }
  } else {
    // ---------------- consumers ----------------
    uint32_t qb[8][NT][2];
    {
      int64_t off[NT];
      bool live[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + g;
        live[nt] = r < w.nrows;
        off[nt] = row_offset(p, w.q0, w.h, w.row0 + (live[nt] ? r : 0));
      }
      q8_load_q<NT>(static_cast<const uint16_t*>(p.q), off, live, c, qb);
    }
    int limit[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = nt * 8 + 2 * c + e;
        limit[nt][e] = r < w.nrows ? row_limit(p, w.L, w.nq, w.row0 + r) : -1;
      }

    // Blocks go in pairs (2p, 2p+1) to warp p % kQ8Consumers; a lone last
    // block is a pair of one. Every phase of a stage is consumed by the same
    // warp because kQ8Stages is a multiple of 2 * kQ8Consumers. Blocks from
    // nmain on (fused writes) are taken afterwards by the same owners, once
    // the producer warp has requantised them.
    bool timed_out = false;
    for (int pi = warp; 2 * pi < nmain; pi += kQ8Consumers) {
      const int j0 = 2 * pi;
      const bool two = j0 + 1 < nmain;
      const int s0 = j0 % kQ8Stages, s1 = (j0 + 1) % kQ8Stages;
      if (!mbar_wait(bar_full + 8 * s0, (j0 / kQ8Stages) & 1, p.wait_limit_ns) ||
          (two && !mbar_wait(bar_full + 8 * s1, ((j0 + 1) / kQ8Stages) & 1, p.wait_limit_ns))) {
        timed_out = true;
        break;
      }
      const uint8_t* p0 = sbase + Q8Smem::stages + s0 * kQ8StageBytes;
      const uint8_t* p1 = sbase + Q8Smem::stages + s1 * kQ8StageBytes;
      const uint32_t g0 = base + Q8Smem::stages + s0 * kQ8StageBytes;
      const uint32_t g1 = base + Q8Smem::stages + s1 * kQ8StageBytes;
      if (two) {
        const uint32_t stg[2] = {g0, g1};
        const float* const ks[2] = {reinterpret_cast<const float*>(p0 + kQ8KsOff),
                                    reinterpret_cast<const float*>(p1 + kQ8KsOff)};
        const float* const vs[2] = {reinterpret_cast<const float*>(p0 + kQ8VsOff),
                                    reinterpret_cast<const float*>(p1 + kQ8VsOff)};
        attend_blocks_q8<NT, 2>(stg, ks, vs, qb, limit, w.t0 + j0 * kBlockSize, p.scale_log2, ln, st);
      } else {
        const uint32_t stg[1] = {g0};
        const float* const ks[1] = {reinterpret_cast<const float*>(p0 + kQ8KsOff)};
        const float* const vs[1] = {reinterpret_cast<const float*>(p0 + kQ8VsOff)};
        attend_blocks_q8<NT, 1>(stg, ks, vs, qb, limit, w.t0 + j0 * kBlockSize, p.scale_log2, ln, st);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s0);
        if (two) mbar_arrive(bar_empty + 8 * s1);
      }
    }
    for (int j = nmain; j < nblk && !timed_out; ++j) {
      if ((j >> 1) % kQ8Consumers != warp) continue;
      const int s0 = j % kQ8Stages;
      if (!mbar_wait(bar_full + 8 * s0, (j / kQ8Stages) & 1, p.wait_limit_ns)) {
        timed_out = true;
        break;
      }
      if (!mbar_wait(bar_fixed + 8 * (j - nmain), 0, p.wait_limit_ns)) {
        timed_out = true;
        break;
      }
      const uint8_t* p0 = sbase + Q8Smem::stages + s0 * kQ8StageBytes;
      const uint32_t stg[1] = {base + Q8Smem::stages + s0 * kQ8StageBytes};
      const float* const ks[1] = {reinterpret_cast<const float*>(p0 + kQ8KsOff)};
      const float* const vs[1] = {reinterpret_cast<const float*>(p0 + kQ8VsOff)};
      attend_blocks_q8<NT, 1>(stg, ks, vs, qb, limit, w.t0 + j * kBlockSize, p.scale_log2, ln, st);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s0);
    }
    if (timed_out) {
      raise_flag(p.status, PA_FLAG_TIMEOUT);
      s_flag[2] = 1;
    }
    st.reduce_l();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (s_flag[2]) {
    if (threadIdx.x == 0) {
      const int issued = s_flag[1];
      for (int j = max(0, issued - kQ8Stages); j < issued; ++j)
        (void)mbar_wait(bar_full + 8 * (j % kQ8Stages), (j / kQ8Stages) & 1);
    }
    __syncthreads();
    return;
  }

  // Cross-warp combine. Accumulator tile mt holds dims 16mt + 2g (elements
  // 0, 1) and 16mt + 2g + 1 (elements 2, 3).
  float* cbuf = reinterpret_cast<float*>(sbase + Q8Smem::stages);
  if (warp < kQ8Consumers) {
    float* mine = cbuf + warp * kRowSlots * kCombineStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + 2 * c, d = mt * 16 + 2 * g;
        mine[r * kCombineStride + d] = st.o[mt][nt][0];
        mine[(r + 1) * kCombineStride + d] = st.o[mt][nt][1];
        mine[r * kCombineStride + d + 1] = st.o[mt][nt][2];
        mine[(r + 1) * kCombineStride + d + 1] = st.o[mt][nt][3];
      }
    if (g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s_m[warp * kRowSlots + nt * 8 + 2 * c + e] = st.m[nt][e];
          s_l[warp * kRowSlots + nt * 8 + 2 * c + e] = st.l[nt][e];
        }
    }
  }
  __syncthreads();
  split_epilogue<uint16_t>(p, w, cbuf, s_m, s_l, kQ8Consumers, s_flag);
}

template <int NT>
static cudaError_t launch_q8_nt(const Q8Maps& maps, const AttnParams& p, dim3 grid, bool after_append,
                                cudaStream_t stream) {
  static PerDeviceOnce once;
  const cudaError_t e = once.run([](int) {
    return cudaFuncSetAttribute(attn_q8_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Q8Smem::alloc);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kQ8Threads, 1, 1);
  cfg.dynamicSmemBytes = Q8Smem::alloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_append ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_q8_kernel<NT>, maps, p);
}

// Host entry. after_append: launched right behind the quantised append of
// the same call (verify), as its programmatic dependent.
cudaError_t launch_attn_q8(const Q8Maps& maps, const AttnParams& p, dim3 grid, bool after_append,
                           cudaStream_t stream) {
  return p.rows > 8 ? launch_q8_nt<2>(maps, p, grid, after_append, stream)
                    : launch_q8_nt<1>(maps, p, grid, after_append, stream);
}

}  // namespace pa
