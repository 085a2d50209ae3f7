// Paged decode / verify attention, bf16, W warps per work item (sm_103a).
//
// A work item is one fixed-size context split of one (sequence, KV head, row
// group): every query row that reads this KV head (the query-head group for
// decode, (k+1) x group rows for verify) over at most `split_tokens` tokens
// ("From 183 ms to 19 ms per decode step", sections "1. Grouped attention",
// "3. A Triton paged-decode kernel", "Then speculative decoding got slower").
// The split size is fixed, so a sequence's result depends on its own length
// only, never on its batch-mates. Each CTA of W warps owns one item; block j
// of the item goes to warp j % W, and the W running states are combined at
// the end.
//
// Staging. Each warp reads its 16-token blocks, K and V (8 KiB, two
// contiguous 4 KiB tiles of the head-major cache: "2. Head-major KV cache"),
// with 16-byte non-caching loads, PF of its blocks ahead, into registers.
// Before use a block is stored into the warp's shared-memory slot in the
// swizzled tile layout and consumed by the shared tensor-core step
// (mma_tile.cuh). Plain loads were
// chosen over TMA bulk-tensor copies by measurement: on these scattered 4 KiB
// tiles the TMA and cp.async paths both level off near 4.7 TB/s on GB300,
// while 16-byte loads into registers reach about 5.4 TB/s.
//
// Masking happens while staging: rows of a partial last block are stored as
// zeros (a zero key is not neutral in the scores, so those positions are also
// masked to -inf; zero V rows keep 0 x stale = 0: "A Rust inference server for
// Qwen2 on Apple Silicon", Day 3 "Known gaps").
//
// Fused verify: positions of the new tokens are read from k_new / v_new
// instead of the cache, and the row-group-0 item that holds them writes them
// to the cache, so no item depends on another's write.
//
// Epilogue: the W warps' states are combined in shared memory (element-wise
// per lane: the fragment layout is the same in every warp); one split writes
// the output; otherwise the item writes its normalised partial and
// log-sum-exp, and merge_kernel, launched as a programmatic dependent,
// combines the splits.
#include "mma_tile.cuh"

namespace pa {

cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream);

__device__ __forceinline__ uint4 ld_stream(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

template <int NT, int W>
struct LdgCfg {
  static constexpr int kCombWords = 32 * NT + 4 * NT;  // o fragments, then m, l, per lane
  static constexpr int kSlots = W * kBlockBytes;
  static constexpr int kComb = W * kCombWords * 32 * 4;
  static constexpr int kBytes = kSlots > kComb ? kSlots : kComb;
};

// Register budget: K+V of PF blocks in flight (64 registers each) plus the
// attention state; it sets the warps resident per SM (12 for NT = PF = 1,
// 8 otherwise), hence the CTAs per SM for W warps each.
template <int NT, int PF, int W>
__global__ void __launch_bounds__(32 * W, ((NT == 1 && PF == 1) ? 12 : 8) / W)
    attn_ldg_kernel(const AttnParams p) {
  using C = LdgCfg<NT, W>;
  __shared__ __align__(1024) uint8_t smem[C::kBytes];
  __shared__ int s_ids[kMaxSplitTokens / kBlockSize];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* slot = smem + warp * kBlockBytes;

  const int units = p.batch * p.kv_heads * p.row_groups;
  const int item = blockIdx.x;
  const int split = item / units;
  const int unit = item - split * units;
  const int rg = unit % p.row_groups;
  const int bh = unit / p.row_groups;
  const int h = bh % p.kv_heads, b = bh / p.kv_heads;
  int L = __ldg(p.context_lens + b);
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0 && rg == 0) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    L = L < 0 ? 0 : cap;
  }
  const int ssize = split_for(p, L);
  const int nsplit = (L + ssize - 1) / ssize;
  if (split >= max(nsplit, 1)) return;  // uniform across the CTA
  const int row0 = rg * p.rows_per_cta;
  const int nrows = min(p.rows_per_cta, p.rows - row0);
  const int t0 = split * ssize;
  const int t1 = min(L, t0 + ssize);
  const int nblk = (t1 - t0 + kBlockSize - 1) / kBlockSize;
  const int new0 = L - p.num_queries;  // first position of a new (verify) token
  const bool fused = p.fused_write != 0;

  // Block ids of the split (a bad id reads zeros and raises a flag).
  for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
    int id = __ldg(p.block_tables + int64_t(b) * p.mbps + t0 / kBlockSize + j);
    if (id < 0 || id >= p.num_blocks) {
      raise_flag(p.status, PA_FLAG_BAD_BLOCK);
      id = -1;
    }
    s_ids[j] = id;
  }

  const Lanes ln(lane);
  // Q^T as the B operand: qb[kk][nt][0] = row nt*8+g, dims 16kk+2c,+1; [1] = dims +8.
  uint32_t qb[8][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = nt * 8 + ln.g;
    const bool live = r < nrows;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                             row_offset(p, int64_t(b) * p.num_queries, h, row0 + (live ? r : 0)));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qb[kk][nt][0] = live ? __ldg(qrow + kk * 8 + ln.c) : 0u;
      qb[kk][nt][1] = live ? __ldg(qrow + kk * 8 + 4 + ln.c) : 0u;
    }
  }
  int limit[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = nt * 8 + 2 * ln.c + e;
      limit[nt][e] = r < nrows ? row_limit(p, L, p.num_queries, row0 + r) : -1;
    }
  __syncthreads();  // block ids visible

  const uint16_t* kc = static_cast<const uint16_t*>(p.k_cache);
  const uint16_t* vc = static_cast<const uint16_t*>(p.v_cache);
  const uint16_t* kn = static_cast<const uint16_t*>(p.k_new);
  const uint16_t* vn = static_cast<const uint16_t*>(p.v_new);
  // Lane roles while staging: chunk e*32 + lane of a 4 KiB tile is token row
  // 2e + lane/16, 16-byte chunk lane%16 (each instruction reads 512
  // contiguous bytes of one tile).
  const int col = lane & 15, row_lo = lane >> 4;

  // Read block j into registers: v[0..7] K chunks, v[8..15] V chunks. Rows
  // past the context are zeros; new (verify) positions come from the inputs.
  auto load_block = [&](int j, uint4 (&v)[16]) {
    const int tok0 = t0 + j * kBlockSize;
    const int valid = min(kBlockSize, L - tok0);
    const int id = s_ids[j];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int row = 2 * e + row_lo;
      const int pos = tok0 + row;
      uint4 k4 = make_uint4(0, 0, 0, 0), v4 = make_uint4(0, 0, 0, 0);
      if (row < valid) {
        // A new (verify) token is read from the inputs when its slot is the
        // table slot of its position; otherwise the pool's row stays (a
        // negative slot is not written).
        const bool from_new =
            fused && pos >= new0 && id >= 0 &&
            __ldg(p.slot_mapping + b * p.num_queries + (pos - new0)) == id * kBlockSize + row;
        if (from_new) {
          const int64_t src = (int64_t(b * p.num_queries + (pos - new0)) * p.kv_heads + h) * kHeadDim + col * 8;
          k4 = __ldg(reinterpret_cast<const uint4*>(kn + src));
          v4 = __ldg(reinterpret_cast<const uint4*>(vn + src));
        } else if (id >= 0) {
          const int64_t src = ((int64_t(h) * p.num_blocks + id) * kBlockSize + row) * kHeadDim + col * 8;
          k4 = ld_stream(kc + src);
          v4 = ld_stream(vc + src);
        }
      }
      v[e] = k4;
      v[8 + e] = v4;
    }
  };

  // Store block j into this warp's slot; the row-group-0 item also writes the
  // verify step's new rows to the cache.
  auto store_block = [&](int j, const uint4 (&v)[16]) {
    const int tok0 = t0 + j * kBlockSize;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int row = 2 * e + row_lo;
      *reinterpret_cast<uint4*>(slot + tile_off(row, col)) = v[e];
      *reinterpret_cast<uint4*>(slot + kTileBytes + tile_off(row, col)) = v[8 + e];
    }
    if (fused && rg == 0 && tok0 + kBlockSize > new0) {
      const int valid = min(kBlockSize, L - tok0);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int row = 2 * e + row_lo;
        const int pos = tok0 + row;
        if (row < valid && pos >= new0) {
          const int s_id = __ldg(p.slot_mapping + b * p.num_queries + (pos - new0));
          if (s_id >= 0 && s_id < p.num_blocks * kBlockSize) {
            const int64_t dst =
                ((int64_t(h) * p.num_blocks + s_id / kBlockSize) * kBlockSize + s_id % kBlockSize) * kHeadDim +
                col * 8;
            const int64_t src = (int64_t(b * p.num_queries + (pos - new0)) * p.kv_heads + h) * kHeadDim + col * 8;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_cache_w) + dst) = __ldg(reinterpret_cast<const uint4*>(kn + src));
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_cache_w) + dst) = __ldg(reinterpret_cast<const uint4*>(vn + src));
          } else if (s_id >= 0 && col == 0) {
            raise_flag(p.status, PA_FLAG_BAD_SLOT);
          }
        }
      }
    }
  };

  // This warp's blocks: j = warp + k*W, k < mine.
  const int mine = nblk > warp ? (nblk - warp + W - 1) / W : 0;
  RowState<NT> st;
  st.reset();
  const uint32_t kt = smem_u32(slot), vt = kt + kTileBytes;
  uint4 buf[PF][16];
#pragma unroll
  for (int u = 0; u < PF; ++u)
    if (u < mine) load_block(warp + u * W, buf[u]);
  for (int k0 = 0; k0 < mine; k0 += PF) {
#pragma unroll
    for (int u = 0; u < PF; ++u) {
      const int k = k0 + u;
      if (k < mine) {
        const int j = warp + k * W;
        __syncwarp();  // the previous block's reads of the slot are done
        store_block(j, buf[u]);
        __syncwarp();  // the slot is visible to every lane
        if (k + PF < mine) load_block(warp + (k + PF) * W, buf[u]);
        attend_block<NT>(kt, vt, qb, limit, t0 + j * kBlockSize, p.scale_log2, ln, st);
      }
    }
  }
  st.reduce_l();

  // Combine the W states (lane-major words: conflict-free); warp w then
  // finishes m-tiles [w*8/W, (w+1)*8/W).
  float* comb = reinterpret_cast<float*>(smem);
  __syncthreads();  // every slot read is done before the buffer is reused
  {
    float* mine_w = comb + warp * C::kCombWords * 32 + lane;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) mine_w[((mt * NT + nt) * 4 + e) * 32] = st.o[mt][nt][e];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mine_w[(32 * NT + nt * 2 + e) * 32] = st.m[nt][e];
        mine_w[(34 * NT + nt * 2 + e) * 32] = st.l[nt][e];
      }
  }
  __syncthreads();
  float M[NT][2], l_tot[NT][2], f[W][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w) mx = fmaxf(mx, comb[(w * C::kCombWords + 32 * NT + nt * 2 + e) * 32 + lane]);
      M[nt][e] = mx;
      float lt = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float mw = comb[(w * C::kCombWords + 32 * NT + nt * 2 + e) * 32 + lane];
        f[w][nt][e] = (mx == -INFINITY) ? 0.f : fast_exp2(mw - mx);
        lt += f[w][nt][e] * comb[(w * C::kCombWords + 34 * NT + nt * 2 + e) * 32 + lane];
      }
      l_tot[nt][e] = lt;
    }
  const bool single = nsplit <= 1;
  const size_t pslot = size_t(unit) * p.max_splits + split;
  constexpr int kMtPerWarp = 8 / W;
#pragma unroll
  for (int q2 = 0; q2 < kMtPerWarp; ++q2) {
    const int mt = warp * kMtPerWarp + q2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ee = e & 1;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) acc += f[w][nt][ee] * comb[(w * C::kCombWords + (mt * NT + nt) * 4 + e) * 32 + lane];
        const float val = l_tot[nt][ee] > 0.f ? acc / l_tot[nt][ee] : 0.f;
        const int r = nt * 8 + 2 * ln.c + ee;
        const int d = mt * 16 + ln.g + (e >> 1) * 8;
        if (r < nrows) {
          if (single) {
            uint16_t* dst = static_cast<uint16_t*>(p.out) + row_offset(p, int64_t(b) * p.num_queries, h, row0 + r) + d;
            *dst = uint16_t(pack_bf16x2(val, 0.f) & 0xffffu);
          } else {
            p.part_o[(pslot * kRowSlots + r) * kHeadDim + d] = val;
          }
        }
      }
  }
  if (!single && warp == 0 && ln.g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = nt * 8 + 2 * ln.c + e;
        if (r < nrows)
          p.part_lse[pslot * kRowSlots + r] = l_tot[nt][e] > 0.f ? M[nt][e] + __log2f(l_tot[nt][e]) : -INFINITY;
      }
  }
  pdl_launch_dependents();
}

template <int NT, int PF>
static void launch_w(const AttnParams& p, int warps, unsigned grid, cudaStream_t stream) {
  if (warps >= 4)
    attn_ldg_kernel<NT, PF, 4><<<grid, 128, 0, stream>>>(p);
  else if (warps == 2)
    attn_ldg_kernel<NT, PF, 2><<<grid, 64, 0, stream>>>(p);
  else
    attn_ldg_kernel<NT, PF, 1><<<grid, 32, 0, stream>>>(p);
}

// Host entry. p.rows_per_cta must be 16; NT = 1 serves up to 8 rows per
// (sequence, KV head), NT = 2 up to 16 (more rows use several row groups).
// prefetch: blocks each warp keeps in flight (1 or 2; 2 only with NT = 1).
// warps: warps per work item (1, 2 or 4).
cudaError_t launch_attn_ldg(const AttnParams& p, int prefetch, int warps, cudaStream_t stream) {
  const int64_t items = int64_t(p.batch) * p.kv_heads * p.row_groups * p.max_splits;
  if (items <= 0) return cudaSuccess;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const unsigned grid = unsigned(items);
  if (p.rows > 8)
    launch_w<2, 1>(p, warps, grid, stream);
  else if (prefetch >= 2)
    launch_w<1, 2>(p, warps, grid, stream);
  else
    launch_w<1, 1>(p, warps, grid, stream);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.max_splits <= 1) return e;
  return launch_merge(p, stream);
}

}  // namespace pa
