// Paged prefill attention, bf16, tensor-core products (sm_103a).
//
// A prefill (or chunked-prefill) step attends every token of a prompt chunk
// to the sequence's cache, causally: token i of an n-token chunk sits at
// position L - n + i and sees positions t <= L - n + i ("From 183 ms to 19 ms
// per decode step", section "What's next": paged prefill; the causal form is
// the plain masked softmax of "Anatomy of a Decode-Step Stall",
// Model._layer, with many query rows). The chunk's own K/V are in the cache
// already (written by pa_cache_write), so a chunk is read in place through
// its block table like any other context.
//
// Decode gives each (sequence, KV head) one 16-row group; a chunk has
// n x group rows, and one CTA per 16 rows would read the context once per
// group. Here one CTA takes 128 rows (8 consumer warps x 16 rows, token-major
// rows r = i * group + g) of one (sequence, KV head), and every K/V block the
// producer stages is consumed by all eight warps: each block is read from HBM
// once per 128 rows. The per-warp step is the decode kernels' tensor-core
// block step (csrc/mma_tile.cuh) with 16 rows. A warp skips the blocks that
// lie wholly after its rows' causal limits, but still releases them.
//
// The last block of a context may hold rows past the context, which can be
// anything (NaN included); before the consumers read it, the producer warp
// zeroes those V rows (a zero weight times a stale V must stay zero).
#include "mma_tile.cuh"

namespace pa {

constexpr int kPfWarps = 8;                 // consumer warps, 16 query rows each
constexpr int kPfRows = kPfWarps * 16;      // query rows per CTA
constexpr int kPfStages = 6;
constexpr int kPfThreads = (kPfWarps + 1) * 32;

struct PfSmem {
  static constexpr int stages = 0;
  static constexpr int bars = kPfStages * kBlockBytes;   // full[S], empty[S], tail
  static constexpr int total = bars + (2 * kPfStages + 1) * 8;
  static constexpr int alloc = total + 1024;
};
static_assert(kPfWarps * 16 * kHeadDim * 2 <= kPfStages * kBlockBytes, "output staging must fit the ring");

__global__ void __launch_bounds__(kPfThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t bar_full = base + PfSmem::bars;
  const uint32_t bar_empty = bar_full + kPfStages * 8;
  const uint32_t bar_tail = bar_empty + kPfStages * 8;  // last block's stale V rows zeroed

  const int b = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == kPfWarps * 32) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  int q0, nq;
  seq_queries(p, b, blockIdx.x == 0 && h == 0, &q0, &nq);
  int L = __ldg(p.context_lens + b);
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  if (L < 0 || L > cap) {
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    L = L < 0 ? 0 : cap;
  }
  const int rows_b = nq * p.group;
  const int row0 = blockIdx.x * kPfRows;
  if (row0 >= rows_b) return;
  const int nrows = min(kPfRows, rows_b - row0);
  // Positions the CTA's last row may see; every earlier row sees fewer.
  const int kv_end = max(0, min(L, L - nq + (row0 + nrows - 1) / p.group + 1));
  const int nblk = (kv_end + kBlockSize - 1) / kBlockSize;
  const int tail_valid = kv_end - (nblk - 1) * kBlockSize;  // rows of the last block inside the context

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kPfWarps);
    }
    mbar_init(bar_tail, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Consumer state at function scope: the output is written after the join.
  const int wrow0 = row0 + warp * 16;
  const int wrows = warp < kPfWarps ? max(0, min(16, rows_b - wrow0)) : 0;
  RowState<2> st;
  st.reset();
  const Lanes ln(lane);
  bool timed_out = false;
  int issued = 0;
  if (warp == kPfWarps) {
    // ---------------- producer (the whole warp) ----------------
    // Block ids come 32 at a time, one per lane, the next chunk loaded while
    // the current one is issued; lane 0 issues the TMA loads.
    const uint64_t policy = policy_evict_first();
    const int32_t* table = p.block_tables + int64_t(b) * p.mbps;
    int ids = lane < nblk ? __ldg(table + lane) : 0;
    for (int c0 = 0; c0 < nblk && !timed_out; c0 += 32) {
      const int next = (c0 + 32 + lane < nblk) ? __ldg(table + c0 + 32 + lane) : 0;
      const int n = min(32, nblk - c0);
      for (int k = 0; k < n; ++k) {
        const int j = c0 + k;
        int id = __shfl_sync(0xffffffffu, ids, k);
        if (lane == 0) {
          const int s = j % kPfStages, ph = j / kPfStages;
          if (ph > 0 && !mbar_wait(bar_empty + 8 * s, (ph - 1) & 1, p.wait_limit_ns)) {
            timed_out = true;
          } else {
            if (id < 0 || id >= p.num_blocks) {
              raise_flag(p.status, PA_FLAG_BAD_BLOCK);
              id = -1;
            }
            const uint32_t stg = base + PfSmem::stages + s * kBlockBytes;
            const uint32_t fb = bar_full + 8 * s;
            const int y = id >= 0 ? id * kBlockSize : -kBlockSize;
            mbar_arrive_expect_tx(fb, kBlockBytes);
            tma_load_3d(stg, &tmap_k, 0, y, h, fb, policy);
            tma_load_3d(stg + kHalfTile, &tmap_k, 64, y, h, fb, policy);
            tma_load_3d(stg + kTileBytes, &tmap_v, 0, y, h, fb, policy);
            tma_load_3d(stg + kTileBytes + kHalfTile, &tmap_v, 64, y, h, fb, policy);
            issued = j + 1;
          }
        }
        timed_out = __shfl_sync(0xffffffffu, timed_out, 0);
        if (timed_out) break;
      }
      ids = next;
    }
    // Zero the last block's V rows past the context once it has landed.
    if (!timed_out && nblk > 0) {
      const int j = nblk - 1, s = j % kPfStages;
      if (tail_valid < kBlockSize) {
        if (__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (j / kPfStages) & 1, p.wait_limit_ns))) {
          uint8_t* vt = sbase + PfSmem::stages + s * kBlockBytes + kTileBytes;
          for (int e = lane; e < (kBlockSize - tail_valid) * 16; e += 32) {
            const int t = tail_valid + (e >> 4), ch = e & 15;
            *reinterpret_cast<uint4*>(vt + tile_off(t, ch)) = make_uint4(0, 0, 0, 0);
          }
        } else {
          timed_out = true;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tail);
    }
    if (timed_out && lane == 0) {
      raise_flag(p.status, PA_FLAG_TIMEOUT);
      // Let the loads already issued land (bounded) before the CTA can leave.
      for (int j = max(0, issued - kPfStages); j < issued; ++j)
        (void)mbar_wait(bar_full + 8 * (j % kPfStages), (j / kPfStages) & 1);
    }
  } else {
    // ---------------- consumers: warp w owns rows row0 + 16w .. +15 ----------------
    const int g = ln.g, c = ln.c;
    uint32_t qb[8][2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = nt * 8 + g;
      const bool live = r < wrows;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                               row_offset(p, q0, h, wrow0 + (live ? r : 0)));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][nt][0] = live ? __ldg(qrow + kk * 8 + c) : 0u;
        qb[kk][nt][1] = live ? __ldg(qrow + kk * 8 + 4 + c) : 0u;
      }
    }
    int limit[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = nt * 8 + 2 * c + e;
        limit[nt][e] = r < wrows ? row_limit(p, L, nq, wrow0 + r) : -1;
      }
    // The warp's last visible position: blocks after it are skipped.
    const int wlast = wrows > 0 ? row_limit(p, L, nq, wrow0 + wrows - 1) : -1;
    for (int j = 0; j < nblk; ++j) {
      const int s = j % kPfStages;
      if (!mbar_wait(bar_full + 8 * s, (j / kPfStages) & 1, p.wait_limit_ns) ||
          (j == nblk - 1 && !mbar_wait(bar_tail, 0, p.wait_limit_ns))) {
        timed_out = true;
        break;
      }
      if (j * kBlockSize <= wlast) {
        const uint32_t kt = base + PfSmem::stages + s * kBlockBytes;
        attend_block<2>(kt, kt + kTileBytes, qb, limit, j * kBlockSize, p.scale_log2, ln, st);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (timed_out && lane == 0) raise_flag(p.status, PA_FLAG_TIMEOUT);
    st.reduce_l();
  }
  __syncthreads();  // every warp is done with the ring: it becomes the output staging area
  if (warp == kPfWarps) return;

  // Normalise (rows that see nothing, at a negative position, give zeros),
  // stage this warp's 16 rows as bf16 [16][128], write them in 16-byte pieces.
  const int g = ln.g, c = ln.c;
  float inv[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) inv[nt][e] = st.l[nt][e] > 0.f ? 1.f / st.l[nt][e] : 0.f;
  uint16_t* stage = reinterpret_cast<uint16_t*>(sbase + PfSmem::stages) + warp * 16 * kHeadDim;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = nt * 8 + 2 * c, d = mt * 16 + g;
      const uint32_t lo = pack_bf16x2(st.o[mt][nt][0] * inv[nt][0], st.o[mt][nt][2] * inv[nt][0]);  // row r: d, d+8
      const uint32_t hi = pack_bf16x2(st.o[mt][nt][1] * inv[nt][1], st.o[mt][nt][3] * inv[nt][1]);  // row r+1
      stage[r * kHeadDim + d] = uint16_t(lo & 0xffffu);
      stage[r * kHeadDim + d + 8] = uint16_t(lo >> 16);
      stage[(r + 1) * kHeadDim + d] = uint16_t(hi & 0xffffu);
      stage[(r + 1) * kHeadDim + d + 8] = uint16_t(hi >> 16);
    }
  __syncwarp();
  for (int e = lane; e < wrows * (kHeadDim / 8); e += 32) {
    const int r = e / (kHeadDim / 8), ch = e % (kHeadDim / 8);
    uint16_t* dst = static_cast<uint16_t*>(p.out) + row_offset(p, q0, h, wrow0 + r) + ch * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(stage + r * kHeadDim + ch * 8);
  }
}

cudaError_t launch_attn_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, dim3 grid,
                                cudaStream_t stream) {
  static PerDeviceOnce once;
  const cudaError_t e = once.run([](int) {
    return cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem::alloc);
  });
  if (e != cudaSuccess) return e;
  attn_prefill_kernel<<<grid, kPfThreads, PfSmem::alloc, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace pa
