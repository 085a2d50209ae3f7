// Paged prefill attention on the fifth-generation tensor cores (tcgen05), bf16.
//
// Same operation as attn_prefill.cu (causal attention of a prompt chunk over
// the sequence's paged cache: "From 183 ms to 19 ms per decode step", section
// "What's next"; the masked softmax of "Anatomy of a Decode-Step Stall",
// Model._layer). A work item is one row tile of one (sequence, KV head): the
// rows r = i * group + g of floor(128 / group) query tokens (rows_per_cta <=
// 128; the MMA's spare rows are zero). The products run as single-thread-
// issued tcgen05.mma with the accumulators in tensor memory:
//
//   S (128 rows x 64 positions, fp32)  = Q . K^T   A = Q in shared memory,  B = K tile in shared memory
//   O (128 rows x 128 dims, fp32)     += P . V     A = P in tensor memory, B = V tile in shared memory
//
// Tensor memory (256 columns of 128 lanes, lane = query row): O in columns
// 0..127, S in 128..191, P in 192..255 as bf16 pairs. P enters the product
// as hi + lo (hi = bf16(p), lo = bf16(p - hi)), so the weights keep about 16
// mantissa bits, as in the warp-level kernels: the high parts in columns
// 192..223, the low parts in 224..255. Q is a K-major 128-byte-swizzled
// [2 halves][128 rows][64 dims] tile in shared memory, loaded by two TMA
// boxes of 64 dims x group heads x tokens, whose rows land in r order.
//
// The grid is persistent: two CTAs per SM walk the items, largest first
// (later row tiles see more context), dealt out in snake order. Barrier phases
// count context steps across items, so one item's first loads and products
// overlap the previous item's last steps and output. Roles (192 threads):
// warps 0..3 own one query row per thread (tensor-memory lane = thread): they
// run the online softmax on S, write P, rescale O when the running max moves
// by more than 2^8, zero the V rows past the context of an item's last block
// (a zero weight times a stale V must stay zero), and write the output. Warp
// 4 loads each item's Q and stages K and V tiles of 64 positions (4 blocks,
// one 3-D TMA box of 16 rows x 64 dims per block and half) through 2-stage
// rings. Warp 5 allocates the tensor memory and one of its threads issues the
// products. Shared memory holds 96 KiB (Q and the rings), so two CTAs share an
// SM and one's softmax overlaps the other's products.
//
// Per step: as soon as the softmax has read S into registers the next S is
// issued (the next item's first S when this is an item's last step, once its
// Q has landed), so it runs during the exponentials; P.V runs once P is
// written, during the next step's softmax, which waits for it only before it
// touches O or overwrites P. An item's Q is reloaded once its predecessor's
// last S has completed, and its first P.V (which overwrites O) waits until the
// softmax has read the predecessor's O.
#include "tc.cuh"

namespace pa {

constexpr int kTcRows = 128;                  // query rows per tile (tensor-memory lanes)
constexpr int kTcTile = 64;                   // context positions per step
constexpr int kTcTileBlocks = kTcTile / kBlockSize;
constexpr int kTcStages = 2;
constexpr int kTcThreads = 192;               // 4 softmax warps, TMA warp, MMA warp
constexpr int kTcTileBytes = kTcTile * kHeadDim * 2;  // one K or V tile: [2 halves][64 positions][64 dims]
constexpr int kTcHalf = kTcTileBytes / 2;
constexpr uint32_t kTcCols = 256;             // tensor-memory columns per CTA
constexpr uint32_t kColO = 0, kColS = 128, kColP = 192;
constexpr float kRescaleLog2 = 8.f;           // O is rescaled once the max grows by more than this
constexpr int kTcCtasPerSm = 2;

constexpr int kTcQBytes = kTcRows * kHeadDim * 2;  // Q: [2 halves][128 rows][64 dims] bf16

struct TcSmem {
  static constexpr int k = 0;
  static constexpr int v = kTcStages * kTcTileBytes;
  static constexpr int q = 2 * kTcStages * kTcTileBytes;
  static constexpr int bars = q + kTcQBytes;
  // k_full[S], k_empty[S], v_full[S], v_empty[S], q_full, q_free, s_full, s_free, p_full, o_done, o_free, drain
  static constexpr int nbars = 4 * kTcStages + 8;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int total = abort_flag + 4;
  static constexpr int alloc = total + 1024;
};

// One work item: a row tile of (sequence b, KV head h).
struct TcItem {
  int b, h, q0, nq, L, row0, nrows, nblk, ntile, tail_valid;
};

// The item at position pos of the largest-first order: row tile descending,
// then KV head, then sequence. report: raise the length flags (one thread).
__device__ __forceinline__ TcItem tc_item(const AttnParams& p, int pos, int rpt, bool report) {
  TcItem it;
  const int per_x = p.kv_heads * p.batch;
  const int xi = pos / per_x, rem = pos - xi * per_x;
  const int x = p.row_groups - 1 - xi;
  it.h = rem % p.kv_heads;
  it.b = rem / p.kv_heads;
  const bool rep = report && x == 0 && it.h == 0;
  query_range(p, __ldg(p.query_start + it.b), __ldg(p.query_start + it.b + 1), rep, &it.q0, &it.nq);
  int L = __ldg(p.context_lens + it.b);
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  if (L < 0 || L > cap) {
    if (rep) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    L = L < 0 ? 0 : cap;
  }
  it.L = L;
  it.row0 = x * rpt;
  it.nrows = max(0, min(rpt, it.nq * p.group - it.row0));
  // Positions the tile's last row may see; every earlier row sees fewer.
  const int kv_end = it.nrows > 0 ? max(0, min(L, L - it.nq + (it.row0 + it.nrows - 1) / p.group + 1)) : 0;
  it.nblk = (kv_end + kBlockSize - 1) / kBlockSize;
  it.ntile = (it.nblk + kTcTileBlocks - 1) / kTcTileBlocks;
  it.tail_valid = kv_end - (it.nblk - 1) * kBlockSize;  // rows of the last block inside kv_end
  return it;
}

// Position of this CTA's k-th item: snake order over the grid, so that with
// items sorted largest first every CTA gets a similar total.
__device__ __forceinline__ int tc_item_pos(int k) {
  return k * int(gridDim.x) + ((k & 1) ? int(gridDim.x) - 1 - int(blockIdx.x) : int(blockIdx.x));
}

__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const __grid_constant__ CUtensorMap tmap_q, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t bk_full = base + TcSmem::bars;
  const uint32_t bk_empty = bk_full + 8 * kTcStages;
  const uint32_t bv_full = bk_empty + 8 * kTcStages;
  const uint32_t bv_empty = bv_full + 8 * kTcStages;
  const uint32_t b_qfull = bv_empty + 8 * kTcStages;
  const uint32_t b_qfree = b_qfull + 8;  // every S of the item has completed: Q may be reloaded
  const uint32_t b_sfull = b_qfree + 8;
  const uint32_t b_sfree = b_sfull + 8;  // the softmax has read S (S may be overwritten)
  const uint32_t b_pfull = b_sfree + 8;
  const uint32_t b_odone = b_pfull + 8;
  const uint32_t b_ofree = b_odone + 8;  // the softmax has read the item's O (O may be overwritten)
  const uint32_t b_drain = b_ofree + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + TcSmem::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + TcSmem::abort_flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rpt = p.rows_per_cta;  // rows of a tile: a multiple of the group, at most 128
  const int items = p.row_groups * p.kv_heads * p.batch;

  if (threadIdx.x >= rpt && threadIdx.x < kTcRows) {
    // A spare MMA row past the tile: Q stays zero so that its scores are finite.
    uint8_t* qs = sbase + TcSmem::q + threadIdx.x * 128;
#pragma unroll
    for (int c = 0; c < kHeadDim / 8; ++c)
      *reinterpret_cast<uint4*>(qs + (c >> 3) * (kTcQBytes / 2) + ((c & 7) << 4)) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(bk_full + 8 * s, 1);
      mbar_init(bk_empty + 8 * s, 1);
      mbar_init(bv_full + 8 * s, 1);
      mbar_init(bv_empty + 8 * s, 1);
    }
    mbar_init(b_qfull, 1);
    mbar_init(b_qfree, 1);
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, kTcRows);
    mbar_init(b_pfull, kTcRows);
    mbar_init(b_odone, 1);
    mbar_init(b_ofree, kTcRows);
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tc_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTcCols);
    tc_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&tmap_q);
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const uint64_t once = policy_evict_first();   // Q is read once
    const uint64_t policy = policy_evict_last();  // other row tiles re-read the same context
    bool failed = false;
    int g = 0, nitem = 0;  // context steps issued and items with steps so far
    int k_ahead = 0;       // lane 0: 1 while step g's K is issued but its V is not
    for (int k = 0; !failed; ++k) {
      const int pos = tc_item_pos(k);
      if (pos >= items) break;
      const TcItem w = tc_item(p, pos, rpt, false);
      if (w.ntile == 0) continue;
      if (lane == 0) {
        // Q of this item, once every S of the previous one has completed.
        if (*abort_flag || (nitem > 0 && !mbar_wait(b_qfree, (nitem - 1) & 1, p.wait_limit_ns))) {
          failed = true;
        } else {
          const int z = w.q0 + w.row0 / p.group;
          mbar_arrive_expect_tx(b_qfull, 2 * rpt * 128);
          tma_load_3d(base + TcSmem::q, &tmap_q, 0, w.h * p.group, z, b_qfull, once);
          tma_load_3d(base + TcSmem::q + kTcQBytes / 2, &tmap_q, 64, w.h * p.group, z, b_qfull, once);
        }
      }
      failed = __shfl_sync(0xffffffffu, failed, 0);
      if (failed) break;
      ++nitem;
      // Block ids come 32 at a time, one per lane; lane 0 issues the loads.
      const int32_t* table = p.block_tables + int64_t(w.b) * p.mbps;
      int chunk0 = 0;
      int ids = lane < w.nblk ? __ldg(table + lane) : -1;
      for (int j = 0; j < w.ntile && !failed; ++j) {
        if (j * kTcTileBlocks >= chunk0 + 32) {
          chunk0 += 32;
          ids = chunk0 + lane < w.nblk ? __ldg(table + chunk0 + lane) : -1;
        }
        int id[kTcTileBlocks];
#pragma unroll
        for (int i = 0; i < kTcTileBlocks; ++i) id[i] = __shfl_sync(0xffffffffu, ids, j * kTcTileBlocks - chunk0 + i);
        if (lane == 0) {
          const int s = g % kTcStages, ph = g / kTcStages;
          int y[kTcTileBlocks];
#pragma unroll
          for (int i = 0; i < kTcTileBlocks; ++i) {
            const bool real = j * kTcTileBlocks + i < w.nblk;
            if (real && (id[i] < 0 || id[i] >= p.num_blocks)) raise_flag(p.status, PA_FLAG_BAD_BLOCK);
            // Blocks past the context, and bad ids, read as zeros (out-of-range rows).
            y[i] = (real && id[i] >= 0 && id[i] < p.num_blocks) ? id[i] * kBlockSize : -kBlockSize;
          }
          // K once the stage's S has completed, V once its P.V has.
          if (*abort_flag || (ph > 0 && !mbar_wait(bk_empty + 8 * s, (ph - 1) & 1, p.wait_limit_ns))) {
            failed = true;
          } else {
            k_ahead = 1;  // this step's K is in flight until its V is issued too
            const uint32_t kd = base + TcSmem::k + s * kTcTileBytes, kb = bk_full + 8 * s;
            mbar_arrive_expect_tx(kb, kTcTileBytes);
#pragma unroll
            for (int i = 0; i < kTcTileBlocks; ++i) {
              tma_load_3d(kd + i * kBlockSize * 128, &tmap_k, 0, y[i], w.h, kb, policy);
              tma_load_3d(kd + kTcHalf + i * kBlockSize * 128, &tmap_k, 64, y[i], w.h, kb, policy);
            }
          }
          if (!failed && ph > 0 && !mbar_wait(bv_empty + 8 * s, (ph - 1) & 1, p.wait_limit_ns)) failed = true;
          if (!failed) {
            const uint32_t vd = base + TcSmem::v + s * kTcTileBytes, vb = bv_full + 8 * s;
            mbar_arrive_expect_tx(vb, kTcTileBytes);
#pragma unroll
            for (int i = 0; i < kTcTileBlocks; ++i) {
              tma_load_3d(vd + i * kBlockSize * 128, &tmap_v, 0, y[i], w.h, vb, policy);
              tma_load_3d(vd + kTcHalf + i * kBlockSize * 128, &tmap_v, 64, y[i], w.h, vb, policy);
            }
            k_ahead = 0;
          }
        }
        failed = __shfl_sync(0xffffffffu, failed, 0);
        if (!failed) ++g;
      }
    }
    if (failed && lane == 0) {
      raise_flag(p.status, PA_FLAG_TIMEOUT);
      *abort_flag = 1;
      // Let the loads already issued land (bounded) before the CTA can leave.
      for (int gg = max(0, g + k_ahead - kTcStages); gg < g + k_ahead; ++gg) {
        const int s = gg % kTcStages, par = (gg / kTcStages) & 1;
        (void)mbar_wait(bk_full + 8 * s, par);
        if (gg < g) (void)mbar_wait(bv_full + 8 * s, par);
      }
      if (nitem > 0) (void)mbar_wait(b_qfull, (nitem - 1) & 1);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      const uint32_t id_s = tc_idesc_bf16(kTcRows, kTcTile, false, false);
      const uint32_t id_o = tc_idesc_bf16(kTcRows, kHeadDim, false, true);
      // Descriptors are built once; a byte offset d within an operand adds
      // d >> 4 to the descriptor's start-address field.
      const uint64_t q_desc = tc_smem_desc(base + TcSmem::q, 16, 1024);
      const uint64_t k_desc = tc_smem_desc(base + TcSmem::k, 16, 1024);
      const uint64_t v_desc = tc_smem_desc(base + TcSmem::v, kTcHalf, 1024);
      // S = Q . K^T for context step gg: 8 steps of 16 dims; Q and K are
      // K-major (rows x dims).
      auto issue_s = [&](int gg) {
        const int s = gg % kTcStages;
        const uint64_t kd = k_desc + uint64_t((s * kTcTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTcHalf + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (kTcQBytes / 2) + (kk & 3) * 32;
          tc_mma(tmem + kColS, q_desc + (qoff >> 4), kd + (off >> 4), id_s, kk > 0);
        }
        tc_commit(b_sfull);
        tc_commit(bk_empty + 8 * s);
      };
      // The next item with context steps at item index k or later.
      auto next_item = [&](int& k, TcItem& w) {
        for (;; ++k) {
          const int pos = tc_item_pos(k);
          if (pos >= items) return false;
          w = tc_item(p, pos, rpt, false);
          if (w.ntile > 0) return true;
        }
      };
      bool ok = true;
      int k = 0;
      TcItem cur, nxt;
      bool have = next_item(k, cur);
      ++k;
      bool have_nxt = have && next_item(k, nxt);
      ++k;
      int g = 0, nitem = 0;
      if (have) {
        ok = mbar_wait(b_qfull, 0, p.wait_limit_ns) && mbar_wait(bk_full, 0, p.wait_limit_ns);
        if (ok) {
          tc_fence_after_sync();
          issue_s(0);
          if (cur.ntile == 1) tc_commit(b_qfree);
        }
      }
      while (have && ok) {
        for (int j = 0; j < cur.ntile && ok; ++j) {
          const int gg = g + j, s = gg % kTcStages, par = (gg / kTcStages) & 1;
          // The next step's S: this item's, or the next item's first (once its Q has landed).
          const bool more = j + 1 < cur.ntile;
          if (more || have_nxt) {
            const int g1 = gg + 1, s1 = g1 % kTcStages, par1 = (g1 / kTcStages) & 1;
            if (*abort_flag || !mbar_wait(b_sfree, gg & 1, p.wait_limit_ns) || !mbar_wait(bk_full + 8 * s1, par1, p.wait_limit_ns) ||
                (!more && !mbar_wait(b_qfull, (nitem + 1) & 1, p.wait_limit_ns))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_s(g1);
            // Q may be reloaded once its item's last S has completed.
            if ((more && j + 2 == cur.ntile) || (!more && nxt.ntile == 1)) tc_commit(b_qfree);
          }
          // P.V of this step; an item's first P.V overwrites O, once the
          // softmax has read the previous item's.
          if (!mbar_wait(b_pfull, gg & 1, p.wait_limit_ns) || !mbar_wait(bv_full + 8 * s, par, p.wait_limit_ns) ||
              (j == 0 && nitem > 0 && !mbar_wait(b_ofree, (nitem - 1) & 1, p.wait_limit_ns))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // O += P_hi . V + P_lo . V: 4 steps of 16 positions. P (rows x
          // positions) is in tensor memory; V is MN-major (positions x dims,
          // dims contiguous): 64-dim halves kTcHalf apart, 8-position groups
          // 1024 bytes apart.
          const uint64_t vd = v_desc + uint64_t((s * kTcTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTcTile / 16; ++kk) {
            tc_mma_ts(tmem + kColO, tmem + kColP + kk * 8, vd + uint64_t((kk * 2048) >> 4), id_o, j > 0 || kk > 0);
            tc_mma_ts(tmem + kColO, tmem + kColP + 32 + kk * 8, vd + uint64_t((kk * 2048) >> 4), id_o, true);
          }
          tc_commit(b_odone);
          tc_commit(bv_empty + 8 * s);
        }
        g += cur.ntile;
        ++nitem;
        cur = nxt;
        have = have_nxt;
        if (have) {
          have_nxt = next_item(k, nxt);
          ++k;
        }
      }
      if (!ok) {
        raise_flag(p.status, PA_FLAG_TIMEOUT);
        *abort_flag = 1;
      }
      // Every MMA issued above has finished before the tensor memory is freed.
      tc_commit(b_drain);
      (void)mbar_wait(b_drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------- softmax: thread r owns row r of each item's tile ----------------
    const int r = threadIdx.x;
    const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int pos = tc_item_pos(k);
      if (pos >= items) break;
      const TcItem w = tc_item(p, pos, rpt, r == 0);
      const bool live = r < w.nrows;
      if (w.ntile == 0) {
        // No rows, or every row sits at a negative position: zeros.
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row_offset(p, w.q0, w.h, w.row0 + r));
#pragma unroll
          for (int c = 0; c < kHeadDim / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int lim = live ? row_limit(p, w.L, w.nq, w.row0 + r) : -1;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < w.ntile; ++j) {
        const int gg = g + j;
        if (__any_sync(0xffffffffu, *abort_flag != 0) || !__all_sync(0xffffffffu, mbar_wait(b_sfull, gg & 1, p.wait_limit_ns))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t sr[kTcTile / 2], sr2[kTcTile / 2];
        tc_ld32_issue(trow + kColS, sr);
        tc_ld32_issue(trow + kColS + 32, sr2);
        tc_wait_ld(sr);
        tc_wait_ld(sr2);
        tc_fence_before_sync();
        mbar_arrive(b_sfree);
        float s[kTcTile];
#pragma unroll
        for (int i = 0; i < kTcTile / 2; ++i) {
          s[i] = __uint_as_float(sr[i]);
          s[kTcTile / 2 + i] = __uint_as_float(sr2[i]);
        }
        // Tile max in base-2 units. A tile wholly inside the row's limit takes
        // the max of the raw scores (scale >= 0) and folds the scale into the
        // exponent's FMA; otherwise the scores are scaled and masked here.
        const int t0 = j * kTcTile;
        const bool whole = t0 + kTcTile - 1 <= lim && p.scale_log2 >= 0.f;
        float mk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mk[q] = -INFINITY;
        if (whole) {
#pragma unroll
          for (int i = 0; i < kTcTile; ++i) mk[i & 7] = fmaxf(mk[i & 7], s[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kTcTile; ++i) {
            s[i] = t0 + i <= lim ? s[i] * p.scale_log2 : -INFINITY;
            mk[i & 7] = fmaxf(mk[i & 7], s[i]);
          }
        }
        float mx = fmaxf(fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])), fmaxf(fmaxf(mk[4], mk[5]), fmaxf(mk[6], mk[7])));
        const float mul = whole ? p.scale_log2 : 1.f;
        if (whole) mx *= mul;
        // Online softmax with a lazy reference max: m moves (and O, l are
        // rescaled) only when the tile max exceeds it by more than 2^8, so
        // weights stay <= 256.
        const float m_new = fmaxf(m, mx);
        const bool move = m_new > m + kRescaleLog2;
        // The previous step's P.V must be done before O is touched or P
        // rewritten: waited for here only when O needs rescaling, else after
        // the exponentials. An item's first step has no O to rescale (its
        // first P.V overwrites O).
        bool pv_done = gg == 0;
        if (__any_sync(0xffffffffu, move)) {
          const float alpha = move ? fast_exp2(m - m_new) : 1.f;
          if (move) {
            l *= alpha;
            m = m_new;
          }
          if (j > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(b_odone, (gg - 1) & 1, p.wait_limit_ns))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            pv_done = true;
#pragma unroll 1
            for (int c = 0; c < kHeadDim / 32; ++c) {
              float o[32];
              tc_ld32(trow + kColO + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tc_st32(trow + kColO + c * 32, o);
            }
          }
        }
        // p = 2^(s * mul - m), summed in 8 partial sums; P = hi + lo as bf16 pairs.
        const float m_use = m == -INFINITY ? 0.f : m;
        const uint64_t mul2 = f2_pack(mul, mul), neg2 = f2_pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), mul2, neg2), a0, a1);
          const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
          const uint64_t pp = f2_pack(p0, p1);
          acc[c & 3] = f2_add(acc[c & 3], pp);
          const uint32_t x = pack_bf16x2(p0, p1);
          hi[c] = x;
          float r0, r1;
          f2_unpack(f2_sub(pp, f2_pack(bf16_lo(x), bf16_hi(x))), r0, r1);
          lo[c] = pack_bf16x2(r0, r1);
        }
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a0, a1;
          f2_unpack(acc[q], a0, a1);
          sum += a0 + a1;
        }
        l += sum;
        if (!pv_done) {
          if (!__all_sync(0xffffffffu, mbar_wait(b_odone, (gg - 1) & 1, p.wait_limit_ns))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        if (j == w.ntile - 1 && w.tail_valid < kBlockSize) {
          // The item's last block: zero its V rows past the context once they
          // have landed, before P hands the stage to the product.
          const int s = gg % kTcStages;
          if (!__all_sync(0xffffffffu, mbar_wait(bv_full + 8 * s, (gg / kTcStages) & 1, p.wait_limit_ns))) {
            ok = false;
            break;
          }
          uint8_t* vt = sbase + TcSmem::v + s * kTcTileBytes;
          const int n0 = (w.nblk - 1 - j * kTcTileBlocks) * kBlockSize;  // the block's first row in the tile
          for (int e = r; e < (kBlockSize - w.tail_valid) * 16; e += kTcRows) {
            const int n = n0 + w.tail_valid + (e >> 4), c = e & 15;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kTcHalf + n * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_st32_issue(trow + kColP, hi);
        tc_st32_issue(trow + kColP + 32, lo);
        tc_wait_st();
        tc_fence_before_sync();
        mbar_arrive(b_pfull);
      }
      if (!ok) break;
      g += w.ntile;
      // The item's output: O after its last P.V, read out, handed back, then stored.
      if (!__all_sync(0xffffffffu, mbar_wait(b_odone, (g - 1) & 1, p.wait_limit_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t o0[32], o1[32], o2[32], o3[32];
      tc_ld32_issue(trow + kColO, o0);
      tc_ld32_issue(trow + kColO + 32, o1);
      tc_ld32_issue(trow + kColO + 64, o2);
      tc_ld32_issue(trow + kColO + 96, o3);
      tc_wait_ld(o0);
      tc_wait_ld(o1);
      tc_wait_ld(o2);
      tc_wait_ld(o3);
      tc_fence_before_sync();
      mbar_arrive(b_ofree);
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row_offset(p, w.q0, w.h, w.row0 + r));
        auto put = [&](const uint32_t (&o)[32], int c0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c0 + c] = make_uint4(
                pack_bf16x2(__uint_as_float(o[8 * c]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
        };
        put(o0, 0);
        put(o1, 4);
        put(o2, 8);
        put(o3, 12);
      }
    }
    if (!ok) {
      if (lane == 0) raise_flag(p.status, PA_FLAG_TIMEOUT);
      *abort_flag = 1;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tc_dealloc(tmem, kTcCols);
  }
}

cudaError_t launch_attn_prefill_tc(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                                   const AttnParams& p, cudaStream_t stream) {
  static PerDeviceOnce once;
  static int sms[kMaxDevices] = {0};
  const cudaError_t e = once.run([](int dev) {
    cudaError_t r = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcSmem::alloc);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return r;
  });
  if (e != cudaSuccess) return e;
  int dev = 0;
  cudaGetDevice(&dev);  // in range: run() checked it
  const int64_t items = int64_t(p.row_groups) * p.kv_heads * p.batch;
  const int64_t slots = int64_t(kTcCtasPerSm) * sms[dev];
  const unsigned grid = unsigned(items < slots ? items : slots);
  attn_prefill_tc_kernel<<<grid, kTcThreads, TcSmem::alloc, stream>>>(tk, tv, tq, p);
  return cudaGetLastError();
}

}  // namespace pa
