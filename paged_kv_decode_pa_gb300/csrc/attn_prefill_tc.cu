// Paged prefill attention on the fifth-generation tensor cores (tcgen05), bf16.
//
// Same operation as attn_prefill.cu (causal attention of a prompt chunk over
// the sequence's paged cache: "From 183 ms to 19 ms per decode step", section
// "What's next"; the masked softmax of "Anatomy of a Decode-Step Stall",
// Model._layer), for the rows r = i * group + g of floor(128 / group) query
// tokens of one (sequence, KV head) per CTA (rows_per_cta <= 128; the MMA's
// spare rows are zero). Here the products run as single-thread-issued
// tcgen05.mma with the accumulators in tensor memory:
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
// Roles (192 threads): warps 0..3 own one query row per thread (tensor-memory
// lane = thread): they run the online softmax on S, write P, rescale O when
// the running max moves by more than 2^8, and write the output. Warp 4 loads
// Q and stages K and V tiles of 64 positions (4 blocks, one 3-D TMA box of 16
// rows x 64 dims per block and half) through 2-stage rings. Warp 5 allocates the
// tensor memory and one of its threads issues the MMAs. Shared memory holds
// 96 KiB (Q and the rings), so two CTAs share an SM and one's softmax overlaps the other's
// products.
//
// Per 64-position step j: as soon as the softmax has read S_j into registers
// the next S_{j+1} is issued, so it runs during step j's exponentials; P.V_j
// runs once P_j is written, during step j + 1's softmax, which waits for it
// only before it touches O or overwrites P. Context rows past the end of the
// last block read as zero weights; their V rows are zeroed in shared memory
// before the product (a zero weight times a stale V must stay zero).
#include "tc.cuh"

namespace pa {

constexpr int kTcRows = 128;                  // query rows per CTA (tensor-memory lanes)
constexpr int kTcTile = 64;                   // context positions per step
constexpr int kTcTileBlocks = kTcTile / kBlockSize;
constexpr int kTcStages = 2;
constexpr int kTcThreads = 192;               // 4 softmax warps, TMA warp, MMA warp
constexpr int kTcTileBytes = kTcTile * kHeadDim * 2;  // one K or V tile: [2 halves][64 positions][64 dims]
constexpr int kTcHalf = kTcTileBytes / 2;
constexpr uint32_t kTcCols = 256;             // tensor-memory columns per CTA
constexpr uint32_t kColO = 0, kColS = 128, kColP = 192;
constexpr float kRescaleLog2 = 8.f;           // O is rescaled once the max grows by more than this

constexpr int kTcQBytes = kTcRows * kHeadDim * 2;  // Q: [2 halves][128 rows][64 dims] bf16

struct TcSmem {
  static constexpr int k = 0;
  static constexpr int v = kTcStages * kTcTileBytes;
  static constexpr int q = 2 * kTcStages * kTcTileBytes;
  static constexpr int bars = q + kTcQBytes;
  // k_full[S], k_empty[S], v_full[S], v_empty[S], v_land, q_full, s_full, s_free, p_full, o_done, drain
  static constexpr int nbars = 4 * kTcStages + 7;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int total = abort_flag + 4;
  static constexpr int alloc = total + 1024;
};

__global__ void __launch_bounds__(kTcThreads, 2)
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
  const uint32_t b_vland = bv_empty + 8 * kTcStages;  // last V tile, before its stale rows are zeroed
  const uint32_t b_qfull = b_vland + 8;
  const uint32_t b_sfull = b_qfull + 8;
  const uint32_t b_sfree = b_sfull + 8;  // the softmax has read S (S may be overwritten)
  const uint32_t b_pfull = b_sfree + 8;
  const uint32_t b_odone = b_pfull + 8;
  const uint32_t b_drain = b_odone + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + TcSmem::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + TcSmem::abort_flag);

  const int b = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rpt = p.rows_per_cta;  // rows of this tile: a multiple of the group, at most 128
  // The sequence's query range and length are loaded first; the barrier
  // setup and the tensor-memory allocation below overlap their latency.
  const int qs_a = __ldg(p.query_start + b), qs_e = __ldg(p.query_start + b + 1);
  const int L_raw = __ldg(p.context_lens + b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(bk_full + 8 * s, 1);
      mbar_init(bk_empty + 8 * s, 1);
      mbar_init(bv_full + 8 * s, 1);
      mbar_init(bv_empty + 8 * s, 1);
    }
    mbar_init(b_vland, 1);
    mbar_init(b_qfull, 1 + (kTcRows - rpt));  // the Q loads, and the threads that zero the spare rows
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, kTcRows);
    mbar_init(b_pfull, kTcRows);
    mbar_init(b_odone, 1);
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

  int q0, nq;
  query_range(p, qs_a, qs_e, blockIdx.x == 0 && h == 0, &q0, &nq);
  int L = L_raw;
  const int cap = min(p.max_context_len, p.mbps * kBlockSize);
  if (L < 0 || L > cap) {
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) raise_flag(p.status, PA_FLAG_BAD_LENGTH);
    L = L < 0 ? 0 : cap;
  }
  const int rows_b = nq * p.group;
  const int row0 = blockIdx.x * rpt;
  const int nrows = max(0, min(rpt, rows_b - row0));
  // Positions the CTA's last row may see; every earlier row sees fewer.
  const int kv_end = nrows > 0 ? max(0, min(L, L - nq + (row0 + nrows - 1) / p.group + 1)) : 0;
  const int nblk = (kv_end + kBlockSize - 1) / kBlockSize;
  const int ntile = (nblk + kTcTileBlocks - 1) / kTcTileBlocks;
  const int tail_valid = kv_end - (nblk - 1) * kBlockSize;  // rows of the last block inside kv_end

  if (ntile == 0) {
    // No rows here, or every row sits at a negative position (zeros).
    if (threadIdx.x < nrows) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row_offset(p, q0, h, row0 + threadIdx.x));
#pragma unroll
      for (int c = 0; c < kHeadDim / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    }
  } else if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // Q rows row0 .. row0 + rpt - 1: tokens q0 + row0 / group onwards, the
      // group's heads, one box per 64-dim half.
      const uint64_t once = policy_evict_first();
      const int tq = rpt / p.group;
      mbar_arrive_expect_tx(b_qfull, 2 * rpt * 128);
      tma_load_3d(base + TcSmem::q, &tmap_q, 0, h * p.group, q0 + blockIdx.x * tq, b_qfull, once);
      tma_load_3d(base + TcSmem::q + kTcQBytes / 2, &tmap_q, 64, h * p.group, q0 + blockIdx.x * tq, b_qfull, once);
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const uint64_t policy = policy_evict_last();  // sibling row tiles re-read the same context
    const int32_t* table = p.block_tables + int64_t(b) * p.mbps;
    int chunk0 = 0;
    int ids = lane < nblk ? __ldg(table + lane) : -1;
    bool failed = false;
    int issued = 0;
    for (int j = 0; j < ntile && !failed; ++j) {
      if (j * kTcTileBlocks >= chunk0 + 32) {
        chunk0 += 32;
        ids = chunk0 + lane < nblk ? __ldg(table + chunk0 + lane) : -1;
      }
      int id[kTcTileBlocks];
#pragma unroll
      for (int i = 0; i < kTcTileBlocks; ++i) id[i] = __shfl_sync(0xffffffffu, ids, j * kTcTileBlocks - chunk0 + i);
      if (lane == 0) {
        const int s = j % kTcStages, ph = j / kTcStages;
        int y[kTcTileBlocks];
#pragma unroll
        for (int i = 0; i < kTcTileBlocks; ++i) {
          const bool real = j * kTcTileBlocks + i < nblk;
          if (real && (id[i] < 0 || id[i] >= p.num_blocks)) raise_flag(p.status, PA_FLAG_BAD_BLOCK);
          // Blocks past the context, and bad ids, read as zeros (out-of-range rows).
          y[i] = (real && id[i] >= 0 && id[i] < p.num_blocks) ? id[i] * kBlockSize : -kBlockSize;
        }
        if (*abort_flag || (ph > 0 && !mbar_wait(bk_empty + 8 * s, (ph - 1) & 1))) {
          failed = true;
        } else {
          const uint32_t dst = base + TcSmem::k + s * kTcTileBytes, fb = bk_full + 8 * s;
          mbar_arrive_expect_tx(fb, kTcTileBytes);
#pragma unroll
          for (int i = 0; i < kTcTileBlocks; ++i) {
            tma_load_3d(dst + i * kBlockSize * 128, &tmap_k, 0, y[i], h, fb, policy);
            tma_load_3d(dst + kTcHalf + i * kBlockSize * 128, &tmap_k, 64, y[i], h, fb, policy);
          }
        }
        if (!failed && ph > 0 && !mbar_wait(bv_empty + 8 * s, (ph - 1) & 1)) failed = true;
        if (!failed) {
          const bool zero_tail = j == ntile - 1 && tail_valid < kBlockSize;
          const uint32_t dst = base + TcSmem::v + s * kTcTileBytes;
          const uint32_t fb = zero_tail ? b_vland : bv_full + 8 * s;
          mbar_arrive_expect_tx(fb, kTcTileBytes);
#pragma unroll
          for (int i = 0; i < kTcTileBlocks; ++i) {
            tma_load_3d(dst + i * kBlockSize * 128, &tmap_v, 0, y[i], h, fb, policy);
            tma_load_3d(dst + kTcHalf + i * kBlockSize * 128, &tmap_v, 64, y[i], h, fb, policy);
          }
          issued = j + 1;
        }
      }
      failed = __shfl_sync(0xffffffffu, failed, 0);
    }
    // Zero the last block's V rows past kv_end once the tile has landed.
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (!failed && tail_valid < kBlockSize) {
      const int j = ntile - 1, s = j % kTcStages;
      if (__all_sync(0xffffffffu, mbar_wait(b_vland, 0))) {
        uint8_t* vt = sbase + TcSmem::v + s * kTcTileBytes;
        const int n0 = (nblk - 1 - j * kTcTileBlocks) * kBlockSize;  // the block's first row in the tile
        for (int e = lane; e < (kBlockSize - tail_valid) * 16; e += 32) {
          const int n = n0 + tail_valid + (e >> 4), c = e & 15;
          *reinterpret_cast<uint4*>(vt + (c >> 3) * kTcHalf + n * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bv_full + 8 * s);
      } else {
        failed = true;
      }
    }
    if (failed && lane == 0) {
      raise_flag(p.status, PA_FLAG_TIMEOUT);
      *abort_flag = 1;
      // Let the loads already issued land (bounded) before the CTA can leave.
      for (int j = max(0, issued - kTcStages); j < issued; ++j) {
        const int s = j % kTcStages, par = (j / kTcStages) & 1;
        (void)mbar_wait(bk_full + 8 * s, par);
        if (j == ntile - 1 && tail_valid < kBlockSize)
          (void)mbar_wait(b_vland, 0);
        else
          (void)mbar_wait(bv_full + 8 * s, par);
      }
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
      // S = Q . K^T: 8 steps of 16 dims; Q and K are K-major (rows x dims).
      auto issue_s = [&](int j) {
        const int s = j % kTcStages;
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
      bool ok = mbar_wait(b_qfull, 0) && mbar_wait(bk_full, 0);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0);
      }
      for (int j = 0; j < ntile && ok; ++j) {
        const int s = j % kTcStages, par = (j / kTcStages) & 1;
        if (j + 1 < ntile) {
          const int s1 = (j + 1) % kTcStages, par1 = ((j + 1) / kTcStages) & 1;
          if (*abort_flag || !mbar_wait(b_sfree, j & 1) || !mbar_wait(bk_full + 8 * s1, par1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(j + 1);
        }
        if (!mbar_wait(b_pfull, j & 1) || !mbar_wait(bv_full + 8 * s, par)) {
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
    // ---------------- softmax: thread r owns query row row0 + r ----------------
    const int r = threadIdx.x;
    const bool live = r < nrows;
    const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
    if (r >= rpt) {
      // A spare MMA row past the tile: zero Q so that its scores are finite.
      uint8_t* qs = sbase + TcSmem::q + r * 128;
#pragma unroll
      for (int c = 0; c < kHeadDim / 8; ++c)
        *reinterpret_cast<uint4*>(qs + (c >> 3) * (kTcQBytes / 2) + ((c & 7) << 4)) = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      mbar_arrive(b_qfull);
    }
    const int lim = live ? row_limit(p, L, nq, row0 + r) : -1;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0) || !__all_sync(0xffffffffu, mbar_wait(b_sfull, j & 1))) {
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
      for (int k = 0; k < 8; ++k) mk[k] = -INFINITY;
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
      // P.V of the previous step must be done before O is touched or P
      // rewritten: waited for here only when O needs rescaling, else after
      // the exponentials.
      bool pv_done = j == 0;
      if (__any_sync(0xffffffffu, move)) {
        if (!pv_done) {
          if (!__all_sync(0xffffffffu, mbar_wait(b_odone, (j - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          pv_done = true;
        }
        const float alpha = move ? fast_exp2(m - m_new) : 1.f;
        if (move) {
          l *= alpha;
          m = m_new;
        }
        if (j > 0) {
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
      for (int k = 0; k < 4; ++k) {
        float a0, a1;
        f2_unpack(acc[k], a0, a1);
        sum += a0 + a1;
      }
      l += sum;
      if (!pv_done) {
        if (!__all_sync(0xffffffffu, mbar_wait(b_odone, (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      tc_st32_issue(trow + kColP, hi);
      tc_st32_issue(trow + kColP + 32, lo);
      tc_wait_st();
      tc_fence_before_sync();
      mbar_arrive(b_pfull);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b_odone, (ntile - 1) & 1));
    if (!ok) {
      if (lane == 0) raise_flag(p.status, PA_FLAG_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row_offset(p, q0, h, row0 + (live ? r : 0)));
#pragma unroll 1
      for (int c = 0; c < kHeadDim / 32; ++c) {
        float o[32];
        tc_ld32(trow + kColO + c * 32, o);
        if (live) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[c * 4 + k] = make_uint4(pack_bf16x2(o[8 * k] * inv, o[8 * k + 1] * inv),
                                        pack_bf16x2(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                        pack_bf16x2(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                        pack_bf16x2(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
        }
      }
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
                                   const AttnParams& p, dim3 grid, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcSmem::alloc);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  attn_prefill_tc_kernel<<<grid, kTcThreads, TcSmem::alloc, stream>>>(tk, tv, tq, p);
  return cudaGetLastError();
}

}  // namespace pa
