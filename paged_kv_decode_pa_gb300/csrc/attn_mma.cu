// Paged decode / verify attention, bf16, tensor-core products (sm_103a).
//
// One CTA per (context split, KV head, sequence x row group), holding every
// query row of the group that reads this KV head: the query-head group for
// decode, (k+1) x group rows for verify ("From 183 ms to 19 ms per decode
// step", sections "1. Grouped attention", "3. A Triton paged-decode kernel",
// "Then speculative decoding got slower"). The split is a fixed number of
// tokens, so a sequence's result depends on its own length only.
//
// Warp roles (3 warps):
//   warp 2      producer: one lane walks the split's block-table entries and
//               issues TMA tensor loads of each 16-token block, one box for
//               K and one for V, into a ring of shared-memory stages
//               (128-byte swizzle, so ldmatrix reads are bank-conflict free). Each block is a contiguous
//               16 x 128 tile of the head-major cache ("2. Head-major KV
//               cache"): no gather, no padded copy.
//   warps 0..1  consumers: block j goes to warp j % 2. Per block, a warp
//               computes S^T = K Q^T (16 tokens x up to 16 rows) with
//               m16n8k16 bf16 MMAs, masks, runs the fp32 online softmax
//               (running max and sum, rescaled per block: "3. A Triton
//               paged-decode kernel"), turns P^T into the B operand in
//               registers (movmatrix; P split into two bf16 parts), and
//               accumulates O^T += V^T P^T.
// Then the two warps' states are combined and the split epilogue writes the
// output, or a partial plus the log-sum-exp that the last split merges.
//
// Masking: a position beyond the sequence (or beyond a verify row's causal
// limit) gets score -inf, and the V rows of a partial last block are zeroed in
// shared memory before use, since stale rows may hold anything ("A Rust
// inference server for Qwen2 on Apple Silicon", Day 3 "Known gaps": a zero key
// is not neutral; 0 x NaN is NaN).
//
// Fused verify: the CTA whose split holds a new token's position writes that
// token's K/V row to the cache (row group 0 only) and patches the row into its
// shared-memory tile from the inputs, so no CTA depends on another's write.
// The producer warp does the patching: a block holding new tokens lands on a
// barrier of its own, the producer patches the stage and then completes the
// stage's full barrier, so the consumers carry no code for it. A new token
// whose slot is not the table slot of its position (a negative slot is not
// written) keeps the pool's row, as a separate append followed by attention
// would see it.
#include "mma_tile.cuh"

namespace pa {

// CTA shape, chosen by measurement on GB300 (c2..c5 workloads): two consumer
// warps and a six-block ring per CTA, four CTAs per SM (three with 16 query
// rows). The same 24 blocks in flight per SM as three CTAs of four warps with
// eight stages, but more CTAs, and so more TMA issuers and a finer grid, per SM.
constexpr int kMmaConsumers = 2;
constexpr int kStages = 6;                 // shared-memory ring depth (blocks in flight per CTA)
constexpr int kStageBytes = kBlockBytes;   // one K+V block: one TMA box per tile (16 rows x 2 halves x 64 dims)
constexpr int kMmaThreads = (kMmaConsumers + 1) * 32;

struct MmaSmem {
  // Offsets from the 1024-byte aligned base.
  static constexpr int stages = 0;
  static constexpr int bars = kStages * kStageBytes;            // full, empty, landed [kStages] each
  static constexpr int ids = bars + 3 * kStages * 8;            // block ids of the split
  static constexpr int ml = ids + (kMaxSplitTokens / kBlockSize) * 4;  // m, l per warp and row
  static constexpr int flag = ml + 2 * kMmaConsumers * kRowSlots * 4;
  static constexpr int total = flag + 16;
  static constexpr int alloc = total + 1024;  // slack for aligning the base
};
static_assert(kMmaConsumers * kRowSlots * kCombineStride * 4 <= kStages * kStageBytes,
              "cross-warp buffer must fit in the stage ring");
// Every phase of a stage's full barrier must be awaited by the same consumer
// warp (block j uses stage j % kStages and warp j % kMmaConsumers). Otherwise
// a fast warp could wait for phase k of a stage whose phase k-1 (another
// warp's block) has not completed yet, and the parity test would pass early.
static_assert(kStages % kMmaConsumers == 0, "stages must be a multiple of the consumer warps");

template <int NT>
__global__ void __launch_bounds__(kMmaThreads, NT == 1 ? 4 : 3)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  int32_t* s_ids = reinterpret_cast<int32_t*>(sbase + MmaSmem::ids);
  float* s_m = reinterpret_cast<float*>(sbase + MmaSmem::ml);
  float* s_l = s_m + kMmaConsumers * kRowSlots;
  int* s_flag = reinterpret_cast<int*>(sbase + MmaSmem::flag);
  const uint32_t bar_full = base + MmaSmem::bars;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_land = bar_empty + kStages * 8;  // blocks holding new tokens land here

  // The descriptor fetch overlaps the loads below instead of delaying the
  // first TMA issue.
  if (threadIdx.x == kMmaConsumers * 32) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // The sequence's length and the split's block-table entries are loaded
  // together: with the base split size the entries do not depend on the
  // length, so the two memory latencies overlap instead of adding up.
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_land + 8 * s, 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Consumer state lives at function scope so that it survives until the
  // combine below (the producer warp carries an unused copy).
  RowState<NT> st;
  st.reset();
  const Lanes ln(lane);
  const int g = ln.g, c = ln.c;

  if (warp == kMmaConsumers) {
    // ---------------- producer ----------------
    // Blocks from jf on hold new tokens: they land on bar_land, and the whole
    // warp's patch_next() turns them into ordinary stages.
    const int new0 = w.L - w.nq;
    const int jf = (p.fused_write && w.t1 > new0) ? max(0, new0 - w.t0) / kBlockSize : nblk;
    if (jf < nblk) {
      // This split holds the new tokens: bring their K/V rows (two 128-byte
      // lines each) and their slots into L2 now, so that the patch does not
      // wait on memory once per row.
      for (int e = lane; e < w.nq * 4; e += 32) {
        const int i = e >> 2, half = e & 1;
        const void* base_new = (e & 2) ? p.v_new : p.k_new;
        prefetch_l2(static_cast<const uint16_t*>(base_new) +
                    (int64_t(w.q0 + i) * p.kv_heads + w.h) * kHeadDim + half * 64);
      }
      if (lane == 0) prefetch_l2(p.slot_mapping + w.q0);
    }
    int patched = jf;  // next block holding new tokens to patch
    // Patch block `patched` once it has landed: the new tokens' rows whose
    // slot is the table slot of their position come from the inputs; row
    // group 0 writes every in-pool slot to the cache; V rows past the
    // context are zeroed. Then the stage's full barrier completes.
    auto patch_next = [&]() -> bool {
      const int k = patched, s = k % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_land + 8 * s, ((k - jf) / kStages) & 1, p.wait_limit_ns))) return false;
      uint8_t* kt_ptr = sbase + MmaSmem::stages + s * kStageBytes;
      uint8_t* vt_ptr = kt_ptr + kTileBytes;
      const int tok0 = w.t0 + k * kBlockSize;
      const int pos_lo = max(tok0, new0), pos_hi = min(tok0 + kBlockSize, w.L);
      const int id = s_ids[k];
      const bool id_ok = id >= 0 && id < p.num_blocks;
      const int ch = lane & 15;  // lanes 0..15 move K chunks, lanes 16..31 V chunks
      const bool is_v = lane >= 16;
      for (int pos = pos_lo; pos < pos_hi; ++pos) {
        const int i = pos - new0, t = pos - tok0;
        const int slot = __ldg(p.slot_mapping + w.q0 + i);
        const int64_t src = (int64_t(w.q0 + i) * p.kv_heads + w.h) * kHeadDim + ch * 8;
        const uint4 val =
            __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(is_v ? p.v_new : p.k_new) + src));
        if (id_ok && slot == id * kBlockSize + t)
          *reinterpret_cast<uint4*>((is_v ? vt_ptr : kt_ptr) + tile_off(t, ch)) = val;
        if (w.rg == 0) {
          if (slot >= 0 && slot < p.num_blocks * kBlockSize) {
            const int64_t dst =
                ((int64_t(w.h) * p.num_blocks + slot / kBlockSize) * kBlockSize + slot % kBlockSize) * kHeadDim +
                ch * 8;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(is_v ? p.v_cache_w : p.k_cache_w) + dst) = val;
          } else if (slot >= 0 && lane == 0) {
            raise_flag(p.status, PA_FLAG_BAD_SLOT);
          }
        }
      }
      const int valid = min(kBlockSize, w.L - tok0);
      for (int e = lane; e < (kBlockSize - valid) * 16; e += 32) {
        const int t = valid + (e >> 4), c16 = e & 15;
        *reinterpret_cast<uint4*>(vt_ptr + tile_off(t, c16)) = make_uint4(0, 0, 0, 0);
      }
      // These generic writes come before the next tensor load into the stage.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_full + 8 * s);
      ++patched;
      return true;
    };
    // Lane 0 issues the loads. A block that holds new tokens lands on
    // bar_land; its stage can be reused only once it is patched, so lane 0
    // runs ahead to kStages blocks past the first of them, and the whole warp
    // then patches them in order, issuing one more block after each patch
    // when there are more (over 80 new tokens in the split).
    const uint64_t policy = policy_evict_first();
    auto issue = [&](int j) -> bool {  // lane 0
      const int s = j % kStages, n = j / kStages;
      if (n > 0 && !mbar_wait(bar_empty + 8 * s, (n - 1) & 1, p.wait_limit_ns)) return false;
      const uint32_t st = base + MmaSmem::stages + s * kStageBytes;
      const uint32_t fb = (j >= jf ? bar_land : bar_full) + 8 * s;
      int id = s_ids[j];
      if (id < 0 || id >= p.num_blocks) {  // outside the pool: TMA reads zeros instead
        raise_flag(p.status, PA_FLAG_BAD_BLOCK);
        id = -1;
      }
      const int y = id >= 0 ? id * kBlockSize : -kBlockSize;
      mbar_arrive_expect_tx(fb, kStageBytes);
      tma_load_4d(st, &tmap_k, 0, y, 0, w.h, fb, policy);
      tma_load_4d(st + kTileBytes, &tmap_v, 0, y, 0, w.h, fb, policy);
      return true;
    };
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      const int ahead = min(nblk, jf + kStages);
      while (issued < ahead && (ok = issue(issued))) ++issued;
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    while (ok && patched < issued) {
      ok = patch_next();
      if (ok && issued < nblk) {
        if (lane == 0 && (ok = issue(issued))) ++issued;
        issued = __shfl_sync(0xffffffffu, issued, 0);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (lane == 0) {
      if (!ok) {
        raise_flag(p.status, PA_FLAG_TIMEOUT);
        s_flag[2] = 1;
      }
      s_flag[1] = issued;
    }
  } else {
    // ---------------- consumers ----------------
    // Q^T as the B operand of S^T = K Q^T, kept in registers for the split:
    // qb[kk][nt][0] holds row nt*8+g, dims 16kk + 2c, +1; [1] dims +8.
    uint32_t qb[8][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = nt * 8 + g;
      const bool live = r < w.nrows;
      const uint32_t* qrow =
          reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                            row_offset(p, w.q0, w.h, w.row0 + (live ? r : 0)));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][nt][0] = live ? __ldg(qrow + kk * 8 + c) : 0u;
        qb[kk][nt][1] = live ? __ldg(qrow + kk * 8 + 4 + c) : 0u;
      }
    }
    // Causal limit of this thread's rows (nt*8 + 2c + e); rows past the group
    // get -1, i.e. fully masked.
    int limit[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = nt * 8 + 2 * c + e;
        limit[nt][e] = r < w.nrows ? row_limit(p, w.L, w.nq, w.row0 + r) : -1;
      }

    const int new0 = w.L - w.nq;  // first position of a new (verify) token

    for (int j = warp; j < nblk; j += kMmaConsumers) {
      const int s = j % kStages;
      if (!mbar_wait(bar_full + 8 * s, (j / kStages) & 1, p.wait_limit_ns)) {
        raise_flag(p.status, PA_FLAG_TIMEOUT);
        s_flag[2] = 1;
        break;
      }
      const uint32_t kt = base + MmaSmem::stages + s * kStageBytes;
      const uint32_t vt = kt + kTileBytes;
      uint8_t* kt_ptr = sbase + MmaSmem::stages + s * kStageBytes;
      uint8_t* vt_ptr = kt_ptr + kTileBytes;
      const int tok0 = w.t0 + j * kBlockSize;

      // Zero the V rows past the context, so that 0 x (stale row) stays 0.
      // The producer has done so, and patched the tile, for a block holding
      // new tokens.
      bool patched = false;
      const int valid = min(kBlockSize, w.L - tok0);  // rows of this block inside the context
      if (valid < kBlockSize && !(p.fused_write && tok0 + kBlockSize > new0)) {
        for (int e = lane; e < (kBlockSize - valid) * 16; e += 32) {
          const int t = valid + (e >> 4), ch = e & 15;
          *reinterpret_cast<uint4*>(vt_ptr + tile_off(t, ch)) = make_uint4(0, 0, 0, 0);
        }
        patched = true;
      }
      if (patched) __syncwarp();

      attend_block<NT>(kt, vt, qb, limit, tok0, p.scale_log2, ln, st);

      // Hand the stage back to the producer. Generic-proxy writes made above
      // must be ordered before the next TMA write into this stage.
      if (patched) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    st.reduce_l();  // row sums were kept per lane (over its tokens)
  }
  __syncthreads();
  pdl_launch_dependents();  // the merge kernel (if any) may start launching

  if (s_flag[2]) {
    // A wait gave up: let every load already issued land (bounded) before the
    // CTA leaves, and write nothing.
    if (threadIdx.x == 0) {
      const int issued = s_flag[1];
      const int new0 = w.L - w.nq;
      const int jf = (p.fused_write && w.t1 > new0) ? max(0, new0 - w.t0) / kBlockSize : nblk;
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        if (j >= jf)
          (void)mbar_wait(bar_land + 8 * (j % kStages), ((j - jf) / kStages) & 1);
        else
          (void)mbar_wait(bar_full + 8 * (j % kStages), (j / kStages) & 1);
      }
    }
    __syncthreads();
    return;
  }

  // Every stage has been consumed; the ring now holds the cross-warp combine.
  float* cbuf = reinterpret_cast<float*>(sbase + MmaSmem::stages);
  if (warp < kMmaConsumers) {
    float* mine = cbuf + warp * kRowSlots * kCombineStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + 2 * c, d = mt * 16 + g;
        mine[r * kCombineStride + d] = st.o[mt][nt][0];
        mine[(r + 1) * kCombineStride + d] = st.o[mt][nt][1];
        mine[r * kCombineStride + d + 8] = st.o[mt][nt][2];
        mine[(r + 1) * kCombineStride + d + 8] = st.o[mt][nt][3];
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
  split_epilogue<uint16_t>(p, w, cbuf, s_m, s_l, kMmaConsumers, s_flag);
}

size_t mma_smem_bytes() { return MmaSmem::alloc; }

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             dim3 grid, cudaStream_t stream) {
  static PerDeviceOnce once;
  const cudaError_t e = once.run([](int) {
    return cudaFuncSetAttribute(attn_mma_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, MmaSmem::alloc);
  });
  if (e != cudaSuccess) return e;
  attn_mma_kernel<NT><<<grid, kMmaThreads, MmaSmem::alloc, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

// Host entry: NT = 1 covers up to 8 query rows per (sequence, KV head),
// NT = 2 up to 16 (more rows use several row groups).
cudaError_t launch_attn_mma(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                            dim3 grid, cudaStream_t stream) {
  return p.rows > 8 ? launch_nt<2>(tk, tv, p, grid, stream) : launch_nt<1>(tk, tv, p, grid, stream);
}

}  // namespace pa
