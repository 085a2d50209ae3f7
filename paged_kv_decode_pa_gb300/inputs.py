"""Seeded synthetic inputs for paged-KV decode attention.

This module holds no attention arithmetic. It draws random numbers, rounds
them to the storage type, assigns physical blocks and builds the per-step
inputs (block tables, context lengths, slot mappings) that an engine would
hand to the kernels. Both the CUDA path (tests, benchmark) and the CPU oracle
(tests) are fed from here, and nothing here depends on either.

The pages describe the inputs but publish no tensors, so every workload is a
synthetic stand-in with the pages' shapes:

* 16-token blocks in a fixed pool, one block table per sequence ("A Rust
  inference server for Qwen2 on Apple Silicon", Day 3; "From 183 ms to 19 ms
  per decode step", section "4. CUDA graphs per batch bucket").
* head-major caches [kv_heads, num_blocks, block_size, head_dim] ("From 183 ms
  to 19 ms per decode step", section "2. Head-major KV cache").
* Qwen2-1.5B heads, 12 query / 2 KV, head_dim 128 ("A Rust inference server
  for Qwen2 on Apple Silicon", "Target architecture").
* a spare block that only padded rows touch ("From 183 ms to 19 ms per decode
  step", section "4. CUDA graphs per batch bucket").
* k + 1 query tokens per sequence for verify ("From 183 ms to 19 ms per decode
  step", section "Then speculative decoding got slower").

Values are N(0, 1) drawn with numpy's PCG64 and rounded to bf16 with
round-to-nearest-even (or kept as float32). Cache rows that no sequence
reads (unused blocks, and the rows of a last block beyond its sequence's
length) hold NaN, so any kernel that lets a masked or unused row leak into a
result fails loudly.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

HEAD_DIM = 128
BLOCK_SIZE = 16

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits.

    Inputs are finite draws from N(0, 1); no NaN or overflow handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Spec:
    """Shape and recipe of one synthetic workload."""

    name: str
    batch: int
    q_heads: int
    kv_heads: int
    num_blocks: int
    dtype: str  # "bf16" or "f32"
    seed: int
    context_lens: tuple = ()          # explicit lengths (overrides the range below)
    len_range: tuple = (0, 0)         # inclusive uniform range of prior context
    len_offset: int = 0               # added to every drawn length
    num_queries: int = 1              # 1 = decode; k + 1 for verify
    spare_block: bool = False         # reserve the last block as the padding block
    padded_rows: int = 0              # trailing rows that only touch the spare block
    permute_whole_pool: bool = False  # block ids drawn from a permutation of the whole pool
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    description: str = ""


# The five workloads of the hot-path scope, in order (tiny fp32, Qwen2-1.5B
# decode, 64-sequence decode with a spare block, 32k context, verify).
CONFIGS = {
    "c1": Spec("c1", batch=4, q_heads=12, kv_heads=2, num_blocks=32, dtype="f32", seed=1,
               context_lens=(1, 17, 33, 64), permute_whole_pool=True,
               description="tiny fp32 decode: 4 seqs, lens {1,17,33,64}, 12/2 heads, 32-block pool"),
    "c2": Spec("c2", batch=32, q_heads=12, kv_heads=2, num_blocks=4096, dtype="bf16", seed=2,
               len_range=(64, 512),
               description="Qwen2-1.5B-shaped decode: 32 seqs, lens U[64,512], 12/2 heads, 4096 blocks"),
    "c3": Spec("c3", batch=64, q_heads=16, kv_heads=8, num_blocks=8192, dtype="bf16", seed=3,
               len_range=(0, 256), len_offset=256, spare_block=True,
               description="Qwen3-0.6B-shaped decode: 64 seqs, lens 256+U[0,256], 16/8 heads, "
                           "8192 blocks, spare block 8191"),
    "c4": Spec("c4", batch=8, q_heads=12, kv_heads=2, num_blocks=16384, dtype="bf16", seed=4,
               context_lens=(32768,) * 8, permute_whole_pool=True,
               description="long-context decode: 8 seqs at 32768, 12/2 heads, 16384-block pool"),
    "c5": Spec("c5", batch=64, q_heads=16, kv_heads=8, num_blocks=8192, dtype="bf16", seed=5,
               len_range=(128, 1024), len_offset=5, num_queries=5,
               description="speculative verify: 64 seqs x 5 queries, prior U[128,1024], 16/8 heads, "
                           "8192 blocks, fused write of 320 new tokens"),
}


@dataclass
class Workload:
    spec: Spec
    k_cache: np.ndarray        # [kv_heads, num_blocks, block_size, head_dim] (uint16 bf16 bits or float32)
    v_cache: np.ndarray
    q: np.ndarray              # decode: [batch, q_heads, head_dim]; verify: [batch, nq, q_heads, head_dim]
    k_new: np.ndarray          # [batch * num_queries, kv_heads, head_dim]
    v_new: np.ndarray
    slot_mapping: np.ndarray   # [batch * num_queries] int32
    block_tables: np.ndarray   # [batch, max_blocks_per_seq] int32
    context_lens: np.ndarray   # [batch] int32 (includes the new tokens)
    scale: float
    spare_block: Optional[int] = None
    real_rows: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def _draw(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def _nan_fill(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    return np.full(shape, np.nan, dtype=np.float32)


def slots_for(block_tables: np.ndarray, context_lens: np.ndarray, num_queries: int,
              block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Cache slot of each new token: token i of sequence b sits at position
    L_b - num_queries + i, in block block_tables[b, pos // block_size]; -1 when
    that position is negative."""
    batch = len(context_lens)
    slots = np.full(batch * num_queries, -1, dtype=np.int32)
    for b in range(batch):
        for i in range(num_queries):
            pos = int(context_lens[b]) - num_queries + i
            if pos >= 0:
                slots[b * num_queries + i] = int(block_tables[b, pos // block_size]) * block_size + pos % block_size
    return slots


def generate(spec: Spec, seed: Optional[int] = None) -> Workload:
    """Build one seeded workload from a Spec (see CONFIGS for the five standard ones)."""
    rng = np.random.Generator(np.random.PCG64(spec.seed if seed is None else seed))
    bs, d, hkv, hq, nq = spec.block_size, spec.head_dim, spec.kv_heads, spec.q_heads, spec.num_queries
    assert hq % hkv == 0
    real = spec.batch - spec.padded_rows
    spare = spec.num_blocks - 1 if (spec.spare_block or spec.padded_rows) else None

    # Context lengths (they count the tokens being decoded or verified).
    if spec.context_lens:
        lens = np.asarray(spec.context_lens, dtype=np.int64)
        assert lens.size == spec.batch
    else:
        lo, hi = spec.len_range
        lens = rng.integers(lo, hi + 1, size=spec.batch, dtype=np.int64) + spec.len_offset
    if spec.padded_rows:
        lens[real:] = rng.integers(max(nq, 1), bs + 1, size=spec.padded_rows)

    # Physical blocks: a seeded permutation of the pool (minus the spare), taken
    # consecutively per sequence, so neighbouring logical blocks are far apart.
    nblk = (lens + bs - 1) // bs
    pool = spec.num_blocks - (1 if spare is not None else 0)
    perm = rng.permutation(pool).astype(np.int32)
    need = int(nblk[:real].sum())
    if need > pool:
        raise ValueError(f"{spec.name}: {need} blocks needed, pool has {pool}")
    mbps = max(int(nblk.max()) if nblk.size else 1, 1)
    filler = spare if spare is not None else 0
    tables = np.full((spec.batch, mbps), filler, dtype=np.int32)
    cursor = 0
    for b in range(real):
        n = int(nblk[b])
        tables[b, :n] = perm[cursor:cursor + n]
        cursor += n
    if spec.padded_rows:
        tables[real:, :] = spare

    # Caches: NaN everywhere, then N(0, 1) rows for every position a real
    # sequence holds (the spare block gets finite rows too: padded rows read it).
    kc = _nan_fill((hkv, spec.num_blocks, bs, d), spec.dtype)
    vc = _nan_fill((hkv, spec.num_blocks, bs, d), spec.dtype)
    blk_idx, row_idx = [], []
    for b in range(real):
        t = np.arange(int(lens[b]))
        blk_idx.append(tables[b, t // bs])
        row_idx.append(t % bs)
    if spare is not None:
        blk_idx.append(np.full(bs, spare, dtype=np.int32))
        row_idx.append(np.arange(bs))
    if blk_idx:
        bi = np.concatenate(blk_idx)
        ri = np.concatenate(row_idx)
        kc[:, bi, ri, :] = _draw(rng, (hkv, bi.size, d), spec.dtype)
        vc[:, bi, ri, :] = _draw(rng, (hkv, bi.size, d), spec.dtype)

    # Queries and the new tokens' K/V with their slots: token i of sequence b
    # sits at position L_b - nq + i.
    qshape = (spec.batch, hq, d) if nq == 1 else (spec.batch, nq, hq, d)
    q = _draw(rng, qshape, spec.dtype)
    k_new = _draw(rng, (spec.batch * nq, hkv, d), spec.dtype)
    v_new = _draw(rng, (spec.batch * nq, hkv, d), spec.dtype)
    slots = slots_for(tables, lens, nq, bs)

    return Workload(spec=spec, k_cache=kc, v_cache=vc, q=q, k_new=k_new, v_new=v_new,
                    slot_mapping=slots, block_tables=tables,
                    context_lens=lens.astype(np.int32), scale=1.0 / float(np.sqrt(d)),
                    spare_block=spare, real_rows=real)


def make(name: str, **overrides) -> Workload:
    """One of the standard workloads ("c1" … "c5"), optionally with fields overridden."""
    spec = CONFIGS[name]
    if overrides:
        spec = Spec(**{**spec.__dict__, **overrides})
    return generate(spec)


def custom(batch: int, q_heads: int, kv_heads: int, context_lens, num_blocks: int,
           dtype: str = "bf16", seed: int = 0, num_queries: int = 1, spare_block: bool = False,
           padded_rows: int = 0, head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE) -> Workload:
    """A workload with explicit context lengths (used for small and edge-case tests)."""
    spec = Spec("custom", batch=batch, q_heads=q_heads, kv_heads=kv_heads, num_blocks=num_blocks,
                dtype=dtype, seed=seed, context_lens=tuple(int(x) for x in context_lens),
                num_queries=num_queries, spare_block=spare_block, padded_rows=padded_rows,
                head_dim=head_dim, block_size=block_size)
    return generate(spec)


@dataclass
class Q8Pool:
    """An int8 KV pool: bytes (value + 128) with K scales per (head, block,
    channel) and V scales per (head, block, row)."""
    k_codes: np.ndarray   # [kv_heads, num_blocks, block_size, head_dim] uint8
    v_codes: np.ndarray
    k_scale: np.ndarray   # [kv_heads, num_blocks, head_dim] float32
    v_scale: np.ndarray   # [kv_heads, num_blocks, block_size] float32


def q8_pool(w: Workload, seed: Optional[int] = None) -> Q8Pool:
    """A seeded int8 pool for a workload's tables and lengths.

    Every row a sequence holds (and the spare block's rows) gets bell-shaped
    bytes (a rounded N(0, 1) x 42 draw, clipped to [1, 255]); every other row
    holds byte 128, a zero. K scales are drawn from U(0.005, 0.05) for every
    (head, block, channel); V scales likewise for held rows and NaN for the
    rest, so a read of a row no sequence holds shows up. Draws only: no
    quantiser runs here.
    """
    s = w.spec
    rng = np.random.Generator(np.random.PCG64((s.seed if seed is None else seed) + 7919))
    hkv, nb, bs, d = s.kv_heads, s.num_blocks, s.block_size, s.head_dim
    held = np.zeros((nb, bs), dtype=bool)
    for b in range(w.real_rows):
        t = np.arange(int(w.context_lens[b]))
        held[w.block_tables[b, t // bs], t % bs] = True
    if w.spare_block is not None:
        held[w.spare_block, :] = True
    def codes():
        c = np.full((hkv, nb, bs, d), 128, dtype=np.uint8)
        draw = np.clip(np.rint(rng.standard_normal((hkv, int(held.sum()), d)) * 42.0), -127, 127)
        c[:, held, :] = (draw + 128).astype(np.uint8)
        return c
    kq, vq = codes(), codes()
    ks = rng.uniform(0.005, 0.05, size=(hkv, nb, d)).astype(np.float32)
    vs = np.full((hkv, nb, bs), np.nan, dtype=np.float32)
    vs[:, held] = rng.uniform(0.005, 0.05, size=(hkv, int(held.sum()))).astype(np.float32)
    return Q8Pool(kq, vq, ks, vs)


@dataclass
class RaggedWorkload:
    """A step whose sequences carry different numbers of new tokens."""
    base: Workload             # the uniform workload it is cut from (num_queries = the most)
    nq: np.ndarray             # [batch] new tokens of each sequence
    query_start: np.ndarray    # [batch + 1] int32
    q: np.ndarray              # [total, q_heads, head_dim]
    k_new: np.ndarray          # [total, kv_heads, head_dim]
    v_new: np.ndarray
    slot_mapping: np.ndarray   # [total] int32

    @property
    def max_queries(self) -> int:
        return int(self.nq.max()) if self.nq.size else 1


def ragged(w: Workload, nq_per_seq) -> RaggedWorkload:
    """Keep, for sequence b, the last nq_per_seq[b] of a uniform verify
    workload's new tokens (those at positions L - n_b .. L - 1). A decode
    sequence keeps one; zero keeps none."""
    nq_max = w.spec.num_queries
    n = np.asarray(nq_per_seq, dtype=np.int64)
    assert n.shape == (w.spec.batch,) and n.min() >= 0 and n.max() <= nq_max
    q4 = w.q if w.q.ndim == 4 else w.q[:, None]
    rows = [b * nq_max + i for b in range(w.spec.batch) for i in range(nq_max - int(n[b]), nq_max)]
    qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = q4.reshape(-1, *q4.shape[2:])[rows]
    return RaggedWorkload(base=w, nq=n.astype(np.int32), query_start=qs, q=np.ascontiguousarray(q),
                          k_new=np.ascontiguousarray(w.k_new[rows]), v_new=np.ascontiguousarray(w.v_new[rows]),
                          slot_mapping=np.ascontiguousarray(w.slot_mapping[rows]))
