"""Properties the pages state, checked on the CUDA path (GPU).

* paged == contiguous under any relabelling of physical blocks, bit for bit
  ("A Rust inference server for Qwen2 on Apple Silicon", Day 3 "Correctness");
* a sequence's result does not depend on its batch-mates (fixed split plan),
  and padded rows that only touch the spare block change nothing real ("From
  183 ms to 19 ms per decode step", section "4. CUDA graphs per batch bucket");
* a one-token context returns V exactly;
* masked and unused rows hold NaN in every workload, so any leak shows;
* grouped-query attention equals attention over repeated K/V.
"""

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, gpu_decode, gpu_verify, to_f64, workload
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_block_relabelling_is_bit_identical(kernel):
    w = inputs.custom(batch=5, q_heads=12, kv_heads=2, context_lens=(3, 40, 333, 600, 1100),
                      num_blocks=200, dtype="bf16", seed=17)
    base, _, _ = gpu_decode(w, kernel=kernel)
    perm = np.random.default_rng(3).permutation(200).astype(np.int32)
    w2 = inputs.custom(batch=5, q_heads=12, kv_heads=2, context_lens=(3, 40, 333, 600, 1100),
                       num_blocks=200, dtype="bf16", seed=17)
    w2.k_cache = np.empty_like(w.k_cache)
    w2.v_cache = np.empty_like(w.v_cache)
    w2.k_cache[:, perm] = w.k_cache
    w2.v_cache[:, perm] = w.v_cache
    w2.block_tables = perm[w.block_tables]
    bs = 16
    w2.slot_mapping = (perm[w.slot_mapping // bs] * bs + w.slot_mapping % bs).astype(np.int32)
    got, _, _ = gpu_decode(w2, kernel=kernel)
    assert np.array_equal(base, got)


def test_batch_invariance():
    w = workload("c2")
    full, _, _ = gpu_decode(w)
    rows = np.arange(0, 32, 3)
    sub, _, _ = gpu_decode(w, rows=rows)
    assert np.array_equal(full[rows], sub), "a sequence's output changed with its batch-mates"


_SPLIT_LENS = (100, 700, 800, 1500, 4096, 4100, 9000, 20)  # across both split thresholds


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_batch_invariance_across_split_rules(kernel):
    """Sequences on either side of the short and long default splits (one
    split, several, the long-context rule): each one's output is the same bits
    alone, in a subset, or in the whole batch."""
    w = inputs.custom(batch=len(_SPLIT_LENS), q_heads=12, kv_heads=2, context_lens=_SPLIT_LENS,
                      num_blocks=1400, dtype="bf16", seed=29)
    full, _, _ = gpu_decode(w, kernel=kernel, write=False)
    for rows in ([6], [2, 5], [0, 3, 7, 1], [4]):
        sub, _, _ = gpu_decode(w, kernel=kernel, write=False, rows=np.array(rows))
        assert np.array_equal(full[rows], sub), f"rows {rows}: output changed with the batch-mates"


def test_int8_batch_invariance_across_split_rules():
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=len(_SPLIT_LENS), q_heads=12, kv_heads=2, context_lens=_SPLIT_LENS,
                      num_blocks=1400, dtype="bf16", seed=31)
    pool = inputs.q8_pool(w)
    dev = torch.device("cuda")
    kq, vq, ks, vs = (pa.to_torch(a, dev) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))

    def run(rows):
        q = np.ascontiguousarray(w.q[rows])
        ws = pa.new_workspace(len(rows), 1, 12, 2, w.max_context_len, dev)
        out = pa.pa_decode(kq, vq, pa.to_torch(q, dev), pa.to_torch(np.ascontiguousarray(w.block_tables[rows]), dev),
                           pa.to_torch(np.ascontiguousarray(w.context_lens[rows]), dev), w.max_context_len,
                           w.scale, ws, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert pa.pa_workspace_status(ws) == 0
        return pa.to_numpy(out)

    full = run(np.arange(len(_SPLIT_LENS)))
    for rows in ([6], [2, 5], [0, 3, 7, 1]):
        assert np.array_equal(full[rows], run(np.array(rows))), f"int8 rows {rows}"


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_batch_invariance_across_merge_forms(kv):
    """The merge takes a warp per row while the batch's longest sequence has at
    most 8 splits and a CTA per row beyond; a sequence of a few splits must get
    the same bits under both."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    # 32 sequences of 4 to 8 splits under the long-context rule (and one short one), then a
    # 32k-token sequence whose 29 splits switch the merge to a CTA per row.
    rng = np.random.Generator(np.random.PCG64(41))
    lens = tuple(int(x) for x in rng.integers(4200, 9200, size=32)) + (800, 32768)
    w = inputs.custom(batch=len(lens), q_heads=12, kv_heads=2, context_lens=lens,
                      num_blocks=sum(-(-x // 16) for x in lens) + 8, dtype="bf16", seed=37)
    dev = torch.device("cuda")
    if kv == "int8":
        pool = inputs.q8_pool(w)
        kc, vc, ks, vs = (pa.to_torch(a, dev) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))
        scales = {"k_scale": ks, "v_scale": vs}
    else:
        kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
        scales = {}

    def run(rows):
        rows = np.array(rows)
        ws = pa.new_workspace(len(rows), 1, 12, 2, w.max_context_len, dev)
        out = pa.pa_decode(kc, vc, pa.to_torch(np.ascontiguousarray(w.q[rows]), dev),
                           pa.to_torch(np.ascontiguousarray(w.block_tables[rows]), dev),
                           pa.to_torch(np.ascontiguousarray(w.context_lens[rows]), dev), w.max_context_len,
                           w.scale, ws, **scales)
        torch.cuda.synchronize()
        assert pa.pa_workspace_status(ws) == 0
        return pa.to_numpy(out)

    n = len(lens)
    full = run(list(range(n)))
    short = list(range(n - 1))
    assert np.array_equal(full[short], run(short)), f"{kv}: outputs changed with a 32k-token batch-mate"
    assert np.array_equal(full[[n - 1]], run([n - 1]))


def test_padded_rows_touch_only_the_spare_block():
    w = workload("c3", padded_rows=7)
    full, gk, gv = gpu_decode(w)
    real, _, _ = gpu_decode(w, rows=np.arange(57))
    assert np.array_equal(full[:57], real)
    spare = w.spare_block
    keep = np.ones(w.spec.num_blocks, bool)
    keep[spare] = False
    ok, ov = w.k_cache.copy(), w.v_cache.copy()
    oracle.cache_write(ok, ov, w.k_new[:57], w.v_new[:57], w.slot_mapping[:57])
    assert gk[:, keep].tobytes() == ok[:, keep].tobytes()
    assert gv[:, keep].tobytes() == ov[:, keep].tobytes()
    ref = oracle.decode(ok, ov, w.q[:57], w.block_tables[:57], w.context_lens[:57], w.scale)
    assert_close(to_f64(full[:57]), ref, "bf16", "c3 padded, real rows")


@pytest.mark.parametrize("dtype,kernel", [("bf16", "mma"), ("bf16", "simt"), ("f32", "simt")])
def test_single_token_returns_v_exactly(dtype, kernel):
    w = inputs.custom(batch=4, q_heads=16, kv_heads=8, context_lens=(1, 1, 1, 1), num_blocks=8,
                      dtype=dtype, seed=23)
    out, _, gv = gpu_decode(w, kernel=kernel)
    for b in range(4):
        blk = w.block_tables[b, 0]
        for hq in range(16):
            assert np.array_equal(out[b, hq], gv[hq // 2, blk, 0]), "L = 1 must return V exactly"


def test_gqa_equals_repeated_kv():
    w = inputs.custom(batch=4, q_heads=12, kv_heads=2, context_lens=(9, 100, 257, 700),
                      num_blocks=100, dtype="bf16", seed=29)
    grouped, gk, gv = gpu_decode(w)
    x = inputs.custom(batch=4, q_heads=12, kv_heads=12, context_lens=(9, 100, 257, 700),
                      num_blocks=100, dtype="bf16", seed=29)
    x.k_cache = np.ascontiguousarray(np.repeat(gk, 6, axis=0))
    x.v_cache = np.ascontiguousarray(np.repeat(gv, 6, axis=0))
    x.q = w.q
    rep, _, _ = gpu_decode(x, write=False)
    # Same products, different row grouping inside the MMA tile: equal to fp32 round-off.
    np.testing.assert_allclose(to_f64(grouped), to_f64(rep), atol=4e-3, rtol=0)


def test_verify_nan_neighbours_do_not_leak():
    """Every unused cache row is NaN in the generated pools; outputs stay finite."""
    w = workload("c5")
    out, _, _ = gpu_verify(w)
    assert np.all(np.isfinite(to_f64(out)))
