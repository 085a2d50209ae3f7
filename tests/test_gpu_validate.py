"""pa_validate and the in-kernel range checks on bad device indices (GPU).

Bad indices are safe by construction: a bad block id becomes a TMA coordinate
outside the tensor (zeros are read) or is skipped on the CUDA-core path; a
slot outside the pool is skipped; a length above the limits is clamped.
"""

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, to_f64
from paged_kv_decode_pa_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _dev(w):
    import paged_kv_decode_pa_gb300 as pa

    return {k: pa.to_torch(getattr(w, k)) for k in
            ("k_cache", "v_cache", "q", "block_tables", "context_lens", "slot_mapping")}


def test_validate_counts_bad_entries():
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=4, q_heads=12, kv_heads=2, context_lens=(5, 40, 70, 16), num_blocks=64,
                      dtype="bf16", seed=41)
    d = _dev(w)
    rep = pa.pa_validate(d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                         w.max_context_len, d["slot_mapping"], 1)
    torch.cuda.synchronize()
    assert rep.cpu().tolist() == [0, 0, 0, 0]

    tables = w.block_tables.copy()
    tables[1, 1] = 64          # one past the pool
    tables[2, 0] = -5
    lens = w.context_lens.copy()
    lens[3] = 10 ** 6          # beyond max_context_len
    slots = w.slot_mapping.copy()
    slots[0] = slots[0] + 1    # not the slot of its position
    rep = pa.pa_validate(d["k_cache"], d["v_cache"], pa.to_torch(tables), pa.to_torch(lens),
                         w.max_context_len, pa.to_torch(slots), 1)
    torch.cuda.synchronize()
    flags, bad_len, bad_blk, bad_slot = rep.cpu().tolist()
    assert bad_len == 1 and bad_blk == 2 and bad_slot >= 1
    assert flags == _lib.PA_FLAG_BAD_LENGTH | _lib.PA_FLAG_BAD_BLOCK | _lib.PA_FLAG_BAD_SLOT


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_decode_flags_bad_ids_and_reads_nothing_outside(kernel):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=3, q_heads=12, kv_heads=2, context_lens=(40, 40, 40), num_blocks=16,
                      dtype="bf16", seed=43)
    tables = w.block_tables.copy()
    tables[1, 1] = 1 << 30
    d = _dev(w)
    ws = pa.new_workspace(3, 1, 12, 2, 40)
    out = pa.pa_decode(d["k_cache"], d["v_cache"], d["q"], pa.to_torch(tables), d["context_lens"], 40,
                       w.scale, ws, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) & _lib.PA_FLAG_BAD_BLOCK
    good = pa.pa_decode(d["k_cache"], d["v_cache"], d["q"], d["block_tables"], d["context_lens"], 40,
                        w.scale, ws, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    o, g = pa.to_numpy(out), pa.to_numpy(good)
    assert np.array_equal(o[[0, 2]], g[[0, 2]]), "a bad id in one sequence changed another"
    # The bad block reads as zeros: the oracle over a pool with one extra all-zero block in its place.
    kz = np.concatenate([w.k_cache, np.zeros_like(w.k_cache[:, :1])], axis=1)
    vz = np.concatenate([w.v_cache, np.zeros_like(w.v_cache[:, :1])], axis=1)
    tz = w.block_tables.copy()
    tz[1, 1] = w.spec.num_blocks
    ref = oracle.decode(kz, vz, w.q, tz, w.context_lens, w.scale)
    assert_close(to_f64(o[[1]]), ref[[1]], "bf16", f"{kernel}: bad block read as zeros")


def test_int8_decode_bad_id_reads_a_zero_block():
    """The int8 pool's tensor loads read zeros (codes and scales) past the pool:
    the values are those of an all-zero block, and other sequences are untouched."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=3, q_heads=12, kv_heads=2, context_lens=(40, 40, 40), num_blocks=16,
                      dtype="bf16", seed=47)
    pool = inputs.q8_pool(w)
    kq, vq, ks, vs = (pa.to_torch(a) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))
    tables = w.block_tables.copy()
    tables[1, 1] = 1 << 30
    ws = pa.new_workspace(3, 1, 12, 2, 40)
    out = pa.pa_decode(kq, vq, pa.to_torch(w.q), pa.to_torch(tables), pa.to_torch(w.context_lens), 40, w.scale, ws,
                       k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) & _lib.PA_FLAG_BAD_BLOCK
    o = pa.to_numpy(out)

    def extend(a, fill):
        return np.concatenate([a, np.full_like(a[:, :1], fill)], axis=1)

    tz = w.block_tables.copy()
    tz[1, 1] = w.spec.num_blocks
    ref = oracle.decode_q8(extend(pool.k_codes, 128), extend(pool.v_codes, 128), extend(pool.k_scale, 0),
                           extend(pool.v_scale, 0), w.q, tz, w.context_lens, w.scale)
    assert_close(to_f64(o), ref, "bf16", "int8: bad block read as zeros")
