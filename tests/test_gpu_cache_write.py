"""pa_cache_write against the oracle's scatter: bit-exact, whole pool (GPU)."""

import numpy as np
import pytest

import oracle
from gpu_util import workload

pytestmark = pytest.mark.gpu


def _run(w, slots):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    pa.pa_cache_write(kc, vc, pa.to_torch(w.k_new), pa.to_torch(w.v_new), pa.to_torch(slots))
    torch.cuda.synchronize()
    return pa.to_numpy(kc), pa.to_numpy(vc)


@pytest.mark.parametrize("name", ["c1", "c2", "c5"])
def test_write_is_bit_exact(name):
    w = workload(name)
    gk, gv = _run(w, w.slot_mapping)
    ok, ov = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.cache_write(ok, ov, w.k_new, w.v_new, w.slot_mapping) == 0
    # whole pool, including every byte that must not change (NaN rows compare as bytes)
    assert gk.tobytes() == ok.tobytes()
    assert gv.tobytes() == ov.tobytes()


def test_negative_and_out_of_range_slots_are_skipped():
    w = workload("c2")
    slots = w.slot_mapping.copy()
    slots[3] = -1
    slots[5] = w.spec.num_blocks * 16 + 7  # beyond the pool: skipped, nothing written
    gk, gv = _run(w, slots)
    ok, ov = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.cache_write(ok, ov, w.k_new, w.v_new, slots) == 1
    assert gk.tobytes() == ok.tobytes() and gv.tobytes() == ov.tobytes()


def test_empty_write_is_a_no_op():
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = workload("c1")
    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    empty = torch.empty((0, 2, 128), dtype=kc.dtype, device=kc.device)
    pa.pa_cache_write(kc, vc, empty, empty, torch.empty(0, dtype=torch.int32, device=kc.device))
    torch.cuda.synchronize()
    assert np.array_equal(pa.to_numpy(kc), w.k_cache, equal_nan=True)
