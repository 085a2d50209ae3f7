"""pa_verify (fused write + causal k+1 attention) against the oracle (GPU)."""

import numpy as np
import pytest

from gpu_util import assert_close, gpu_decode, gpu_verify, oracle_verify_of, to_f64, workload
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_verify_c5_matches_oracle(kernel):
    w = workload("c5")
    ref, okc, ovc = oracle_verify_of(w)
    out, gk, gv = gpu_verify(w, kernel=kernel)
    assert gk.tobytes() == okc.tobytes(), "fused K write differs from the oracle's scatter"
    assert gv.tobytes() == ovc.tobytes(), "fused V write differs from the oracle's scatter"
    assert_close(to_f64(out), ref, "bf16", f"c5 {kernel}")


@pytest.mark.parametrize("nq,hq,hkv", [(2, 12, 2), (3, 16, 8), (5, 12, 2), (4, 32, 4), (1, 16, 8)])
@pytest.mark.parametrize("split", [0, 16, 48])
def test_verify_shapes(nq, hq, hkv, split):
    """Row groups beyond 16 rows, new tokens straddling block and split edges."""
    lens = tuple(max(nq, x) for x in (1, 5, 16, 17, 18, 47, 48, 49, 300, 513))
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=80,
                      dtype="bf16", seed=nq * 1000 + hq, num_queries=nq)
    if nq == 1:
        w.q = w.q[:, None]
    ref, okc, ovc = oracle_verify_of(w)
    for kernel in ("auto", "simt"):
        out, gk, gv = gpu_verify(w, split_tokens=split, kernel=kernel)
        assert gk.tobytes() == okc.tobytes() and gv.tobytes() == ovc.tobytes()
        assert_close(to_f64(out), ref, "bf16", f"verify nq={nq} {hq}/{hkv} {kernel} split {split}")


def test_verify_fp32():
    w = inputs.custom(batch=4, q_heads=12, kv_heads=2, context_lens=(3, 20, 64, 130), num_blocks=24,
                      dtype="f32", seed=77, num_queries=3)
    ref, okc, ovc = oracle_verify_of(w)
    out, gk, gv = gpu_verify(w)
    assert gk.tobytes() == okc.tobytes()
    assert_close(to_f64(out), ref, "f32", "verify fp32")


def test_one_query_verify_equals_write_then_decode():
    w = inputs.custom(batch=6, q_heads=12, kv_heads=2, context_lens=(1, 16, 17, 200, 512, 999),
                      num_blocks=128, dtype="bf16", seed=31, num_queries=1)
    dec, dk, dv = gpu_decode(w)
    v = inputs.custom(batch=6, q_heads=12, kv_heads=2, context_lens=(1, 16, 17, 200, 512, 999),
                      num_blocks=128, dtype="bf16", seed=31, num_queries=1)
    v.q = v.q[:, None]
    ver, vk, vv = gpu_verify(v)
    assert vk.tobytes() == dk.tobytes() and vv.tobytes() == dv.tobytes()
    assert np.array_equal(ver[:, 0], dec), "fused one-token verify must equal write + decode bit for bit"


def _with_negative_slots(w, which):
    slots = w.slot_mapping.copy()
    slots[list(which)] = -1
    w.slot_mapping = slots
    return w


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 4)])
def test_verify_negative_slots(kernel, hq, hkv):
    """A new token with a negative slot is not written, and attention sees the
    pool's row at its position: the fused call equals the append (which skips
    the token) followed by attention over the pool. One and two row groups."""
    nq = 4
    w = inputs.custom(batch=4, q_heads=hq, kv_heads=hkv, context_lens=(4, 17, 33, 300), num_blocks=64,
                      dtype="bf16", seed=4321 + hq, num_queries=nq)
    # Sequence 0's second token, sequence 1's first two, sequence 3's last.
    w = _with_negative_slots(w, (1, 4, 5, 15))
    ref, okc, ovc = oracle_verify_of(w)
    out, gk, gv = gpu_verify(w, kernel=kernel)
    assert gk.tobytes() == okc.tobytes() and gv.tobytes() == ovc.tobytes()
    assert_close(to_f64(out), ref, "bf16", f"negative slots {hq}/{hkv} {kernel}")


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("split", [0, 48])
def test_verify_many_new_tokens(kernel, split):
    """100 new tokens per sequence, one query head per KV head: seven row
    groups, and (unsplit) more blocks holding new tokens than a CTA's ring has
    stages. Some new tokens have negative slots."""
    nq = 100
    w = inputs.custom(batch=3, q_heads=4, kv_heads=4, context_lens=(100, 150, 700), num_blocks=80,
                      dtype="bf16", seed=2468, num_queries=nq)
    w = _with_negative_slots(w, (7, 99, 100 + 50, 200 + 98))
    ref, okc, ovc = oracle_verify_of(w)
    out, gk, gv = gpu_verify(w, kernel=kernel, split_tokens=split)
    assert gk.tobytes() == okc.tobytes() and gv.tobytes() == ovc.tobytes()
    assert_close(to_f64(out), ref, "bf16", f"100 new tokens {kernel} split {split}")
