"""pa_decode against the fp64 oracle on the five workloads' decode configs (GPU).

c1 is fp32 (tolerance 1e-5); c2-c4 are bf16 (|err| <= 3e-3 + 1e-2 |ref|).
c4 (8 x 32768 tokens) runs at full size in the launch configuration the
benchmark times: default split, split-K with the log-sum-exp merge.
"""

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, gpu_decode, oracle_decode, to_f64, workload
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4"])
def test_decode_matches_oracle(name):
    w = workload(name)
    ref, okc, ovc = oracle_decode(name)
    out, gk, gv = gpu_decode(w)
    assert gk.tobytes() == okc.tobytes() and gv.tobytes() == ovc.tobytes()
    assert_close(to_f64(out), ref, w.spec.dtype, name)


@pytest.mark.parametrize("kernel", ["mma", "simt"])
@pytest.mark.parametrize("split", [16, 64, 128, 8192])
def test_split_sizes_and_kernels(kernel, split):
    w = workload("c2")
    ref, _, _ = oracle_decode("c2")
    out, _, _ = gpu_decode(w, kernel=kernel, split_tokens=split)
    assert_close(to_f64(out), ref, "bf16", f"c2 {kernel} split {split}")


def test_simt_on_long_context():
    w = workload("c4")
    ref, _, _ = oracle_decode("c4")
    out, _, _ = gpu_decode(w, kernel="simt")
    assert_close(to_f64(out), ref, "bf16", "c4 simt")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hq,hkv", [(12, 2), (16, 8), (8, 8), (16, 1), (32, 2)])
def test_ragged_shapes(dtype, hq, hkv):
    """Lengths 1..3 blocks plus ragged tails, several tiles, GQA 1..16, 1..2 row groups."""
    lens = (1, 2, 15, 16, 17, 31, 33, 100, 511, 512, 513, 1025)
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=200,
                      dtype=dtype, seed=hq * 100 + hkv)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.cache_write(kc, vc, w.k_new, w.v_new, w.slot_mapping)
    ref = oracle.decode(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    kernels = ("auto", "simt") if dtype == "bf16" else ("auto",)
    for kernel in kernels:
        for split in (0, 32):
            out, _, _ = gpu_decode(w, split_tokens=split, kernel=kernel)
            assert_close(to_f64(out), ref, dtype, f"{dtype} {hq}/{hkv} {kernel} split {split}")


def test_zero_length_gives_zeros():
    w = inputs.custom(batch=3, q_heads=12, kv_heads=2, context_lens=(0, 5, 0), num_blocks=8,
                      dtype="bf16", seed=5)
    out, _, _ = gpu_decode(w, write=False)
    assert np.all(to_f64(out[0]) == 0) and np.all(to_f64(out[2]) == 0)
    ref = oracle.decode(w.k_cache, w.v_cache, w.q, w.block_tables, w.context_lens, w.scale)
    assert_close(to_f64(out), ref, "bf16", "zero length")


@pytest.mark.parametrize("split", [0, 64])
def test_max_sizes_single_sequence_long(split):
    """One long sequence: many splits plus a ragged tail, merged (split 64 gives
    513 splits, more than one 256-split chunk of the merge)."""
    L = 32768 + 17
    w = inputs.custom(batch=1, q_heads=12, kv_heads=2, context_lens=(L,), num_blocks=(L + 15) // 16 + 1,
                      dtype="bf16", seed=9)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.cache_write(kc, vc, w.k_new, w.v_new, w.slot_mapping)
    ref = oracle.decode(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    out, _, _ = gpu_decode(w, split_tokens=split)
    assert_close(to_f64(out), ref, "bf16", f"long single split {split}")
