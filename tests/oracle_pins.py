"""Pins that tie the fp64 oracle to things other than itself.

Each ``pin_*`` takes an oracle binding (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with an independent fact:

* a pure-Python brute force (tests/bruteforce.py) on tiny paged inputs;
* torch's float64 ``scaled_dot_product_attention`` (a library routine) over
  the gathered context with K/V repeated per query head;
* closed forms: one-hot V rows return the softmax weights (checked against
  scipy's softmax of numpy-computed scores), constant V rows return the
  constant, a two-token case returns the logistic function, and a one-token
  context returns V exactly;
* invariances the pages state: paged == contiguous under any relabelling of
  physical blocks (bit-identical: "A Rust inference server for Qwen2 on Apple
  Silicon", Day 3 "Correctness"), grouped-query attention == attention over
  repeat_kv-expanded K/V ("From 183 ms to 19 ms per decode step", section
  "1. Grouped attention");
* the verify rows' causal reading: row i of a verify step equals a decode
  whose context ends at that row's position;
* the cache write: a numpy fancy-index scatter, with every other byte of the
  pool unchanged.

Run as a script with a library path, it executes every pin against that
library and exits non-zero if any pin fails (used by the mutation test, which
runs each deliberately broken oracle in its own process).
"""

from __future__ import annotations

import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for _p in (ROOT, HERE):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import bruteforce  # noqa: E402
import oracle  # noqa: E402
from paged_kv_decode_pa_gb300 import inputs  # noqa: E402


def _widen(dtype):
    if dtype == "bf16":
        return lambda x: float(oracle.bf16_bits_to_f64(np.asarray([x], dtype=np.uint16))[0])
    return lambda x: float(x)


def _written(w):
    """Caches after the workload's new tokens are scattered in (numpy fancy index)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    bs = kc.shape[2]
    for i, s in enumerate(w.slot_mapping):
        if s >= 0:
            kc[:, s // bs, s % bs, :] = w.k_new[i]
            vc[:, s // bs, s % bs, :] = w.v_new[i]
    return kc, vc


def _q4(w):
    return w.q if w.q.ndim == 4 else w.q[:, None]


def _gather(cache, tables, L, bs):
    """[Hkv, L, D] float64 view of one sequence's context (numpy fancy index)."""
    t = np.arange(L)
    return oracle.to_f64(cache[:, tables[t // bs], t % bs, :])


# ---------------------------------------------------------------------------

def pin_bruteforce(orc):
    cases = [
        dict(batch=2, q_heads=4, kv_heads=2, context_lens=(5, 11), num_blocks=12, dtype="bf16",
             seed=11, head_dim=8, block_size=4),
        dict(batch=3, q_heads=3, kv_heads=1, context_lens=(1, 7, 13), num_blocks=16, dtype="f32",
             seed=12, head_dim=8, block_size=4),
        dict(batch=2, q_heads=4, kv_heads=2, context_lens=(6, 9), num_blocks=10, dtype="bf16",
             seed=13, head_dim=16, block_size=4, num_queries=3),
        dict(batch=2, q_heads=6, kv_heads=3, context_lens=(17, 3), num_blocks=9, dtype="f32",
             seed=14, head_dim=8, block_size=8, num_queries=2),
    ]
    for c in cases:
        w = inputs.custom(**c)
        kc, vc = _written(w)
        got = orc.attend(kc, vc, _q4(w), w.block_tables, w.context_lens, w.scale)
        ref = np.asarray(bruteforce.attend(kc, vc, _q4(w), w.block_tables, w.context_lens,
                                           w.scale, _widen(c["dtype"])))
        err = np.max(np.abs(got - ref))
        assert err <= 1e-12, f"brute force mismatch {err} for {c}"


def pin_sdpa(orc):
    import torch
    import torch.nn.functional as F

    cases = [
        dict(batch=3, q_heads=12, kv_heads=2, context_lens=(40, 77, 130), num_blocks=64,
             dtype="bf16", seed=21),
        dict(batch=2, q_heads=16, kv_heads=8, context_lens=(23, 70), num_blocks=16, dtype="bf16",
             seed=22, num_queries=4),
        dict(batch=2, q_heads=4, kv_heads=4, context_lens=(33, 5), num_blocks=8, dtype="f32",
             seed=23, num_queries=2),
    ]
    for c in cases:
        w = inputs.custom(**c)
        kc, vc = _written(w)
        q4 = _q4(w)
        got = orc.attend(kc, vc, q4, w.block_tables, w.context_lens, w.scale)
        bs = kc.shape[2]
        group = c["q_heads"] // c["kv_heads"]
        nq = q4.shape[1]
        for b in range(w.spec.batch):
            L = int(w.context_lens[b])
            K = torch.from_numpy(_gather(kc, w.block_tables[b], L, bs)).repeat_interleave(group, 0)
            V = torch.from_numpy(_gather(vc, w.block_tables[b], L, bs)).repeat_interleave(group, 0)
            Q = torch.from_numpy(oracle.to_f64(q4[b])).transpose(0, 1)  # [Hq, nq, D]
            pos = torch.arange(L)
            qpos = torch.arange(L - nq, L)
            mask = pos[None, :] <= qpos[:, None]  # [nq, L], True = attend
            ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=w.scale)
            err = np.max(np.abs(got[b] - ref.transpose(0, 1).numpy()))
            assert err <= 1e-12, f"sdpa mismatch {err} for {c}, seq {b}"


def pin_onehot_softmax(orc):
    """V row at position t = e_t, so output element d is the weight of token d."""
    from scipy.special import softmax

    w = inputs.custom(batch=2, q_heads=4, kv_heads=2, context_lens=(37, 90), num_blocks=16,
                      dtype="f32", seed=31)
    kc = w.k_cache.copy()
    vc = np.zeros_like(w.v_cache)
    bs = kc.shape[2]
    for b in range(2):
        for t in range(int(w.context_lens[b])):
            vc[:, w.block_tables[b, t // bs], t % bs, t] = 1.0
    got = orc.attend(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    for b in range(2):
        L = int(w.context_lens[b])
        K = _gather(kc, w.block_tables[b], L, bs)
        for hq in range(4):
            scores = (K[hq // 2] @ w.q[b, hq].astype(np.float64)) * w.scale
            p = softmax(scores)
            row = got[b, hq]
            assert abs(row.sum() - 1.0) <= 1e-12, "weights do not sum to 1"
            assert np.all(row[L:] == 0.0), "weight on a position beyond the context"
            assert np.max(np.abs(row[:L] - p)) <= 1e-13, "weights differ from softmax"


def pin_constant_v(orc):
    w = inputs.custom(batch=3, q_heads=6, kv_heads=2, context_lens=(3, 50, 129), num_blocks=24,
                      dtype="bf16", seed=41, num_queries=2)
    vc = w.v_cache.copy()
    rng = np.random.default_rng(0)
    consts = inputs.f32_to_bf16_bits(rng.standard_normal((2, 128)).astype(np.float32))
    vc[:] = consts[:, None, None, :]
    got = orc.attend(w.k_cache, vc, w.q, w.block_tables, w.context_lens, w.scale)
    want = oracle.to_f64(consts)
    for hq in range(6):
        err = np.max(np.abs(got[:, :, hq, :] - want[hq // 3]))
        assert err <= 1e-12, f"constant V not returned ({err})"


def pin_single_token(orc):
    for dtype in ("bf16", "f32"):
        w = inputs.custom(batch=3, q_heads=8, kv_heads=4, context_lens=(1, 1, 1), num_blocks=8,
                          dtype=dtype, seed=51)
        kc, vc = _written(w)
        got = orc.attend(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
        for b in range(3):
            for hq in range(8):
                v = oracle.to_f64(vc[hq // 2, w.block_tables[b, 0], 0])
                assert np.array_equal(got[b, hq], v), "one-token context must return V exactly"


def pin_two_token_closed_form(orc):
    """q = [2, 0, ...], k0 = 0, k1 = e_0, v0 = e_0, v1 = e_1, scale 1/2: weights are logistic(1)."""
    d, bs = 128, 16
    one = inputs.f32_to_bf16_bits(np.float32([1.0]))[0]
    two = inputs.f32_to_bf16_bits(np.float32([2.0]))[0]
    kc = np.zeros((1, 2, bs, d), np.uint16)
    vc = np.zeros((1, 2, bs, d), np.uint16)
    kc[0, 1, 1, 0] = one          # token 1's key (block 1, row 1); token 0's key is zero
    vc[0, 1, 0, 0] = one          # token 0's value = e_0
    vc[0, 1, 1, 1] = one          # token 1's value = e_1
    q = np.zeros((1, 1, d), np.uint16)
    q[0, 0, 0] = two
    got = orc.attend(kc, vc, q, np.array([[1]], np.int32), np.array([2], np.int32), 0.5)
    e = math.e
    assert abs(got[0, 0, 0] - 1 / (1 + e)) <= 1e-15
    assert abs(got[0, 0, 1] - e / (1 + e)) <= 1e-15
    assert np.all(got[0, 0, 2:] == 0.0)


def pin_block_permutation(orc):
    w = inputs.custom(batch=4, q_heads=6, kv_heads=2, context_lens=(5, 40, 64, 100), num_blocks=32,
                      dtype="bf16", seed=61, num_queries=2)
    kc, vc = _written(w)
    base = orc.attend(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    perm = np.random.default_rng(7).permutation(32).astype(np.int32)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[:, perm] = kc
    vc2[:, perm] = vc
    got = orc.attend(kc2, vc2, w.q, perm[w.block_tables], w.context_lens, w.scale)
    assert np.array_equal(base, got), "result depends on physical block ids"


def pin_gqa_repeat(orc):
    w = inputs.custom(batch=2, q_heads=12, kv_heads=2, context_lens=(30, 81), num_blocks=16,
                      dtype="bf16", seed=71)
    kc, vc = _written(w)
    got = orc.attend(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    kx = np.ascontiguousarray(np.repeat(kc, 6, axis=0))
    vx = np.ascontiguousarray(np.repeat(vc, 6, axis=0))
    ref = orc.attend(kx, vx, w.q, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(got, ref), "grouped-query != attention over repeated K/V"


def pin_verify_rows(orc):
    nq = 4
    w = inputs.custom(batch=3, q_heads=8, kv_heads=4, context_lens=(4, 21, 70), num_blocks=16,
                      dtype="bf16", seed=81, num_queries=nq)
    kc, vc = _written(w)
    got = orc.attend(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
    for i in range(nq):
        lens_i = (w.context_lens - nq + i + 1).astype(np.int32)
        ref = orc.attend(kc, vc, np.ascontiguousarray(w.q[:, i]), w.block_tables, lens_i, w.scale)
        assert np.array_equal(got[:, i], ref), f"verify row {i} != decode at its own position"
    one = inputs.custom(batch=3, q_heads=8, kv_heads=4, context_lens=(4, 21, 70), num_blocks=16,
                        dtype="bf16", seed=81, num_queries=1)
    a = orc.attend(one.k_cache, one.v_cache, one.q[:, None], one.block_tables, one.context_lens,
                   one.scale)[:, 0]
    b = orc.attend(one.k_cache, one.v_cache, one.q, one.block_tables, one.context_lens, one.scale)
    assert np.array_equal(a, b), "verify with one query != decode"


def pin_zero_length(orc):
    w = inputs.custom(batch=2, q_heads=4, kv_heads=2, context_lens=(0, 9), num_blocks=4,
                      dtype="bf16", seed=91)
    got = orc.attend(w.k_cache, w.v_cache, w.q, w.block_tables, w.context_lens, w.scale)
    assert np.all(got[0] == 0.0) and np.all(np.isfinite(got[1]))
    v = inputs.custom(batch=1, q_heads=4, kv_heads=2, context_lens=(2,), num_blocks=4,
                      dtype="bf16", seed=92, num_queries=4)
    got = orc.attend(v.k_cache, v.v_cache, v.q, v.block_tables, v.context_lens, v.scale)
    assert np.all(got[0, :2] == 0.0), "verify rows before position 0 must be zero"


def pin_cache_write(orc):
    for dtype in ("bf16", "f32"):
        w = inputs.custom(batch=5, q_heads=4, kv_heads=2, context_lens=(3, 16, 17, 40, 64),
                          num_blocks=24, dtype=dtype, seed=101, num_queries=3)
        slots = w.slot_mapping.copy()
        slots[4] = -1  # a token with no slot is skipped
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        kr, vr = w.k_cache.copy(), w.v_cache.copy()
        bad = orc.cache_write(kc, vc, w.k_new, w.v_new, slots)
        assert bad == 0
        bs = kr.shape[2]
        ok = slots >= 0
        kr[:, slots[ok] // bs, slots[ok] % bs, :] = w.k_new[ok].transpose(1, 0, 2)
        vr[:, slots[ok] // bs, slots[ok] % bs, :] = w.v_new[ok].transpose(1, 0, 2)
        assert kc.tobytes() == kr.tobytes() and vc.tobytes() == vr.tobytes()
        big = slots.copy()
        big[0] = 24 * 16  # one past the pool
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        assert orc.cache_write(kc, vc, w.k_new, w.v_new, big) == 1


ALL_PINS = [pin_bruteforce, pin_sdpa, pin_onehot_softmax, pin_constant_v, pin_single_token,
            pin_two_token_closed_form, pin_block_permutation, pin_gqa_repeat, pin_verify_rows,
            pin_zero_length, pin_cache_write]


if __name__ == "__main__":
    orc = oracle.Oracle(sys.argv[1])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError as exc:
            failed.append(f"{pin.__name__}: {exc}")
        except Exception as exc:  # a broken oracle may also raise
            failed.append(f"{pin.__name__}: {type(exc).__name__}: {exc}")
    for f in failed:
        print("FAILED", f)
    sys.exit(1 if failed else 0)
