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
  pool unchanged;
* the int8 pool: hand-worked codes and scales (ties to even, the +128
  offset), the requantisation of a block when a channel's maximum grows,
  order independence on the quantisation grid, the half-step error bound, and
  lossless grid values giving attention bit-identical to the bf16 pool.

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


# ---------------------------------------------------------------------------
# int8 pool ("A Rust inference server for Qwen2 on Apple Silicon", Day 4:
# "int8 KV", "Grouping is the whole question", "Partial blocks").

def _bf16(x):
    """float values -> bf16 bit patterns (the values used here are bf16-exact)."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "pin values must be exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _empty_q8(hkv, nb, bs=16, d=128):
    """A pool no row was ever written to: byte 128 (zero) everywhere, zero scales."""
    return (np.full((hkv, nb, bs, d), 128, np.uint8), np.full((hkv, nb, bs, d), 128, np.uint8),
            np.zeros((hkv, nb, d), np.float32), np.zeros((hkv, nb, bs), np.float32))


def _q8_row(d=128):
    """One row with hand-checked codes at scale 15.875 / 127 = 1/8 (exact)."""
    v = np.zeros(d, np.float32)
    v[:8] = [15.875, -15.875, 0.0, 7.9375, 7.8125, -7.8125, 0.0625, 0.1875]
    # x * (127 / 15.875 = 8) = 127, -127, 0, 63.5, 62.5, -62.5, 0.5, 1.5 -> ties go to even.
    want = np.full(d, 128, np.uint8)
    want[:8] = [255, 1, 128, 192, 190, 66, 128, 130]
    return v, want


def pin_q8_row_closed_form(orc):
    """One token into an empty block: V gets the row's own scale and the codes
    worked out by hand (x * 127 / max rounded to nearest, ties to even, +128
    offset); each K
    channel's scale is |k| / 127 (the row is the only non-zero one), its code
    +-127, and every other row stays byte 128."""
    kq, vq, ks, vs = _empty_q8(1, 2)
    v, want = _q8_row()
    row = _bf16(v)[None, None, :]
    assert orc.cache_write_q8(kq, vq, ks, vs, row, row, np.array([16 + 5], np.int32)) == 0
    assert vs[0, 1, 5] == np.float32(0.125)
    assert np.array_equal(vq[0, 1, 5], want)
    nz = v != 0
    assert np.array_equal(ks[0, 1][nz], np.abs(v[nz]) / np.float32(127)) and np.all(ks[0, 1][~nz] == 0)
    assert np.array_equal(kq[0, 1, 5][nz], np.where(v[nz] > 0, 255, 1).astype(np.uint8))
    assert np.all(kq[0, 1, 5][~nz] == 128)
    others = np.ones(16, bool)
    others[5] = False
    assert np.all(kq[0, 1][others] == 128) and np.all(vq[0, 1][others] == 128) and np.all(vs[0, 1][others] == 0)
    assert np.all(kq[0, 0] == 128) and np.all(ks[0, 0] == 0)  # the other block is untouched


def pin_q8_requant_closed_form(orc):
    """A later, larger value in a channel re-scales that channel for the whole
    block (the old row's code is recomputed at the new scale), and a channel
    whose maximum did not change keeps its codes exactly."""
    kq, vq, ks, vs = _empty_q8(1, 1)
    a = np.zeros(128, np.float32)
    a[0] = a[1] = 15.875
    b = np.zeros(128, np.float32)
    b[0], b[1] = 31.75, 1.0
    orc.cache_write_q8(kq, vq, ks, vs, _bf16(a)[None, None], _bf16(a)[None, None], np.array([0], np.int32))
    assert ks[0, 0, 0] == 0.125 and kq[0, 0, 0, 0] == 255
    orc.cache_write_q8(kq, vq, ks, vs, _bf16(b)[None, None], _bf16(b)[None, None], np.array([1], np.int32))
    assert ks[0, 0, 0] == 0.25 and ks[0, 0, 1] == 0.125
    assert kq[0, 0, 0, 0] == 192  # 15.875 * (127 / 31.75 = 4) = 63.5 -> 64
    assert kq[0, 0, 1, 0] == 255 and kq[0, 0, 0, 1] == 255 and kq[0, 0, 1, 1] == 136  # 1 * 8 = 8
    # V rows are independent: the first row's V is untouched by the second write.
    assert vs[0, 0, 0] == 0.125 and vs[0, 0, 1] == 0.25 and vq[0, 0, 0, 0] == 255


def pin_q8_zero_and_partial_block(orc):
    """An all-zero row has scale 0, bytes 128 and dequantises to 0. Rows on the
    quantisation grid fill a block to the same bytes whether they come one per
    call or all in one call: unwritten rows are zeros and cannot raise a
    maximum, and requantising at an unchanged scale returns each code."""
    kq, vq, ks, vs = _empty_q8(1, 1)
    z = np.zeros((1, 1, 128), np.uint16)
    orc.cache_write_q8(kq, vq, ks, vs, z, z, np.array([3], np.int32))
    assert vs[0, 0, 3] == 0 and np.all(vq[0, 0, 3] == 128) and np.all(ks == 0)
    ko, vo = orc.dequant_q8(kq, vq, ks, vs)
    assert np.all(ko == 0) and np.all(vo == 0)

    rng = np.random.default_rng(11)
    ints = rng.integers(-126, 127, size=(4, 128))
    ints[0] = np.where(rng.random(128) < 0.5, 127, -127)  # row 0 holds every channel's maximum
    rows = _bf16(ints.astype(np.float32) / 8)[:, None, :]
    one = _empty_q8(1, 1)
    orc.cache_write_q8(*one, rows, rows, np.arange(4, dtype=np.int32))
    step = _empty_q8(1, 1)
    for r in range(4):
        orc.cache_write_q8(*step, rows[r:r + 1], rows[r:r + 1], np.array([r], np.int32))
    for x, y in zip(one, step):
        assert np.array_equal(x, y)
    assert np.array_equal(one[0][0, 0, :4], (ints + 128).astype(np.uint8))  # lossless on the grid


def pin_q8_error_bound(orc):
    """Every dequantised element is within half a step of its bf16 input: the
    error is about scale / 2 per element ("Grouping is the whole question")."""
    rng = np.random.default_rng(12)
    n, hkv = 40, 2
    vals = (rng.standard_normal((n, hkv, 128)) * rng.uniform(0.1, 8, size=(n, 1, 1))).astype(np.float32)
    vals = ((vals.view(np.uint32) + 0x8000) & 0xFFFF0000).view(np.float32)  # to bf16 values
    k_new, v_new = _bf16(vals), _bf16(vals[::-1].copy())
    slots = rng.permutation(4 * 16)[:n].astype(np.int32)  # several rows per block
    kq, vq, ks, vs = _empty_q8(hkv, 4)
    assert orc.cache_write_q8(kq, vq, ks, vs, k_new, v_new, slots) == 0
    ko, vo = orc.dequant_q8(kq, vq, ks, vs)
    xk = np.zeros((hkv, 4, 16, 128), np.float32)
    xv = np.zeros((hkv, 4, 16, 128), np.float32)
    xk[:, slots // 16, slots % 16] = vals.transpose(1, 0, 2)
    xv[:, slots // 16, slots % 16] = vals[::-1].transpose(1, 0, 2)
    sk = np.abs(xk).max(axis=2, keepdims=True) / 127  # per channel over the block's rows
    sv = np.abs(xv).max(axis=3, keepdims=True) / 127  # per row
    assert np.all(np.abs(ko.astype(np.float64) - xk) <= sk * (0.5 + 1e-5))
    assert np.all(np.abs(vo.astype(np.float64) - xv) <= sv * (0.5 + 1e-5))
    big = slots.copy()
    big[0] = 4 * 16
    assert orc.cache_write_q8(*_empty_q8(hkv, 4), k_new, v_new, big) == 1


def pin_q8_lossless_attention(orc):
    """Values already on the quantisation grid survive the int8 pool exactly, so
    attention over the pool equals the pinned attention over the same values
    held as bf16, bit for bit."""
    rng = np.random.default_rng(13)
    hkv, hq, bs, nb = 2, 6, 16, 12
    lens = np.array([1, 16, 37, 70], np.int32)
    tables = np.zeros((4, 5), np.int32)
    perm = rng.permutation(nb)
    cur = 0
    for b, L in enumerate(lens):
        n = -(-int(L) // bs)
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    slots = np.concatenate([tables[b, np.arange(L) // bs] * bs + np.arange(L) % bs for b, L in enumerate(lens)])
    n = slots.size
    ki = np.clip(np.rint(rng.standard_normal((n, hkv, 128)) * 30), -126, 126)
    vi = np.clip(np.rint(rng.standard_normal((n, hkv, 128)) * 30), -126, 126)
    # K: in every block and channel one written row reaches 127; V: every row reaches 127.
    for blk in np.unique(slots // bs):
        first = np.nonzero(slots // bs == blk)[0][0]
        ki[first] = np.where(rng.random((hkv, 128)) < 0.5, 127, -127)
    vi[:, :, 0] = np.where(rng.random((n, hkv)) < 0.5, 127, -127)
    kb, vb = _bf16(ki / 16), _bf16(vi / 16)
    pool = _empty_q8(hkv, nb)
    assert orc.cache_write_q8(*pool, kb, vb, slots.astype(np.int32)) == 0
    kc = np.zeros((hkv, nb, bs, 128), np.uint16)
    vc = np.zeros((hkv, nb, bs, 128), np.uint16)
    assert orc.cache_write(kc, vc, kb, vb, slots.astype(np.int32)) == 0
    q = _bf16(((rng.standard_normal((4, 1, hq, 128)).astype(np.float32).view(np.uint32)) & 0xFFFF0000).view(np.float32))
    got = orc.decode_q8(*pool, q, tables, lens, 1 / np.sqrt(128))
    ref = orc.attend(kc, vc, q, tables, lens, 1 / np.sqrt(128))
    assert np.array_equal(got, ref)


def pin_ragged_verify(orc):
    """Ragged verify reduces to the pinned uniform verify: with the same count
    for every sequence it is bit-identical to it, and in a mix each sequence's
    rows (and the written pool) equal a uniform verify of that sequence alone
    with its own count."""
    w = inputs.custom(batch=5, q_heads=6, kv_heads=2, context_lens=(9, 20, 33, 16, 47), num_blocks=20,
                      seed=31, num_queries=4)
    same = inputs.ragged(w, [4] * 5)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    got = orc.verify_ragged(kc, vc, same.q, same.k_new, same.v_new, same.slot_mapping, same.query_start,
                            w.block_tables, w.context_lens, w.scale)
    kr, vr = w.k_cache.copy(), w.v_cache.copy()
    ref = orc.verify(kr, vr, w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(got, ref.reshape(got.shape)) and kc.tobytes() == kr.tobytes()
    mix = inputs.ragged(w, [1, 4, 0, 2, 3])
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    got = orc.verify_ragged(kc, vc, mix.q, mix.k_new, mix.v_new, mix.slot_mapping, mix.query_start,
                            w.block_tables, w.context_lens, w.scale)
    for b, n in enumerate(mix.nq):
        if n == 0:
            continue
        a = int(mix.query_start[b])
        one = inputs.custom(batch=1, q_heads=6, kv_heads=2, context_lens=(int(w.context_lens[b]),),
                            num_blocks=20, seed=31, num_queries=int(n))
        ka, va = w.k_cache.copy(), w.v_cache.copy()
        refb = orc.verify(ka, va, mix.q[a:a + n][None], mix.k_new[a:a + n], mix.v_new[a:a + n],
                          mix.slot_mapping[a:a + n], w.block_tables[b:b + 1], w.context_lens[b:b + 1], w.scale)
        assert one.spec.num_queries == n
        assert np.array_equal(got[a:a + n], refb[0])
    # every sequence's written rows land in the pool (none is dropped)
    kr, vr = w.k_cache.copy(), w.v_cache.copy()
    orc.cache_write(kr, vr, mix.k_new, mix.v_new, mix.slot_mapping)
    assert kc.tobytes() == kr.tobytes() and vc.tobytes() == vr.tobytes()


def pin_prefill_sdpa(orc):
    """Prefill (attention of each sequence's last n_b positions over a cache that
    holds them) against torch's float64 scaled_dot_product_attention with the
    causal mask offset by the prefix, over the gathered, repeat_kv-expanded
    context; and n_b = 1 everywhere reduces to decode, bit for bit."""
    import torch
    import torch.nn.functional as F

    lens = (1, 37, 80, 129, 16)
    w = inputs.custom(batch=5, q_heads=12, kv_heads=2, context_lens=lens, num_blocks=40, seed=41, num_queries=33)
    rw = inputs.ragged(w, [1, 33, 17, 20, 16])
    got = orc.attend_ragged(w.k_cache, w.v_cache, rw.q, rw.query_start, w.block_tables, w.context_lens, w.scale)
    bs, group = w.k_cache.shape[2], 6
    for b, L in enumerate(lens):
        a, e = int(rw.query_start[b]), int(rw.query_start[b + 1])
        n = e - a
        K = torch.from_numpy(_gather(w.k_cache, w.block_tables[b], L, bs)).repeat_interleave(group, 0)
        V = torch.from_numpy(_gather(w.v_cache, w.block_tables[b], L, bs)).repeat_interleave(group, 0)
        Q = torch.from_numpy(oracle.to_f64(rw.q[a:e])).transpose(0, 1)  # [Hq, n, D]
        mask = torch.arange(L)[None, :] <= torch.arange(L - n, L)[:, None]
        ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=w.scale).transpose(0, 1).numpy()
        err = np.max(np.abs(got[a:e] - ref))
        assert err <= 1e-12, f"prefill sdpa mismatch {err}, seq {b}"
    one = inputs.ragged(w, [1] * 5)
    got1 = orc.attend_ragged(w.k_cache, w.v_cache, one.q, one.query_start, w.block_tables, w.context_lens, w.scale)
    dec = orc.decode(w.k_cache, w.v_cache, one.q, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(got1, dec)


ALL_PINS = [pin_bruteforce, pin_sdpa, pin_onehot_softmax, pin_constant_v, pin_single_token,
            pin_two_token_closed_form, pin_block_permutation, pin_gqa_repeat, pin_verify_rows,
            pin_zero_length, pin_cache_write, pin_q8_row_closed_form, pin_q8_requant_closed_form,
            pin_q8_zero_and_partial_block, pin_q8_error_bound, pin_q8_lossless_attention,
            pin_ragged_verify, pin_prefill_sdpa]


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
