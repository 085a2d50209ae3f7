"""The seeded input generators (CPU only): determinism and structure."""

import numpy as np
import pytest

from paged_kv_decode_pa_gb300 import inputs


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 3.140625], dtype=np.float32)
    bits = inputs.f32_to_bf16_bits(x)
    back = inputs.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to the even mantissa (1.0)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -7, -2.5, 3.140625]


def test_same_seed_same_workload():
    a = inputs.make("c1")
    b = inputs.make("c1")
    for f in ("k_cache", "v_cache", "q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"):
        assert np.array_equal(getattr(a, f), getattr(b, f), equal_nan=True)


@pytest.mark.parametrize("name", ["c1", "c2", "c5"])
def test_structure(name):
    w = inputs.make(name)
    s = w.spec
    bs = s.block_size
    lens = w.context_lens
    # every real sequence owns distinct blocks
    used = np.concatenate([w.block_tables[b, : (lens[b] + bs - 1) // bs] for b in range(w.real_rows)])
    assert len(np.unique(used)) == used.size
    if w.spare_block is not None:
        assert w.spare_block not in used
    # slots point at the positions of the new tokens
    nq = s.num_queries
    for b in range(s.batch):
        for i in range(nq):
            pos = lens[b] - nq + i
            slot = w.slot_mapping[b * nq + i]
            assert slot == w.block_tables[b, pos // bs] * bs + pos % bs
    # rows beyond each context in its last block are NaN, rows inside are finite
    kf = inputs.bf16_bits_to_f32(w.k_cache) if s.dtype == "bf16" else w.k_cache
    for b in range(w.real_rows):
        L = lens[b]
        last = w.block_tables[b, (L - 1) // bs]
        r = L % bs
        assert np.all(np.isfinite(kf[:, last, : (r or bs)]))
        if r:
            assert np.all(np.isnan(kf[:, last, r:]))


def test_padded_rows_only_touch_the_spare_block():
    w = inputs.make("c3", padded_rows=7)
    assert w.real_rows == 57
    assert np.all(w.block_tables[57:] == w.spare_block)
    assert np.all((w.context_lens[57:] >= 1) & (w.context_lens[57:] <= 16))
    assert np.all(w.slot_mapping[57:] // 16 == w.spare_block)


def test_q8_pool_structure():
    """The int8 pool generator: held rows get drawn bytes in [1, 255] and finite
    V scales; other rows hold byte 128 with NaN V scales; K scales are finite."""
    w = inputs.make("c3")
    p = inputs.q8_pool(w)
    hkv, nb, bs, d = p.k_codes.shape
    assert p.k_scale.shape == (hkv, nb, d) and p.v_scale.shape == (hkv, nb, bs)
    held = np.zeros((nb, bs), bool)
    for b in range(w.real_rows):
        t = np.arange(int(w.context_lens[b]))
        held[w.block_tables[b, t // bs], t % bs] = True
    held[w.spare_block] = True
    assert np.all(p.k_codes[:, ~held] == 128) and np.all(p.v_codes[:, ~held] == 128)
    assert p.k_codes[:, held].min() >= 1 and np.isfinite(p.v_scale[:, held]).all()
    assert np.isnan(p.v_scale[:, ~held]).all() and np.isfinite(p.k_scale).all()
    again = inputs.q8_pool(w)
    assert np.array_equal(again.k_codes, p.k_codes) and np.array_equal(again.v_scale, p.v_scale, equal_nan=True)
