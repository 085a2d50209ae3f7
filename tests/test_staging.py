"""StepStaging layout (CPU) and its single-copy upload feeding pa_verify (GPU)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_decode_pa_gb300 import inputs
from paged_kv_decode_pa_gb300.staging import StepStaging


def _fields(w):
    import paged_kv_decode_pa_gb300 as pa

    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    return {n: pa.to_torch(getattr(w, n), "cpu") for n in names}


def test_layout_aligned_and_disjoint():
    w = inputs.make("c2")
    tens = _fields(w)
    st = StepStaging({n: (tuple(t.shape), t.dtype) for n, t in tens.items()}, device="cpu", pin=False)
    spans = sorted(st.offsets.values())
    for (o, n), (o2, _) in zip(spans, spans[1:]):
        assert o % 256 == 0 and o + n <= o2
    assert st.upload_bytes == sum(t.numel() * t.element_size() for t in tens.values())
    for n, t in tens.items():
        st.host[n].copy_(t)
        assert st.host[n].shape == t.shape and st.host[n].dtype == t.dtype
        assert st.host[n].data_ptr() % 256 == st.host_buf.data_ptr() % 256
    for n, t in tens.items():  # no field overwrote another
        assert torch.equal(st.host[n].view(torch.uint8) if t.dtype == torch.bfloat16 else st.host[n],
                           t.view(torch.uint8) if t.dtype == torch.bfloat16 else t)


@pytest.mark.gpu
def test_staged_verify_matches_oracle():
    import paged_kv_decode_pa_gb300 as pa
    from gpu_util import assert_close, oracle_verify_of, to_f64

    w = inputs.make("c5", batch=8, num_blocks=1024)
    ref, rk, rv = oracle_verify_of(w)
    dev = torch.device("cuda")
    tens = _fields(w)
    st = StepStaging({n: (tuple(t.shape), t.dtype) for n, t in tens.items()}, dev)
    for n, t in tens.items():
        st.host[n].copy_(t)
    st.upload()
    d = st.dev
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    batch, nq, hq, _ = w.q.shape
    ws = pa.new_workspace(batch, nq, hq, w.spec.kv_heads, w.max_context_len, dev)
    out = pa.pa_verify(kc, vc, d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["block_tables"],
                       d["context_lens"], w.max_context_len, w.scale, ws)
    torch.cuda.synchronize()
    for n, t in tens.items():
        assert torch.equal(d[n].cpu().view(torch.uint8), t.view(torch.uint8)), n
    assert pa.pa_workspace_status(ws) == 0
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", "staged verify")
    assert np.array_equal(pa.to_numpy(kc), rk) and np.array_equal(pa.to_numpy(vc), rv)
