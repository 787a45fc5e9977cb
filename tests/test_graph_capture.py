"""GPU: the prefill (CTA-pair and single-CTA kernels) and decode calls captured in
one CUDA graph and replayed on new inputs copied into the same buffers, checked
against the fp64 oracle each time.  The RoPE tables are reserved and each call
made once before capture, so the captured calls allocate and synchronise
nothing."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3


def _close(got, ref, what):
    e = np.abs(got.double().cpu().numpy() - ref)
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, "%s: max %.4g mean %.4g" % (what, e.max(), e.mean())


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_prefill_and_decode_in_a_graph(kernel, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("APEX_ATTN_PREFILL", kernel)
    dev = torch.device("cuda:0")
    B, H_q, H_kv, S, d, W = 2, 8, 2, 300, 128, 100
    Bd, S_k = 3, 500
    pq, pk, pv = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 9100))
    dq, dk, dv = (t.to(dev) for t in inputs.make_qkv(Bd, H_q, H_kv, 1, S_k, d, 9101))
    pout = torch.empty_like(pq)
    dout = torch.empty_like(dq)
    ws = torch.empty(apex.decode_workspace_bytes(Bd, H_q, H_kv, S_k, d), dtype=torch.uint8, device=dev)
    apex.apex_attn_rope_reserve(S_k, d, 10000.0)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        apex.fwd(pq, pk, pv, window=W, out=pout)
        apex.decode(dq, dk, dv, S_k - 1, window=W, out=dout, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        apex.fwd(pq, pk, pv, window=W, out=pout)
        apex.decode(dq, dk, dv, S_k - 1, window=W, out=dout, workspace=ws)

    for seed in (9200, 9300):
        q, k, v = inputs.make_qkv(B, H_q, H_kv, S, S, d, seed)
        qd, kd, vd = inputs.make_qkv(Bd, H_q, H_kv, 1, S_k, d, seed + 1)
        for dst, src in zip((pq, pk, pv, dq, dk, dv), (q, k, v, qd, kd, vd)):
            dst.copy_(src)
        pout.zero_()
        dout.zero_()
        g.replay()
        torch.cuda.synchronize()
        _close(pout, oracle.attn(q, k, v, window=W), "graph prefill %s" % kernel)
        _close(dout, oracle.attn(qd, kd, vd, window=W, q_pos0=S_k - 1), "graph decode")
    assert apex.apex_attn_device_status() == 0
