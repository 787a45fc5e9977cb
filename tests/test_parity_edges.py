"""GPU parity on edge shapes not covered elsewhere: every group size on both
prefill kernels at d_h = 128, single query rows, single keys, tiny ragged
sizes, window 1, whole-sequence prefixes, many small units, decoupled RoPE at
G = 16 and one row, decode on one-key and ragged caches, and 131072-token
prefill and decode.  Tolerance as
everywhere: max |err| <= 2e-2, mean |err| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3


@pytest.fixture(params=["pair", "single"])
def dev(request, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("APEX_ATTN_PREFILL", request.param)
    return torch.device("cuda:0")


def _close(got, ref, what=""):
    e = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(e).all(), what
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, "%s max %.4g mean %.4g" % (what, e.max(), e.mean())


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,window,q_pos0,prefix", [
    (1, 4, 2, 300, 300, 0, 0, 0),       # G = 2
    (1, 16, 2, 300, 300, 50, 0, 0),     # G = 8
    (1, 16, 1, 40, 40, 0, 0, 0),        # G = 16, less than one tile
    (2, 8, 2, 1, 700, 0, 699, 0),       # one query row at the end of the keys
    (1, 8, 2, 1, 1, 0, 0, 0),           # one query, one key
    (1, 4, 4, 3, 3, 0, 0, 0),           # three rows
    (1, 8, 2, 257, 257, 1, 0, 0),       # window 1
    (1, 8, 2, 300, 300, 0, 0, 300),     # the whole sequence is a bidirectional prefix
    (64, 8, 8, 16, 16, 0, 0, 0),        # many small units
    (1, 8, 2, 513, 1024, 200, 511, 100),  # offset queries, window, prefix before them
])
def test_prefill_edges(dev, B, H_q, H_kv, S_q, S_k, window, q_pos0, prefix):
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S_q, S_k, 128, 4000 + S_q + S_k)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, q_pos0=q_pos0, prefix_len=prefix)
    torch.cuda.synchronize()
    _close(out, oracle.attn(q, k, v, window=window, q_pos0=q_pos0, prefix_len=prefix), "prefill edge")
    assert apex.apex_attn_device_status() == 0


def test_window_one_returns_own_value_row(dev):
    """W = 1 leaves each query its own key: out[r] = v[q_pos0 + r] (bf16, exact)."""
    q, k, v = inputs.make_qkv(1, 8, 2, 200, 200, 128, 4100)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=1)
    torch.cuda.synchronize()
    ref = torch.repeat_interleave(v, 4, dim=1)
    assert torch.equal(out.cpu(), ref)


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,window,q_pos0", [
    (1, 32, 2, 300, 300, 77, 0),    # G = 16
    (2, 8, 2, 1, 500, 0, 499),      # one row
    (1, 16, 2, 300, 300, 1, 0),     # window 1
])
def test_mla_edges(B, H_q, H_kv, S_q, S_k, window, q_pos0):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S_q, S_k, 128, 4200 + S_q, d_r=64)
    out = apex.mla_fwd(q.to(d), k.to(d), v.to(d), 64, window=window, q_pos0=q_pos0)
    torch.cuda.synchronize()
    _close(out, oracle.mla_attn(q, k, v, 64, window=window, q_pos0=q_pos0), "mla edge")


@pytest.mark.parametrize("B,H_q,H_kv,S_k,window,q_pos", [
    (2, 8, 2, 1, 0, 0),        # one cached key
    (3, 16, 4, 65, 0, 64),     # one key past a stage
    (2, 8, 2, 300, 1, 299),    # window 1
    (2, 32, 2, 129, 0, 128),   # G = 16
    (4, 8, 8, 1000, 0, 10),    # early query in a long cache
])
def test_decode_edges(B, H_q, H_kv, S_k, window, q_pos):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, 1, S_k, 128, 4300 + S_k + q_pos)
    out = apex.decode(q.to(d), k.to(d), v.to(d), q_pos, window=window)
    torch.cuda.synchronize()
    _close(out, oracle.attn(q, k, v, window=window, q_pos0=q_pos), "decode edge")
    assert apex.apex_attn_device_status() == 0


def test_prefill_131072_keys_sampled_rows():
    """A 131072-token sequence (twice the long workload), window 8192 and causal:
    sampled rows of every head against the oracle (indices and offsets past
    2^16 positions, a 128K-row RoPE table)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    S = 131072
    q, k, v = inputs.make_qkv(1, 8, 2, S, S, 128, 4400)
    rows = sorted(set(range(0, 32)) | set(range(S - 32, S)) | set(range(8192 - 8, 8192 + 8)) |
                  set(int(x) for x in np.random.default_rng(4400).integers(0, S, 24)))
    for window in (8192, 0):
        out = apex.fwd(q.to(d), k.to(d), v.to(d), window=window)
        torch.cuda.synchronize()
        _close(out[:, :, rows], oracle.attn(q, k, v, window=window, rows=rows), "prefill 128K W%d" % window)
    assert apex.apex_attn_device_status() == 0


def test_decode_131072_keys():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    S_k = 131072
    q, k, v = inputs.make_qkv(2, 8, 2, 1, S_k, 128, 4500)
    for window, q_pos in ((0, S_k - 1), (8192, S_k - 1), (0, 70000)):
        out = apex.decode(q.to(d), k.to(d), v.to(d), q_pos, window=window)
        torch.cuda.synchronize()
        _close(out, oracle.attn(q, k, v, window=window, q_pos0=q_pos), "decode 128K W%d q%d" % (window, q_pos))
    assert apex.apex_attn_device_status() == 0
