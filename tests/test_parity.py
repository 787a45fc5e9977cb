"""GPU parity: the CUDA library against the fp64 oracle on the same seeded bf16
inputs.  Tolerance for every floating-point comparison: max |err| <= 2e-2 and
mean |err| <= 2e-3 on the bf16 outputs widened to fp64."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _errs(got, ref):
    e = np.abs(got.double().cpu().numpy() - ref)
    return float(e.max()), float(e.mean())


def _assert_close(got, ref, what=""):
    mx, mean = _errs(got, ref)
    assert np.isfinite(mx), what
    assert mx <= MAX_ERR and mean <= MEAN_ERR, "%s max %.4g mean %.4g" % (what, mx, mean)


def _status_ok():
    assert apex.apex_attn_device_status() == 0


# ------------------------------------------------------------------ prefill
PREFILL_CASES = [
    # B, H_q, H_kv, S_q, S_k, d, window, q_pos0
    (1, 4, 2, 128, 128, 64, 0, 0),        # the tiny workload shape
    (1, 2, 2, 200, 200, 128, 0, 0),       # G = 1, ragged tail
    (2, 8, 2, 300, 300, 128, 0, 0),       # G = 4, several key tiles
    (1, 8, 1, 333, 333, 64, 100, 0),      # G = 8, window, d 64
    (1, 16, 1, 261, 261, 128, 64, 0),     # G = 16, window smaller than a tile
    (2, 4, 2, 77, 333, 128, 0, 256),      # queries at the end of a longer key range
    (1, 4, 4, 130, 500, 64, 37, 300),     # offset queries with a window
    (1, 32, 8, 1024, 1024, 128, 256, 0),  # GQA workload shape, scaled down
]


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,d,window,q_pos0", PREFILL_CASES)
def test_prefill_matches_oracle(B, H_q, H_kv, S_q, S_k, d, window, q_pos0):
    dev = _dev()
    q = inputs.normal_bf16((B, H_q, S_q, d), 100 + S_q, 0)
    k = inputs.normal_bf16((B, H_kv, S_k, d), 100 + S_q, 1)
    v = inputs.normal_bf16((B, H_kv, S_k, d), 100 + S_q, 2)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, q_pos0=q_pos0)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos0)
    _assert_close(out, ref, "prefill")
    _status_ok()


def test_prefill_tiny_workload():
    dev = _dev()
    w = inputs.WORKLOADS["tiny"]
    q, k, v = inputs.workload_inputs(w)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=w.window)
    torch.cuda.synchronize()
    _assert_close(out, oracle.attn(q, k, v, window=w.window), "tiny")


def test_prefill_window_one_is_value():
    """W = 1: out[r] = v[r] exactly (softmax over a single key)."""
    dev = _dev()
    q = inputs.normal_bf16((1, 4, 150, 128), 7, 0)
    k = inputs.normal_bf16((1, 2, 150, 128), 7, 1)
    v = inputs.normal_bf16((1, 2, 150, 128), 7, 2)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=1).cpu()
    assert torch.equal(out, v.repeat_interleave(2, dim=1))


def test_prefill_window_ge_seq_is_causal_bitwise():
    dev = _dev()
    q = inputs.normal_bf16((1, 8, 300, 128), 8, 0).to(dev)
    k = inputs.normal_bf16((1, 2, 300, 128), 8, 1).to(dev)
    v = inputs.normal_bf16((1, 2, 300, 128), 8, 2).to(dev)
    a = apex.fwd(q, k, v, window=0)
    b = apex.fwd(q, k, v, window=300)
    c = apex.fwd(q, k, v, window=100000)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_prefill_deterministic():
    dev = _dev()
    q = inputs.normal_bf16((2, 8, 400, 128), 9, 0).to(dev)
    k = inputs.normal_bf16((2, 2, 400, 128), 9, 1).to(dev)
    v = inputs.normal_bf16((2, 2, 400, 128), 9, 2).to(dev)
    a = apex.fwd(q, k, v, window=150)
    b = apex.fwd(q, k, v, window=150)
    assert torch.equal(a, b)


def test_prefill_gqa_equals_mha_on_repeated_kv():
    dev = _dev()
    G = 4
    q = inputs.normal_bf16((1, 8, 256, 128), 10, 0).to(dev)
    k = inputs.normal_bf16((1, 2, 256, 128), 10, 1).to(dev)
    v = inputs.normal_bf16((1, 2, 256, 128), 10, 2).to(dev)
    a = apex.fwd(q, k, v)
    b = apex.fwd(q, k.repeat_interleave(G, 1).contiguous(), v.repeat_interleave(G, 1).contiguous())
    mx, mean = _errs(a.cpu(), b.double().cpu().numpy())
    assert mx <= MAX_ERR and mean <= MEAN_ERR


# ------------------------------------------------------------------ decode
DECODE_CASES = [
    # B, H_q, H_kv, S_k, d, window, q_pos
    (1, 4, 2, 128, 64, 0, 127),
    (2, 8, 2, 1000, 128, 0, 999),      # ragged last stage
    (3, 16, 4, 777, 128, 100, 700),    # window, query before the end of the cache
    (1, 16, 1, 513, 128, 0, 512),      # G = 16 (two query n-tiles)
    (2, 8, 8, 300, 64, 0, 5),          # G = 1, very short visible range
    (1, 32, 8, 4096, 128, 1024, 4095),
]


@pytest.mark.parametrize("B,H_q,H_kv,S_k,d,window,q_pos", DECODE_CASES)
def test_decode_matches_oracle(B, H_q, H_kv, S_k, d, window, q_pos):
    dev = _dev()
    q = inputs.normal_bf16((B, H_q, 1, d), 200 + S_k, 0)
    k = inputs.normal_bf16((B, H_kv, S_k, d), 200 + S_k, 1)
    v = inputs.normal_bf16((B, H_kv, S_k, d), 200 + S_k, 2)
    out = apex.decode(q.to(dev), k.to(dev), v.to(dev), q_pos, window=window)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos)
    _assert_close(out, ref, "decode")
    _status_ok()


def test_decode_equals_last_prefill_row():
    dev = _dev()
    S = 640
    q = inputs.normal_bf16((2, 8, S, 128), 11, 0).to(dev)
    k = inputs.normal_bf16((2, 2, S, 128), 11, 1).to(dev)
    v = inputs.normal_bf16((2, 2, S, 128), 11, 2).to(dev)
    full = apex.fwd(q, k, v, window=200)
    dec = apex.decode(q[:, :, -1:].contiguous(), k, v, S - 1, window=200)
    mx, mean = _errs(dec.cpu(), full[:, :, -1:].double().cpu().numpy())
    assert mx <= MAX_ERR and mean <= MEAN_ERR


def test_decode_deterministic():
    dev = _dev()
    q = inputs.normal_bf16((4, 8, 1, 128), 12, 0).to(dev)
    k = inputs.normal_bf16((4, 2, 3000, 128), 12, 1).to(dev)
    v = inputs.normal_bf16((4, 2, 3000, 128), 12, 2).to(dev)
    a = apex.decode(q, k, v, 2999)
    b = apex.decode(q, k, v, 2999)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ full-size workloads
def _sample_rows(w, n_rand=48):
    S = w.S_q
    rng = np.random.default_rng(w.seed)
    rows = set(range(min(64, S))) | set(range(max(0, S - 64), S)) | set(int(x) for x in rng.integers(0, S, n_rand))
    if w.window > 0:
        for r in range(w.window - 8, w.window + 8):
            if 0 <= r < S:
                rows.add(r)
    return sorted(rows)


def _item_rows(w):
    """One seeded row in each of the four M tiles of every work item of the
    CTA-pair prefill kernel (an item is 4 * 128 / G consecutive query rows of
    one (batch, KV head) unit; tile T of it holds rows T * 128 / G onwards, the
    G heads of each row packed into one 128-row tile), so every item -- the
    first of a unit, the middle ones, the last and ragged one, those whose
    window starts in another key tile -- and both CTAs' tiles are checked in
    every (batch, KV head) unit; plus the rows of _sample_rows."""
    P = 128 // w.G
    rng = np.random.default_rng(10_000 + w.seed)
    rows = set(_sample_rows(w))
    for r0 in range(0, w.S_q, 4 * P):
        for T in range(4):
            lo = r0 + T * P
            if lo < w.S_q:
                rows.add(int(rng.integers(lo, min(lo + P, w.S_q))))
    return sorted(rows)


def test_prefill_gqa_full_workload_every_row():
    """The gqa workload in the bench's launch configuration (keys rotated once
    into a workspace first), and without a workspace (keys rotated in the
    kernel): every output element of every (batch, head, row) against the
    oracle."""
    dev = _dev()
    w = inputs.WORKLOADS["gqa"]
    q, k, v = inputs.workload_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = apex.fwd(qd, kd, vd, window=w.window, q_pos0=w.q_pos0)
    out2 = apex.fwd(qd, kd, vd, window=w.window, q_pos0=w.q_pos0, workspace=False)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=w.window, q_pos0=w.q_pos0)
    _assert_close(out, ref, "gqa")
    _assert_close(out2, ref, "gqa, keys rotated in the kernel")
    _status_ok()


@pytest.mark.parametrize("name", ["wide", "long"])
def test_prefill_full_workload_every_item(name):
    """Full-size workloads in the launch configuration the bench times; the oracle
    checks every head of a row set that touches every work item and both tiles of
    each CTA of the pair kernel, plus the first and last 64 rows, the window edge
    and random rows."""
    dev = _dev()
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_inputs(w)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=w.window, q_pos0=w.q_pos0)
    torch.cuda.synchronize()
    rows = _item_rows(w)
    assert len(rows) >= w.S_q // (128 // w.G)
    ref = oracle.attn(q, k, v, window=w.window, q_pos0=w.q_pos0, rows=rows)
    _assert_close(out[:, :, rows], ref, name)
    _status_ok()


def test_decode_full_workload():
    dev = _dev()
    w = inputs.WORKLOADS["decode"]
    q, k, v = inputs.workload_inputs(w)
    out = apex.decode(q.to(dev), k.to(dev), v.to(dev), w.q_pos0, window=w.window)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=w.window, q_pos0=w.q_pos0)
    _assert_close(out, ref, "decode")
    _status_ok()
