"""GPU parity of multi-head latent attention with decoupled RoPE
(APEX-1 Mathematical Reference -- Part 2, §9.3): rows [content (128) |
rope part (64)], only the rope part rotated, values of 128 entries.  Same
tolerance as the plain block: max |err| <= 2e-2, mean |err| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3
D_H, D_R = 128, 64


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _close(got, ref, what=""):
    e = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(e).all(), what
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, "%s max %.4g mean %.4g" % (what, e.max(), e.mean())


CASES = [  # B, H_q, H_kv, S_q, S_k, window, q_pos0, prefix
    (1, 8, 2, 300, 300, 0, 0, 0),        # G=4, ragged last block
    (2, 16, 1, 200, 200, 64, 0, 0),      # G=16, window
    (1, 4, 4, 260, 260, 0, 0, 0),        # G=1
    (1, 8, 8, 129, 400, 100, 271, 0),    # queries at an offset
    (1, 8, 2, 500, 500, 64, 0, 300),     # prefix longer than the window
    (2, 32, 8, 1000, 1000, 256, 0, 0),   # several items per pair
]


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,window,q_pos0,prefix", CASES)
def test_mla_prefill_matches_oracle(B, H_q, H_kv, S_q, S_k, window, q_pos0, prefix):
    dev = _dev()
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S_q, S_k, D_H, 1500 + S_q + window, d_r=D_R)
    out = apex.mla_fwd(q.to(dev), k.to(dev), v.to(dev), D_R, window=window, q_pos0=q_pos0, prefix_len=prefix)
    torch.cuda.synchronize()
    assert out.shape == (B, H_q, S_q, D_H)
    ref = oracle.mla_attn(q, k, v, D_R, window=window, q_pos0=q_pos0, prefix_len=prefix)
    _close(out, ref, "mla prefill")
    assert apex.apex_attn_device_status() == 0


def test_mla_yarn():
    dev = _dev()
    q, k, v = inputs.make_qkv(1, 8, 2, 400, 400, D_H, 1600, d_r=D_R)
    out = apex.mla_fwd(q.to(dev), k.to(dev), v.to(dev), D_R, yarn_scale=16.0, yarn_beta_fast=8.0,
                       yarn_beta_slow=2.0)
    torch.cuda.synchronize()
    ref = oracle.mla_attn(q, k, v, D_R, yarn_s=16.0, yarn_beta_fast=8.0, yarn_beta_slow=2.0)
    _close(out, ref, "mla yarn")


def test_mla_prerotated_keys():
    """The rope part of k rotated beforehand (by the fp64 oracle, rounded to bf16)."""
    dev = _dev()
    S = 333
    q, k, v = inputs.make_qkv(2, 8, 2, S, S, D_H, 1700, d_r=D_R)
    kd = k.double().numpy()
    pos = np.broadcast_to(np.arange(S)[None, None, :], (2, 2, S)).reshape(-1)
    kd[..., D_H:] = oracle.rope(kd[..., D_H:].reshape(-1, D_R), pos).reshape(2, 2, S, D_R)
    k_rot = torch.from_numpy(kd).to(torch.bfloat16)
    out = apex.mla_fwd(q.to(dev), k_rot.to(dev), v.to(dev), D_R, window=100, keys_prerotated=True)
    torch.cuda.synchronize()
    ref = oracle.mla_attn(q, k_rot, v, D_R, window=100, keys_prerotated=True)
    _close(out, ref, "mla prerotated")


def test_mla_rope_part_zero_matches_oracle():
    """Zero rope parts: only the content dot products remain (scaled by 1/sqrt(192))."""
    dev = _dev()
    q, k, v = inputs.make_qkv(1, 8, 2, 256, 256, D_H, 1800, d_r=D_R)
    q[..., D_H:] = 0
    k[..., D_H:] = 0
    out = apex.mla_fwd(q.to(dev), k.to(dev), v.to(dev), D_R, window=77)
    torch.cuda.synchronize()
    _close(out, oracle.mla_attn(q, k, v, D_R, window=77), "mla content only")


def _item_rows(w, n_rand=48):
    """One seeded row in each of the four M tiles of every work item of the
    CTA-pair prefill (an item is 4 * 128 / G consecutive query rows of one
    (batch, KV head) unit), plus the first and last 64 rows and random rows."""
    P = 128 // w.G
    rng = np.random.default_rng(20_000 + w.seed)
    S = w.S_q
    rows = set(range(64)) | set(range(S - 64, S)) | set(int(x) for x in rng.integers(0, S, n_rand))
    for r0 in range(0, S, 4 * P):
        for T in range(4):
            lo = r0 + T * P
            if lo < S:
                rows.add(int(rng.integers(lo, min(lo + P, S))))
    return sorted(rows)


def test_mla_full_workload_every_item():
    """The global-layer MLA workload at full size, in the bench's launch
    configuration, checked on every head of a row set that touches every work
    item and both tiles of each CTA of the pair kernel."""
    dev = _dev()
    w = inputs.WORKLOADS["mla"]
    q, k, v = inputs.workload_inputs(w)
    out = apex.mla_fwd(q.to(dev), k.to(dev), v.to(dev), w.d_r, window=w.window)
    torch.cuda.synchronize()
    rows = _item_rows(w)
    assert len(rows) >= w.S_q // (128 // w.G)
    got = out[:, :, rows].cpu()
    ref = oracle.mla_attn(q, k, v, w.d_r, window=w.window, rows=rows)
    _close(got, ref, "mla full")


def test_mla_rejects_unsupported():
    dev = _dev()
    q, k, v = [t.to(dev) for t in inputs.make_qkv(1, 4, 2, 64, 64, 64, 1900, d_r=64)]
    with pytest.raises(apex.ApexError):
        apex.mla_fwd(q, k, v, 64)   # d_h = 64: unsupported
    q, k, v = [t.to(dev) for t in inputs.make_qkv(1, 4, 2, 64, 64, D_H, 1901, d_r=D_R)]
    with pytest.raises(apex.ApexError):
        apex.mla_fwd(q, k, v, D_R, prefix_len=65)


DECODE_CASES = [  # B, H_q, H_kv, S_k, window, q_pos, prefix
    (2, 8, 2, 1000, 0, 999, 0),
    (3, 16, 4, 777, 100, 700, 0),
    (2, 32, 2, 600, 0, 599, 0),        # G=16: two query tiles per warp
    (2, 8, 8, 650, 64, 649, 0),        # G=1
    (2, 8, 2, 600, 0, 150, 400),       # query inside the prefix
    (1, 32, 8, 4096, 1024, 4095, 0),
]


@pytest.mark.parametrize("B,H_q,H_kv,S_k,window,q_pos,prefix", DECODE_CASES)
def test_mla_decode_matches_oracle(B, H_q, H_kv, S_k, window, q_pos, prefix):
    dev = _dev()
    q, k, v = inputs.make_qkv(B, H_q, H_kv, 1, S_k, D_H, 2000 + S_k + q_pos, d_r=D_R)
    out = apex.mla_decode(q.to(dev), k.to(dev), v.to(dev), q_pos, D_R, window=window, prefix_len=prefix)
    torch.cuda.synchronize()
    assert out.shape == (B, H_q, 1, D_H)
    ref = oracle.mla_attn(q, k, v, D_R, window=window, q_pos0=q_pos, prefix_len=prefix)
    _close(out, ref, "mla decode")
    assert apex.apex_attn_device_status() == 0


def test_mla_decode_yarn_and_prerotated():
    dev = _dev()
    S_k = 900
    q, k, v = inputs.make_qkv(2, 16, 4, 1, S_k, D_H, 2100, d_r=D_R)
    out = apex.mla_decode(q.to(dev), k.to(dev), v.to(dev), S_k - 1, D_R, yarn_scale=16.0, yarn_beta_fast=8.0,
                          yarn_beta_slow=2.0)
    torch.cuda.synchronize()
    _close(out, oracle.mla_attn(q, k, v, D_R, q_pos0=S_k - 1, yarn_s=16.0, yarn_beta_fast=8.0, yarn_beta_slow=2.0),
           "mla decode yarn")
    kd = k.double().numpy()
    pos = np.broadcast_to(np.arange(S_k)[None, None, :], (2, 4, S_k)).reshape(-1)
    kd[..., D_H:] = oracle.rope(kd[..., D_H:].reshape(-1, D_R), pos).reshape(2, 4, S_k, D_R)
    k_rot = torch.from_numpy(kd).to(torch.bfloat16)
    out2 = apex.mla_decode(q.to(dev), k_rot.to(dev), v.to(dev), S_k - 1, D_R, window=200, keys_prerotated=True)
    torch.cuda.synchronize()
    _close(out2, oracle.mla_attn(q, k_rot, v, D_R, q_pos0=S_k - 1, window=200, keys_prerotated=True),
           "mla decode prerotated")


def test_mla_decode_equals_last_prefill_row():
    dev = _dev()
    S = 700
    q, k, v = [t.to(dev) for t in inputs.make_qkv(2, 16, 4, S, S, D_H, 2200, d_r=D_R)]
    pre = apex.mla_fwd(q, k, v, D_R, window=300)
    dec = apex.mla_decode(q[:, :, S - 1:S].contiguous(), k, v, S - 1, D_R, window=300)
    torch.cuda.synchronize()
    d = (pre[:, :, S - 1:S].float() - dec.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3


def test_mla_decode_full_size_sampled_sequences():
    """The decode workload's cache shape (B64 H_q32 H_kv8 S_k 32768) with
    decoupled-RoPE rows; the oracle checks two of the 64 sequences."""
    dev = _dev()
    w = inputs.WORKLOADS["decode"]
    q, k, v = inputs.make_qkv(w.B, w.H_q, w.H_kv, 1, w.S_k, D_H, 2300, d_r=D_R)
    out = apex.mla_decode(q.to(dev), k.to(dev), v.to(dev), w.q_pos0, D_R)
    torch.cuda.synchronize()
    pick = [0, 37]
    ref = oracle.mla_attn(q[pick], k[pick], v[pick], D_R, q_pos0=w.q_pos0)
    _close(out[pick].cpu(), ref, "mla decode full")
