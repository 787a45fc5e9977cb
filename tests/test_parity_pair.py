"""GPU parity of both prefill kernels for d_h = 128 on the plain block: the
CTA-pair kernel (tcgen05 cta_group::2, the default) and the single-CTA kernel
(APEX_ATTN_PREFILL=single, read at each call), same tolerance as everywhere
(max |err| <= 2e-2, mean |err| <= 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3


@pytest.fixture
def pair_kernel(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("APEX_ATTN_PREFILL", "pair")
    yield torch.device("cuda:0")


@pytest.fixture(params=["pair", "single"])
def either_kernel(request, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("APEX_ATTN_PREFILL", request.param)
    yield torch.device("cuda:0")


def _qkv(B, H_q, H_kv, S_q, S_k, d, seed):
    return (inputs.normal_bf16((B, H_q, S_q, d), seed, 0), inputs.normal_bf16((B, H_kv, S_k, d), seed, 1),
            inputs.normal_bf16((B, H_kv, S_k, d), seed, 2))


CASES = [  # B, H_q, H_kv, S_q, S_k, window, q_pos0, prefix
    (1, 8, 2, 300, 300, 0, 0, 0),         # ragged last block, G=4
    (2, 16, 1, 200, 200, 64, 0, 0),       # G=16 (8 positions per tile), window
    (1, 4, 4, 520, 520, 0, 0, 0),         # G=1
    (1, 8, 8, 129, 400, 100, 271, 0),     # queries at an offset, window, G=1
    (1, 8, 2, 500, 500, 64, 0, 300),      # prefix longer than the window
    (3, 16, 2, 1000, 1000, 0, 0, 0),      # several items per pair
]


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,window,q_pos0,prefix", CASES)
def test_prefill_kernels_match_oracle(either_kernel, B, H_q, H_kv, S_q, S_k, window, q_pos0, prefix):
    dev = either_kernel
    q, k, v = _qkv(B, H_q, H_kv, S_q, S_k, 128, 1200 + S_q + window)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, q_pos0=q_pos0, prefix_len=prefix)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, prefix_len=prefix)
    e = np.abs(out.double().cpu().numpy() - ref)
    assert np.isfinite(e).all()
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, (e.max(), e.mean())
    assert apex.apex_attn_device_status() == 0


def test_pair_deterministic_and_close_to_single(pair_kernel, monkeypatch):
    """Two calls give the same bits; the single-CTA kernel (whose key-rotation
    recurrence starts from other rows, so its rotated keys may round
    differently) agrees within the parity tolerance."""
    q, k, v = [t.to(pair_kernel) for t in _qkv(2, 32, 8, 777, 777, 128, 1300)]
    a = apex.fwd(q, k, v, window=256)
    a2 = apex.fwd(q, k, v, window=256)
    monkeypatch.setenv("APEX_ATTN_PREFILL", "single")
    b = apex.fwd(q, k, v, window=256)
    torch.cuda.synchronize()
    assert torch.equal(a, a2)
    d = (a.float() - b.float()).abs()
    assert d.max().item() <= MAX_ERR and d.mean().item() <= MEAN_ERR


def test_pair_yarn_and_prerotated(pair_kernel):
    q, k, v = _qkv(1, 8, 2, 400, 400, 128, 1400)
    out = apex.fwd(q.to(pair_kernel), k.to(pair_kernel), v.to(pair_kernel), yarn_scale=16.0, yarn_beta_fast=8.0,
                   yarn_beta_slow=2.0)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, yarn_s=16.0, yarn_beta_fast=8.0, yarn_beta_slow=2.0)
    e = np.abs(out.double().cpu().numpy() - ref)
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR
    k_rot = apex.rope_keys(k.to(pair_kernel))
    out2 = apex.fwd(q.to(pair_kernel), k_rot, v.to(pair_kernel), keys_prerotated=True)
    torch.cuda.synchronize()
    ref2 = oracle.attn(q, k_rot.cpu(), v, keys_prerotated=True)
    e = np.abs(out2.double().cpu().numpy() - ref2)
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR
