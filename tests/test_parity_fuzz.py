"""GPU parity on seeded random configurations: group sizes 1-16, head dims 64
and 128, ragged lengths, query offsets, windows, bidirectional prefixes and
YaRN, for the prefill (both kernels), the decode and the decoupled-RoPE paths,
each compared with the fp64 oracle.  The configurations are drawn once from a
fixed seed, so every run checks the same cases.  Tolerance as everywhere:
max |err| <= 2e-2, mean |err| <= 2e-3."""
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
    assert np.isfinite(e).all(), what
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, "%s: max %.4g mean %.4g" % (what, e.max(), e.mean())


def _draw_options(rng, S_k):
    window = 0 if rng.random() < 0.4 else int(rng.integers(1, S_k + 1))
    prefix = 0 if rng.random() < 0.7 else int(rng.integers(1, S_k + 1))
    yarn = 1.0 if rng.random() < 0.7 else float(rng.choice([4.0, 16.0, 32.0]))
    return window, prefix, yarn


def _prefill_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        H_kv = int(rng.choice([1, 2]))
        B = int(rng.integers(1, 3))
        S_q = int(rng.integers(1, 601))
        q_pos0 = 0 if rng.random() < 0.6 else int(rng.integers(0, 301))
        S_k = q_pos0 + S_q + (0 if rng.random() < 0.7 else int(rng.integers(1, 200)))
        window, prefix, yarn = _draw_options(rng, S_k)
        cases.append((B, G * H_kv, H_kv, S_q, S_k, d, q_pos0, window, prefix, yarn))
    return cases


def _decode_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        H_kv = int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 5))
        S_k = int(rng.integers(1, 3001))
        q_pos = S_k - 1 if rng.random() < 0.6 else int(rng.integers(0, S_k))
        window, prefix, yarn = _draw_options(rng, S_k)
        cases.append((B, G * H_kv, H_kv, S_k, d, q_pos, window, prefix, yarn))
    return cases


PREFILL = _prefill_cases(48, 20261202)
DECODE = _decode_cases(24, 20261203)
MLA_PREFILL = [c for c in _prefill_cases(24, 20261204) if c[5] == 128][:10]
MLA_DECODE = [c for c in _decode_cases(24, 20261205) if c[4] == 128][:10]


# every case through the single-CTA kernel, and the d_h = 128 ones (the rows the
# CTA-pair kernel serves) through the pair kernel as well
PREFILL_RUNS = [("single", c) for c in PREFILL] + [("pair", c) for c in PREFILL if c[5] == 128]


@pytest.mark.parametrize("kernel,case", PREFILL_RUNS,
                         ids=lambda x: x if isinstance(x, str) else "B%d_Hq%d_Hkv%d_Sq%d_Sk%d_d%d_p%d_W%d_P%d_y%g" % x)
def test_prefill_fuzz(kernel, case, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("APEX_ATTN_PREFILL", kernel)
    B, H_q, H_kv, S_q, S_k, d, q_pos0, window, prefix, yarn = case
    dev = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S_q, S_k, d, 5000 + S_q + 7 * S_k)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, q_pos0=q_pos0, prefix_len=prefix,
                   yarn_scale=yarn)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, prefix_len=prefix, yarn_s=yarn)
    _close(out, ref, "prefill %s %s" % (kernel, case))
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "B%d_Hq%d_Hkv%d_Sk%d_d%d_q%d_W%d_P%d_y%g" % c)
def test_decode_fuzz(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H_q, H_kv, S_k, d, q_pos, window, prefix, yarn = case
    dev = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, 1, S_k, d, 6000 + S_k + 3 * q_pos)
    out = apex.decode(q.to(dev), k.to(dev), v.to(dev), q_pos, window=window, prefix_len=prefix, yarn_scale=yarn)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos, prefix_len=prefix, yarn_s=yarn)
    _close(out, ref, "decode %s" % (case,))
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("case", MLA_PREFILL, ids=lambda c: "B%d_Hq%d_Hkv%d_Sq%d_Sk%d_d%d_p%d_W%d_P%d_y%g" % c)
def test_mla_prefill_fuzz(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H_q, H_kv, S_q, S_k, d, q_pos0, window, prefix, yarn = case
    dev = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S_q, S_k, d, 7000 + S_q + 5 * S_k, d_r=64)
    out = apex.mla_fwd(q.to(dev), k.to(dev), v.to(dev), 64, window=window, q_pos0=q_pos0, prefix_len=prefix,
                       yarn_scale=yarn)
    torch.cuda.synchronize()
    ref = oracle.mla_attn(q, k, v, 64, window=window, q_pos0=q_pos0, prefix_len=prefix, yarn_s=yarn)
    _close(out, ref, "mla prefill %s" % (case,))
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("case", MLA_DECODE, ids=lambda c: "B%d_Hq%d_Hkv%d_Sk%d_d%d_q%d_W%d_P%d_y%g" % c)
def test_mla_decode_fuzz(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H_q, H_kv, S_k, d, q_pos, window, prefix, yarn = case
    dev = torch.device("cuda:0")
    q, k, v = inputs.make_qkv(B, H_q, H_kv, 1, S_k, d, 8000 + S_k + 3 * q_pos, d_r=64)
    out = apex.mla_decode(q.to(dev), k.to(dev), v.to(dev), q_pos, 64, window=window, prefix_len=prefix,
                          yarn_scale=yarn)
    torch.cuda.synchronize()
    ref = oracle.mla_attn(q, k, v, 64, window=window, q_pos0=q_pos, prefix_len=prefix, yarn_s=yarn)
    _close(out, ref, "mla decode %s" % (case,))
    assert apex.apex_attn_device_status() == 0
