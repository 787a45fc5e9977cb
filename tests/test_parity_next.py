"""GPU parity for the options beyond the plain block: YaRN-scaled RoPE with the
attention temperature (Part 1, §5), the bidirectional prefix (Part 2, §11.1) and
keys given pre-rotated, plus the key-rotation helper.  Same tolerance as the
plain block: max |err| <= 2e-2, mean |err| <= 2e-3."""
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


def _close(got, ref, what=""):
    e = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(e).all(), what
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, "%s max %.4g mean %.4g" % (what, e.max(), e.mean())


def _qkv(B, H_q, H_kv, S_q, S_k, d, seed):
    return (inputs.normal_bf16((B, H_q, S_q, d), seed, 0), inputs.normal_bf16((B, H_kv, S_k, d), seed, 1),
            inputs.normal_bf16((B, H_kv, S_k, d), seed, 2))


def _prerotate(k, base=10000.0):
    """Keys rotated to their positions by the fp64 oracle, rounded to bf16 on the CPU."""
    B, H, S, d = k.shape
    pos = np.broadcast_to(np.arange(S)[None, None, :], (B, H, S)).reshape(-1)
    rot = oracle.rope(k.double().numpy().reshape(-1, d), pos, base).reshape(B, H, S, d)
    return torch.from_numpy(rot).to(torch.bfloat16)


YARN = [  # s, beta_fast, beta_slow
    (32.0, 32.0, 1.0),     # the pages' defaults (no interpolation band)
    (16.0, 8.0, 2.0),      # a band of interpolated frequencies
]


@pytest.mark.parametrize("s,bf,bs", YARN)
@pytest.mark.parametrize("B,H_q,H_kv,S,d,window", [(1, 8, 2, 300, 128, 0), (2, 16, 4, 400, 128, 100),
                                                   (1, 4, 4, 260, 64, 0)])
def test_prefill_yarn(s, bf, bs, B, H_q, H_kv, S, d, window):
    dev = _dev()
    q, k, v = _qkv(B, H_q, H_kv, S, S, d, 500 + S)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, yarn_scale=s, yarn_beta_fast=bf,
                   yarn_beta_slow=bs)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, yarn_s=s, yarn_beta_fast=bf, yarn_beta_slow=bs)
    _close(out, ref, "yarn prefill")
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,d,window,prefix,q_pos0", [
    (1, 8, 2, 300, 300, 128, 0, 100, 0),     # prefix inside the first key tile... and beyond
    (1, 8, 2, 500, 500, 128, 64, 300, 0),    # prefix longer than the window, several tiles
    (2, 16, 1, 200, 200, 64, 0, 200, 0),     # the whole sequence is the prefix (bidirectional)
    (1, 4, 2, 70, 400, 128, 50, 350, 300),   # queries straddling the prefix end
])
def test_prefill_prefix(B, H_q, H_kv, S_q, S_k, d, window, prefix, q_pos0):
    dev = _dev()
    q, k, v = _qkv(B, H_q, H_kv, S_q, S_k, d, 600 + S_k + prefix)
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev), window=window, q_pos0=q_pos0, prefix_len=prefix)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, prefix_len=prefix)
    _close(out, ref, "prefix prefill")


@pytest.mark.parametrize("window", [0, 200])
def test_prefill_prerotated_keys(window):
    dev = _dev()
    q, k, v = _qkv(2, 8, 2, 520, 520, 128, 700 + window)
    k_rot = _prerotate(k)
    out = apex.fwd(q.to(dev), k_rot.to(dev), v.to(dev), window=window, keys_prerotated=True)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k_rot, v, window=window, keys_prerotated=True)
    _close(out, ref, "prerotated prefill")


def test_rope_keys_matches_oracle_rotation():
    dev = _dev()
    k = inputs.normal_bf16((2, 4, 300, 128), 800, 1)
    got = apex.rope_keys(k.to(dev)).cpu().double().numpy()
    pos = np.broadcast_to(np.arange(300)[None, None, :], (2, 4, 300)).reshape(-1)
    ref = oracle.rope(k.double().numpy().reshape(-1, 128), pos).reshape(k.shape)
    # one bf16 rounding of each rotated element
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_rope_keys_append_into_cache():
    """Rotating n new keys into rows [pos0, pos0 + n) of a larger cache leaves the rest untouched."""
    dev = _dev()
    S_cache, n, pos0, d = 256, 40, 100, 64
    cache = torch.zeros((3, S_cache, d), dtype=torch.bfloat16, device=dev)
    new = inputs.normal_bf16((3, n, d), 801, 1).to(dev)
    opt = apex._options()
    st = apex.apex_attn_rope_keys(new.data_ptr(), cache[:, pos0:].data_ptr(), 3, n, d, pos0, n * d, S_cache * d,
                                  opt, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    ref = apex.rope_keys(new.view(1, 3, n, d).contiguous(), pos0=pos0).view(3, n, d)
    torch.cuda.synchronize()
    assert torch.equal(cache[:, pos0:pos0 + n], ref)
    assert torch.count_nonzero(cache[:, :pos0]) == 0 and torch.count_nonzero(cache[:, pos0 + n:]) == 0


@pytest.mark.parametrize("B,H_q,H_kv,S_k,d,window,q_pos,prefix,yarn", [
    (2, 8, 2, 1000, 128, 0, 999, 0, (32.0, 32.0, 1.0)),
    (3, 16, 4, 777, 128, 100, 700, 0, (16.0, 8.0, 2.0)),
    (2, 8, 2, 600, 128, 0, 150, 400, None),     # query inside the prefix: sees keys [0, 400)
    (2, 8, 2, 600, 128, 64, 500, 400, None),    # query past the prefix: causal + window
    (1, 32, 8, 4096, 128, 0, 4095, 1024, None),
])
def test_decode_options(B, H_q, H_kv, S_k, d, window, q_pos, prefix, yarn):
    dev = _dev()
    q, k, v = _qkv(B, H_q, H_kv, 1, S_k, d, 900 + S_k + q_pos)
    ys = dict(yarn_scale=yarn[0], yarn_beta_fast=yarn[1], yarn_beta_slow=yarn[2]) if yarn else {}
    out = apex.decode(q.to(dev), k.to(dev), v.to(dev), q_pos, window=window, prefix_len=prefix, **ys)
    torch.cuda.synchronize()
    oys = dict(yarn_s=yarn[0], yarn_beta_fast=yarn[1], yarn_beta_slow=yarn[2]) if yarn else {}
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos, prefix_len=prefix, **oys)
    _close(out, ref, "decode options")


@pytest.mark.parametrize("window", [0, 300])
def test_decode_prerotated_cache(window):
    dev = _dev()
    q, k, v = _qkv(4, 16, 4, 1, 2000, 128, 950 + window)
    k_rot = _prerotate(k)
    out = apex.decode(q.to(dev), k_rot.to(dev), v.to(dev), 1999, window=window, keys_prerotated=True)
    torch.cuda.synchronize()
    ref = oracle.attn(q, k_rot, v, window=window, q_pos0=1999, keys_prerotated=True)
    _close(out, ref, "prerotated decode")


def test_ex_rejects_bad_options():
    dev = _dev()
    q, k, v = [t.to(dev) for t in _qkv(1, 4, 2, 64, 64, 64, 1)]
    with pytest.raises(apex.ApexError):
        apex.fwd(q, k, v, prefix_len=65)
    with pytest.raises(apex.ApexError):
        apex.fwd(q, k, v, yarn_scale=4.0, yarn_beta_fast=-1.0)
