"""Pins of the oracle's multi-head latent attention with decoupled RoPE
(APEX-1 Mathematical Reference -- Part 2, §9.3): query and key rows are
[content (d_h) | rope part (d_r)], only the rope part is rotated (as a
d_r-dimensional RoPE vector), value rows have length d_h.

Each pin reduces the MLA call to other, separately pinned oracle functions
(plain attention, RoPE) through an identity that holds exactly in real
arithmetic, or checks a property any correct implementation has:
  * content parts zero  -> plain RoPE attention of the rope parts (d = d_r),
    with the score scale 1/sqrt(d_h + d_r) carried by the queries;
  * rope parts zero     -> plain attention without RoPE of the content parts;
  * general inputs      -> plain attention without RoPE of the vectors whose
    rope parts were rotated beforehand, values padded with zero columns;
  * GQA                 -> MHA on repeated KV heads (Part 2, §8.2);
  * a wrong choice of rotated entries, frequency dimension or scale fails one
    of the above (checked on planted variants below).
"""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(20260)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _case(B=1, H_q=4, H_kv=2, S=24, d_h=16, d_r=8):
    q = _rand(B, H_q, S, d_h + d_r)
    k = _rand(B, H_kv, S, d_h + d_r)
    v = _rand(B, H_kv, S, d_h)
    return q, k, v


def _rotate_tail(x, d_r, pos, base=10000.0):
    """Rotate the trailing d_r entries of x[B, H, S, d] at positions pos[S] with the pinned RoPE."""
    out = x.copy()
    B, H, S, d = x.shape
    p = np.broadcast_to(np.asarray(pos)[None, None, :], (B, H, S)).reshape(-1)
    out[..., d - d_r:] = oracle.rope(x[..., d - d_r:].reshape(-1, d_r), p, base).reshape(B, H, S, d_r)
    return out


@pytest.mark.parametrize("window", [0, 5])
def test_content_zero_is_rope_attention_of_rope_part(window):
    d_h, d_r = 16, 8
    q, k, v = _case(d_h=d_h, d_r=d_r)
    q[..., :d_h] = 0.0
    k[..., :d_h] = 0.0
    got = oracle.mla_attn(q, k, v, d_r, window=window)
    c = math.sqrt(d_r / (d_h + d_r))  # plain attention divides by sqrt(d_r)
    for blk in range(d_h // d_r):
        ref = oracle.attn(q[..., d_h:] * c, k[..., d_h:], v[..., blk * d_r:(blk + 1) * d_r], window=window)
        np.testing.assert_allclose(got[..., blk * d_r:(blk + 1) * d_r], ref, rtol=0, atol=1e-12)


def test_rope_part_zero_is_plain_attention_without_rope():
    d_h, d_r = 16, 8
    q, k, v = _case(d_h=d_h, d_r=d_r)
    q[..., d_h:] = 0.0
    k[..., d_h:] = 0.0
    got = oracle.mla_attn(q, k, v, d_r, window=7, q_pos0=0)
    c = math.sqrt(d_h / (d_h + d_r))
    ref = oracle.attn(q[..., :d_h] * c, k[..., :d_h], v, window=7, rope_base=0.0)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("window,q_pos0,prefix", [(0, 0, 0), (6, 0, 0), (0, 10, 0), (4, 0, 9)])
def test_general_equals_prerotated_plain_attention(window, q_pos0, prefix):
    d_h, d_r = 16, 8
    B, H_q, H_kv, S_k = 2, 4, 2, 30
    S_q = S_k - q_pos0
    q = _rand(B, H_q, S_q, d_h + d_r)
    k = _rand(B, H_kv, S_k, d_h + d_r)
    v = _rand(B, H_kv, S_k, d_h)
    got = oracle.mla_attn(q, k, v, d_r, window=window, q_pos0=q_pos0, prefix_len=prefix)
    q_rot = _rotate_tail(q, d_r, np.arange(q_pos0, q_pos0 + S_q))
    k_rot = _rotate_tail(k, d_r, np.arange(S_k))
    v_pad = np.concatenate([v, np.zeros((B, H_kv, S_k, d_r))], axis=-1)
    ref = oracle.attn(q_rot, k_rot, v_pad, window=window, q_pos0=q_pos0, rope_base=0.0, prefix_len=prefix)
    np.testing.assert_allclose(got, ref[..., :d_h], rtol=0, atol=1e-12)
    assert np.all(np.abs(ref[..., d_h:]) == 0.0)


def test_keys_prerotated_matches_rotating_in_the_oracle():
    d_h, d_r = 16, 8
    q, k, v = _case(d_h=d_h, d_r=d_r, S=20)
    k_rot = _rotate_tail(k, d_r, np.arange(20))
    a = oracle.mla_attn(q, k, v, d_r)
    b = oracle.mla_attn(q, k_rot, v, d_r, keys_prerotated=True)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_gqa_equals_mha_on_repeated_kv():
    d_h, d_r = 16, 8
    q, k, v = _case(B=1, H_q=6, H_kv=2, S=18, d_h=d_h, d_r=d_r)
    got = oracle.mla_attn(q, k, v, d_r, window=9)
    ref = oracle.mla_attn(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), d_r, window=9)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_bf16_inputs_read_exactly():
    d_h, d_r = 16, 8
    q, k, v = _case(d_h=d_h, d_r=d_r)
    qb, kb, vb = [torch.from_numpy(x).to(torch.bfloat16) for x in (q, k, v)]
    a = oracle.mla_attn(qb, kb, vb, d_r, window=3)
    b = oracle.mla_attn(qb.double().numpy(), kb.double().numpy(), vb.double().numpy(), d_r, window=3)
    np.testing.assert_array_equal(a, b)


def test_rows_subset_and_shape_checks():
    d_h, d_r = 16, 8
    q, k, v = _case(d_h=d_h, d_r=d_r)
    full = oracle.mla_attn(q, k, v, d_r)
    part = oracle.mla_attn(q, k, v, d_r, rows=[3, 17, 0])
    np.testing.assert_array_equal(part, full[:, :, [3, 17, 0]])
    with pytest.raises(ValueError):
        oracle.mla_attn(q, k, v[..., :-1], d_r)
    with pytest.raises(ValueError):
        oracle.mla_attn(q, k, v, 7)


def test_pins_catch_planted_mistakes():
    """Variants with a plausible mistake (rotating the leading entries, thetas
    from the full row length, the scale of d_h alone) differ from the oracle
    by far more than the pins' tolerance."""
    d_h, d_r = 16, 8
    B, H, S = 1, 2, 20
    q = _rand(B, H, S, d_h + d_r)
    k = _rand(B, H, S, d_h + d_r)
    v = _rand(B, H, S, d_h)
    got = oracle.mla_attn(q, k, v, d_r)
    v_pad = np.concatenate([v, np.zeros((B, H, S, d_r))], axis=-1)
    pos = np.arange(S)
    # 1. rotate the leading d_r entries instead of the trailing ones
    lead = lambda x: np.concatenate([oracle.rope(x[..., :d_r].reshape(-1, d_r),
                                                 np.broadcast_to(pos[None, None], (B, H, S)).reshape(-1)
                                                 ).reshape(B, H, S, d_r), x[..., d_r:]], axis=-1)
    bad1 = oracle.attn(lead(q), lead(k), v_pad, rope_base=0.0)[..., :d_h]
    # 2. frequencies of a (d_h + d_r)-dimensional RoPE applied to the whole row
    bad2 = oracle.attn(q, k, v_pad)[..., :d_h]
    # 3. scores divided by sqrt(d_h) instead of sqrt(d_h + d_r)
    c = math.sqrt((d_h + d_r) / d_h)
    bad3 = oracle.attn(_rotate_tail(q, d_r, pos) * c, _rotate_tail(k, d_r, pos), v_pad, rope_base=0.0)[..., :d_h]
    for bad in (bad1, bad2, bad3):
        assert np.abs(bad - got).max() > 1e-3
