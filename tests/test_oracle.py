"""Pins for the fp64 oracle: the pages' worked examples, closed forms,
invariants and an independent dense brute force.  CPU only.

Each check is chosen so that a plausible slip in the oracle -- a wrong rotation
sign, a swapped pair index, a missing 1/sqrt(d_h), an off-by-one in the window,
strided instead of contiguous head groups, a query/key position mix-up -- makes
at least one of them fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from transformer_attention_rope_gb300 import inputs


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Worked examples printed on the pages
# --------------------------------------------------------------------------

def test_sdpa_worked_example(golden_dir):
    """Part 2, §6.4: softmax(QK^T/sqrt(2))V without mask or RoPE."""
    g = _golden(golden_dir, "sdpa_worked_example.json")
    Q = np.array(g["Q"], float)[None, None]
    K = np.array(g["K"], float)[None, None]
    V = np.array(g["V"], float)[None, None]
    out = oracle.attn(Q, K, V, causal=False, rope_base=0.0)[0, 0]
    np.testing.assert_allclose(out, np.array(g["printed_output"]), atol=g["print_precision"], rtol=0)
    # closed form: row 0 is [3, 4] by symmetry; row 1 is [1 + 6a, 2 + 6a] with
    # a = e^c / (1 + 2 e^c), c = 1/sqrt(2)
    c = 1.0 / math.sqrt(2.0)
    a = math.exp(c) / (1.0 + 2.0 * math.exp(c))
    np.testing.assert_allclose(out, [[3.0, 4.0], [1 + 6 * a, 2 + 6 * a]], atol=1e-13, rtol=0)


def test_sdpa_worked_example_weights(golden_dir):
    """The printed softmax weights follow from the oracle's output on one-hot V."""
    g = _golden(golden_dir, "sdpa_worked_example.json")
    Q = np.array(g["Q"], float)[None, None]
    K = np.array(g["K"], float)[None, None]
    w = np.zeros((2, 3))
    for c in range(3):  # V with a single 1 at key c reads out that key's weight
        V = np.zeros((1, 1, 3, 2))
        V[0, 0, c, 0] = 1.0
        w[:, c] = oracle.attn(Q, K, V, causal=False, rope_base=0.0)[0, 0][:, 0]
    np.testing.assert_allclose(w, np.array(g["printed_weights"]), atol=g["print_precision"], rtol=0)


def test_rope_worked_example(golden_dir):
    """Part 1, §4.6: d_head 4, position 3, q = [1, .5, .3, -.2]."""
    g = _golden(golden_dir, "rope_worked_example.json")
    th = oracle.rope_theta(g["d_head"], g["base"])
    np.testing.assert_allclose(th, g["printed_theta"], rtol=1e-12)
    out = oracle.rope(np.array(g["q"]), g["m"], g["base"])
    np.testing.assert_allclose(out, g["printed_output"], atol=g["tolerance"], rtol=0)
    # the page's cos/sin at the printed angles
    ang = g["m"] * th
    np.testing.assert_allclose(np.repeat(np.cos(ang), 2), g["printed_cos"], atol=5e-4)
    np.testing.assert_allclose(np.repeat(np.sin(ang), 2), g["printed_sin"], atol=5e-4)
    # magnitude preserved (the printed figure itself is a misprint)
    assert abs(np.linalg.norm(out) - np.linalg.norm(g["q"])) < 1e-14


def test_rope_theta_geometric():
    """Part 1, §4.3: theta_0 = 1 and successive pairs shrink by base^(-2/d_h)."""
    for d in (8, 64, 128):
        th = oracle.rope_theta(d, 10000.0)
        assert th[0] == 1.0
        np.testing.assert_allclose(th[1:] / th[:-1], 10000.0 ** (-2.0 / d), rtol=1e-13)
        assert np.all(np.diff(th) < 0)


def test_gqa_assignment(golden_dir):
    """Part 2, §8.4: Q0,Q1 use KV head 0 and Q2,Q3 use KV head 1."""
    g = _golden(golden_dir, "gqa_assignment.json")
    rng = np.random.default_rng(7)
    S, d = 9, 8
    q = rng.standard_normal((1, g["H_q"], S, d))
    k = rng.standard_normal((1, g["H_kv"], S, d))
    v = rng.standard_normal((1, g["H_kv"], S, d))
    out = oracle.attn(q, k, v, window=0)
    for h, kvh in enumerate(g["query_head_to_kv_head"]):
        single = oracle.attn(q[:, h:h + 1], k[:, kvh:kvh + 1], v[:, kvh:kvh + 1])
        np.testing.assert_array_equal(out[:, h:h + 1], single)


def test_mask_visual_rows(golden_dir):
    """Part 2, §11.3: which keys rows 4/5/7/9 see, causal and with W = 4.

    With Q = 0 every visible key gets the same weight, and V = identity makes
    row r of the output equal to the indicator of r's visible set / its size.
    """
    g = _golden(golden_dir, "mask_visual.json")
    S = g["S"]
    d = S  # even, and wide enough for one-hot values
    q = np.zeros((1, 1, S, d))
    k = np.random.default_rng(3).standard_normal((1, 1, S, d))
    v = np.eye(S)[None, None]
    for window, rows in ((0, g["global_causal_rows"]), (g["local_window"], g["local_window_rows"])):
        out = oracle.attn(q, k, v, window=window)[0, 0]
        for r, vis in rows.items():
            expect = np.zeros(S)
            expect[vis] = 1.0 / len(vis)
            np.testing.assert_allclose(out[int(r)], expect, atol=1e-15)


# --------------------------------------------------------------------------
# Invariants and closed forms
# --------------------------------------------------------------------------

def test_rope_preserves_norm():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 128))
    pos = rng.integers(0, 200000, size=64)
    y = oracle.rope(x, pos)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 64))
    np.testing.assert_array_equal(oracle.rope(x, 0), x)


def test_rope_composes_additively():
    """A rotation by a then by b is a rotation by a + b (angle linear in m)."""
    x = np.random.default_rng(2).standard_normal((16, 64))
    for a, b in ((3, 5), (100, 4000), (65535, 1)):
        np.testing.assert_allclose(oracle.rope(oracle.rope(x, a), b), oracle.rope(x, a + b),
                                   atol=1e-10)


def test_rope_relative_position():
    """Part 1, §4.5: <RoPE(q,m), RoPE(k,n)> depends on m - n only."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    for m, n in ((10, 3), (4000, 4100), (60000, 59000)):
        ref = oracle.rope(q, m) @ oracle.rope(k, n)
        for c in (1, 17, 1000, 5000):
            got = oracle.rope(q, m + c) @ oracle.rope(k, n + c)
            assert abs(got - ref) < 1e-9 * max(1.0, abs(ref))
    # and it does change with m - n
    assert abs(oracle.rope(q, 10) @ oracle.rope(k, 3) - oracle.rope(q, 11) @ oracle.rope(k, 3)) > 1e-3


def test_rope_rotates_interleaved_pairs():
    """The rotation mixes (x_2i, x_2i+1) only: a vector supported on one pair stays there."""
    d = 16
    for i in range(d // 2):
        x = np.zeros(d)
        x[2 * i] = 1.0
        y = oracle.rope(x, 7)
        th = 10000.0 ** (-2.0 * i / d)
        expect = np.zeros(d)
        expect[2 * i] = math.cos(7 * th)
        expect[2 * i + 1] = math.sin(7 * th)
        np.testing.assert_allclose(y, expect, atol=1e-15)


def _rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def test_gqa_equals_mha_on_repeated_kv():
    """Part 2, §8.2: GQA == MHA with each KV head repeated G times (contiguously)."""
    B, H_q, H_kv, S, d = 2, 8, 2, 37, 16
    q, k, v = _rand_bf16((B, H_q, S, d), 1), _rand_bf16((B, H_kv, S, d), 2), _rand_bf16((B, H_kv, S, d), 3)
    G = H_q // H_kv
    out = oracle.attn(q, k, v, window=5)
    ref = oracle.attn(q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1), window=5)
    np.testing.assert_array_equal(out, ref)
    # strided sharing (head i -> i mod H_kv) is a different function
    bad = oracle.attn(q, k.repeat(1, G, 1, 1), v.repeat(1, G, 1, 1), window=5)
    assert np.abs(bad - out).max() > 1e-2


def test_window_at_least_seq_is_causal():
    B, H, S, d = 1, 2, 40, 8
    q, k, v = _rand_bf16((B, H, S, d), 4), _rand_bf16((B, H, S, d), 5), _rand_bf16((B, H, S, d), 6)
    causal = oracle.attn(q, k, v, window=0)
    for W in (S, S + 1, 10 * S):
        np.testing.assert_array_equal(oracle.attn(q, k, v, window=W), causal)
    assert np.abs(oracle.attn(q, k, v, window=S - 1) - causal).max() > 1e-3


def test_window_one_returns_own_value():
    """W = 1: each query sees only its own key, so out[r] = v[r] exactly."""
    B, H, S, d = 1, 3, 25, 8
    q, k, v = _rand_bf16((B, H, S, d), 7), _rand_bf16((B, H, S, d), 8), _rand_bf16((B, H, S, d), 9)
    out = oracle.attn(q, k, v, window=1)
    np.testing.assert_array_equal(out, v.double().numpy())


def test_first_row_returns_first_value():
    """Causal row 0 sees key 0 only."""
    q, k, v = _rand_bf16((1, 2, 9, 8), 10), _rand_bf16((1, 2, 9, 8), 11), _rand_bf16((1, 2, 9, 8), 12)
    out = oracle.attn(q, k, v)
    np.testing.assert_array_equal(out[:, :, 0], v[:, :, 0].double().numpy())


def test_softmax_shift_invariance_through_query_scale():
    """Scaling q by 0 gives the plain running mean of the visible values."""
    S, d = 12, 8
    q = np.zeros((1, 1, S, d))
    k = np.random.default_rng(0).standard_normal((1, 1, S, d))
    v = np.random.default_rng(1).standard_normal((1, 1, S, d))
    out = oracle.attn(q, k, v)[0, 0]
    expect = np.cumsum(v[0, 0], axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(out, expect, atol=1e-14)


# --------------------------------------------------------------------------
# Independent dense brute force on tiny inputs
# --------------------------------------------------------------------------

def _rot_matrix(m, d, base):
    """Block-diagonal matrix of Part 1, §4.2's 2x2 rotations at position m."""
    R = np.zeros((d, d))
    for i in range(d // 2):
        a = m * base ** (-2.0 * i / d)
        c, s = math.cos(a), math.sin(a)
        R[2 * i, 2 * i], R[2 * i, 2 * i + 1] = c, -s
        R[2 * i + 1, 2 * i], R[2 * i + 1, 2 * i + 1] = s, c
    return R


def _brute(q, k, v, window, q_pos0, base):
    B, H_q, S_q, d = q.shape
    _, H_kv, S_k, _ = k.shape
    G = H_q // H_kv
    out = np.zeros_like(q)
    Rk = np.stack([_rot_matrix(j, d, base) for j in range(S_k)])
    Rq = np.stack([_rot_matrix(q_pos0 + r, d, base) for r in range(S_q)])
    for b in range(B):
        for h in range(H_q):
            kv = [hh for hh in range(H_kv) if hh * G <= h < (hh + 1) * G][0]
            qr = np.einsum("rij,rj->ri", Rq, q[b, h])
            kr = np.einsum("rij,rj->ri", Rk, k[b, kv])
            scores = qr @ kr.T / math.sqrt(d)
            i = q_pos0 + np.arange(S_q)[:, None]
            j = np.arange(S_k)[None, :]
            mask = (j <= i)
            if window > 0:
                mask &= (i - j >= 0) & (i - j < window)
            scores = np.where(mask, scores, -np.inf)
            out[b, h] = softmax(scores, axis=1) @ v[b, kv]
    return out


@pytest.mark.parametrize("B,H_q,H_kv,S_q,S_k,d,window,q_pos0", [
    (1, 1, 1, 7, 7, 2, 0, 0),
    (1, 2, 1, 9, 9, 4, 3, 0),
    (2, 4, 2, 16, 16, 8, 5, 0),
    (1, 4, 4, 5, 13, 8, 0, 8),
    (1, 6, 2, 3, 16, 4, 4, 13),
    (1, 2, 2, 1, 11, 8, 0, 10),
])
def test_matches_dense_brute_force(B, H_q, H_kv, S_q, S_k, d, window, q_pos0):
    rng = np.random.default_rng(B * 1000 + S_k * 10 + d)
    q = rng.standard_normal((B, H_q, S_q, d))
    k = rng.standard_normal((B, H_kv, S_k, d))
    v = rng.standard_normal((B, H_kv, S_k, d))
    got = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, rope_base=500.0)
    ref = _brute(q, k, v, window, q_pos0, 500.0)
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


# --------------------------------------------------------------------------
# Consistency of the oracle's own options
# --------------------------------------------------------------------------

def test_row_subset_and_threads_are_exact():
    B, H_q, H_kv, S, d = 2, 4, 2, 70, 16
    q, k, v = _rand_bf16((B, H_q, S, d), 20), _rand_bf16((B, H_kv, S, d), 21), _rand_bf16((B, H_kv, S, d), 22)
    full = oracle.attn(q, k, v, window=9, threads=1)
    np.testing.assert_array_equal(oracle.attn(q, k, v, window=9, threads=5), full)
    rows = [69, 0, 33, 8, 9]
    np.testing.assert_array_equal(oracle.attn(q, k, v, window=9, rows=rows), full[:, :, rows])


def test_decode_is_last_prefill_row():
    B, H_q, H_kv, S, d = 2, 4, 1, 50, 8
    q, k, v = _rand_bf16((B, H_q, S, d), 30), _rand_bf16((B, H_kv, S, d), 31), _rand_bf16((B, H_kv, S, d), 32)
    full = oracle.attn(q, k, v, window=7)
    dec = oracle.attn(q[:, :, -1:].contiguous(), k, v, window=7, q_pos0=S - 1)
    np.testing.assert_array_equal(dec, full[:, :, -1:])


def test_bf16_inputs_read_exactly():
    """bf16 tensors and their exact float64 values give bitwise-equal results."""
    q, k, v = _rand_bf16((1, 2, 10, 8), 40), _rand_bf16((1, 1, 10, 8), 41), _rand_bf16((1, 1, 10, 8), 42)
    a = oracle.attn(q, k, v)
    b = oracle.attn(q.double().numpy(), k.double().numpy(), v.double().numpy())
    np.testing.assert_array_equal(a, b)


def test_rejects_bad_arguments():
    q = np.zeros((1, 3, 4, 8))
    k = np.zeros((1, 2, 4, 8))
    with pytest.raises(ValueError):
        oracle.attn(q, k, k)  # 3 query heads over 2 KV heads
    with pytest.raises(ValueError):
        oracle.attn(np.zeros((1, 1, 4, 8)), np.zeros((1, 1, 4, 8)), np.zeros((1, 1, 4, 8)), rows=[4])


# --------------------------------------------------------------------------
# The input generator
# --------------------------------------------------------------------------

def test_generator_deterministic_and_seeded():
    a = inputs.normal_bf16((3, 1000), 5, 1)
    b = inputs.normal_bf16((3, 1000), 5, 1)
    c = inputs.normal_bf16((3, 1000), 6, 1)
    d = inputs.normal_bf16((3, 1000), 5, 2)
    assert a.dtype == torch.bfloat16
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_generator_chunking_is_thread_independent(monkeypatch):
    n = inputs.CHUNK * 2 + 123
    a = inputs.normal_bf16((n,), 9, 0)
    monkeypatch.setattr(inputs, "_threads", lambda: 1)
    b = inputs.normal_bf16((n,), 9, 0)
    assert torch.equal(a, b)


def test_generator_score_variance():
    """Part 2, §6.3: for N(0,1) entries Var(q.k) = d_h, so the scaled score has variance 1."""
    d = 128
    q = inputs.normal_bf16((20000, d), 1, 0).double()
    k = inputs.normal_bf16((20000, d), 1, 1).double()
    s = (q * k).sum(1) / math.sqrt(d)
    assert abs(float(s.mean())) < 0.03
    assert abs(float(s.var()) - 1.0) < 0.05
