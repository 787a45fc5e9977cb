"""Pins for the oracle's options beyond the plain block: YaRN frequency scaling
and attention temperature (Part 1, §5), the bidirectional prefix (Part 2, §11.1)
and keys given pre-rotated.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# YaRN (Part 1, §5)
# --------------------------------------------------------------------------

def test_yarn_worked_example(golden_dir):
    """§5.6: theta 1.0 unchanged, 0.0001 -> 0.0001/32, 0.01 (clamped) -> 0.01/32; factor 1.347."""
    g = _golden(golden_dir, "yarn_worked_example.json")
    th = np.array([p["theta"] for p in g["printed_pairs"]])
    got = oracle.yarn_scale_theta(th, g["s"], g["beta_fast"], g["beta_slow"])
    np.testing.assert_allclose(got, [p["theta_scaled"] for p in g["printed_pairs"]], rtol=1e-12)
    # the printed wavelengths 2 pi / theta
    for p in g["printed_pairs"]:
        assert abs(2 * math.pi / p["theta"] - p["wavelength"]) <= 5e-3 * p["wavelength"]
    assert abs(oracle.yarn_attn_factor(g["s"]) - g["printed_attn_factor"]) <= g["attn_factor_precision"]


def test_yarn_scale_one_is_plain_rope():
    """s = 1: no frequency scaling and a temperature of 1 (ln 1 = 0)."""
    assert oracle.yarn_attn_factor(1.0) == 1.0
    np.testing.assert_array_equal(oracle.yarn_theta(128, 10000.0, 1.0), oracle.rope_theta(128))
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((1, 2, 20, 16)), rng.standard_normal((1, 1, 20, 16)), rng.standard_normal((1, 1, 20, 16))
    np.testing.assert_array_equal(oracle.attn(q, k, v, yarn_s=1.0), oracle.attn(q, k, v))


def test_yarn_regime_edges():
    """Below beta_fast nothing changes, above beta_slow * s the frequency is divided
    by s, and inside the band the divisor t s + 1 - t stays in [1, s] (t clamped)."""
    s, bf, bs = 16.0, 8.0, 2.0
    lam = np.array([1.0, 7.9, 8.1, 20.0, 31.9, 32.1, 1e5])
    th = 2 * math.pi / lam
    got = oracle.yarn_scale_theta(th, s, bf, bs)
    assert got[0] == th[0] and got[1] == th[1]               # high frequency
    np.testing.assert_allclose(got[5:], th[5:] / s, rtol=1e-15)  # low frequency
    div = th[2:5] / got[2:5]
    assert np.all(div >= 1.0) and np.all(div <= s)
    t = np.clip((lam[2:5] / bs - 1) / (s - 1), 0, 1)
    np.testing.assert_allclose(div, t * s + 1 - t, rtol=1e-14)


def _rot(m, thetas):
    d = 2 * len(thetas)
    R = np.zeros((d, d))
    for i, th in enumerate(thetas):
        c, s_ = math.cos(m * th), math.sin(m * th)
        R[2 * i, 2 * i], R[2 * i, 2 * i + 1], R[2 * i + 1, 2 * i], R[2 * i + 1, 2 * i + 1] = c, -s_, s_, c
    return R


def _brute(q, k, v, thetas, factor, window=0, q_pos0=0, prefix_len=0):
    B, H_q, S_q, d = q.shape
    _, H_kv, S_k, _ = k.shape
    G = H_q // H_kv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H_q):
            g = h // G
            qr = np.stack([_rot(q_pos0 + r, thetas) @ q[b, h, r] for r in range(S_q)])
            kr = np.stack([_rot(j, thetas) @ k[b, g, j] for j in range(S_k)])
            sc = factor * (qr @ kr.T) / math.sqrt(d)
            m = q_pos0 + np.arange(S_q)[:, None]
            j = np.arange(S_k)[None, :]
            vis = (j <= m)
            if window > 0:
                vis &= (m - j < window)
            pre = (m < prefix_len)
            vis = np.where(pre, j < prefix_len, vis)
            out[b, h] = softmax(np.where(vis, sc, -np.inf), axis=1) @ v[b, g]
    return out


def test_yarn_attention_matches_dense_brute_force():
    """The scaled frequencies go into both rotations and the temperature multiplies
    the scores (factor and scaling rule pinned above)."""
    rng = np.random.default_rng(11)
    d, S, s = 16, 24, 32.0
    q, k, v = rng.standard_normal((1, 4, S, d)), rng.standard_normal((1, 2, S, d)), rng.standard_normal((1, 2, S, d))
    base = 50.0
    th = oracle.yarn_scale_theta(base ** (-2.0 * np.arange(d // 2) / d), s, 32.0, 1.0)
    ref = _brute(q, k, v, th, 0.1 * math.log(s) + 1.0, window=7)
    got = oracle.attn(q, k, v, window=7, rope_base=base, yarn_s=s)
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)
    # and it is not the plain block
    assert np.abs(got - oracle.attn(q, k, v, window=7, rope_base=base)).max() > 1e-3


# --------------------------------------------------------------------------
# Bidirectional prefix (Part 2, §11.1)
# --------------------------------------------------------------------------

def test_prefix_visual_rows(golden_dir):
    """§11.3: with P = 4 rows 0-3 see positions 0-3 in both pictures."""
    g = _golden(golden_dir, "mask_visual.json")
    S, P = g["S"], g["prefix_len"]
    q = np.zeros((1, 1, S, S))
    k = np.random.default_rng(4).standard_normal((1, 1, S, S))
    v = np.eye(S)[None, None]
    for window, rows in ((0, {**g["global_prefix_rows"], **g["global_causal_rows"]}),
                         (g["local_window"], {**g["local_prefix_rows"], **g["local_window_rows"]})):
        out = oracle.attn(q, k, v, window=window, prefix_len=P)[0, 0]
        for r, vis in rows.items():
            expect = np.zeros(S)
            expect[vis] = 1.0 / len(vis)
            np.testing.assert_allclose(out[int(r)], expect, atol=1e-15)


@pytest.mark.parametrize("window,prefix,q_pos0,S_q", [(0, 5, 0, 12), (3, 6, 0, 12), (4, 9, 2, 7), (0, 12, 0, 12)])
def test_prefix_matches_dense_brute_force(window, prefix, q_pos0, S_q):
    rng = np.random.default_rng(window * 100 + prefix)
    d, S_k = 8, 12
    q, k, v = rng.standard_normal((1, 2, S_q, d)), rng.standard_normal((1, 1, S_k, d)), rng.standard_normal((1, 1, S_k, d))
    th = 100.0 ** (-2.0 * np.arange(d // 2) / d)
    ref = _brute(q, k, v, th, 1.0, window=window, q_pos0=q_pos0, prefix_len=prefix)
    got = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, rope_base=100.0, prefix_len=prefix)
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def test_prefix_zero_and_one_are_plain_causal():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((1, 2, 15, 8)), rng.standard_normal((1, 1, 15, 8)), rng.standard_normal((1, 1, 15, 8))
    plain = oracle.attn(q, k, v, window=4)
    np.testing.assert_array_equal(oracle.attn(q, k, v, window=4, prefix_len=0), plain)
    np.testing.assert_array_equal(oracle.attn(q, k, v, window=4, prefix_len=1), plain)


# --------------------------------------------------------------------------
# Keys given already rotated
# --------------------------------------------------------------------------

def test_prerotated_keys_equal_rotating_in_the_block():
    rng = np.random.default_rng(6)
    B, H_q, H_kv, S, d = 2, 4, 2, 17, 16
    q, k, v = rng.standard_normal((B, H_q, S, d)), rng.standard_normal((B, H_kv, S, d)), rng.standard_normal((B, H_kv, S, d))
    k_rot = oracle.rope(k, np.broadcast_to(np.arange(S)[None, None, :], (B, H_kv, S)).reshape(-1))
    k_rot = k_rot.reshape(k.shape)
    a = oracle.attn(q, k, v, window=5)
    b = oracle.attn(q, k_rot, v, window=5, keys_prerotated=True)
    np.testing.assert_allclose(a, b, atol=1e-13, rtol=0)
