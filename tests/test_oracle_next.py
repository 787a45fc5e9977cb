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
    by s, and inside the band the divisor stays in [1, s]."""
    s, bf, bs = 16.0, 8.0, 2.0
    lam = np.array([1.0, 7.9, 8.1, 20.0, 31.9, 32.1, 1e5])
    th = 2 * math.pi / lam
    got = oracle.yarn_scale_theta(th, s, bf, bs)
    assert got[0] == th[0] and got[1] == th[1]               # high frequency
    np.testing.assert_allclose(got[5:], th[5:] / s, rtol=1e-15)  # low frequency
    div = th[2:5] / got[2:5]
    assert np.all(div >= 1.0) and np.all(div <= s)


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


# --------------------------------------------------------------------------
# YaRN middle band: properties the pages fix, not the formula typed again.
# Part 1, §5.3 sorts the pairs into three regimes by wavelength: short ones
# are left alone, long ones (beyond beta_slow * s) get theta / s, and the band
# between them moves gradually from the first treatment to the second.  In
# §5.4, t weighs the two: t = 0 keeps theta, t = 1 gives theta / s.  Hence:
#   (a) the divisor theta / theta' lies in [1, s] everywhere;
#   (b) it never falls as the wavelength grows;
#   (c) the band joins the fully scaled regime without a jump at
#       lambda = beta_slow * s (t reaches 1 there);
#   (d) inside the band, where t is not clamped, the divisor grows strictly.
# The lower edge has a jump under the pages' formula: at lambda = beta_fast,
# t = (beta_fast / beta_slow - 1) / (s - 1), which is 0 only when
# beta_fast = beta_slow (with the defaults 32 and 1 it is 1, so the pairs go
# from unscaled straight to fully scaled); (b) still holds across it.
# --------------------------------------------------------------------------

# (s, beta_fast, beta_slow): the defaults at s = 32 and 8, a band wider than
# the defaults give, and one with beta_fast < beta_slow, where t < 0 occurs
# inside the band and the clamp decides
YARN_CONFIGS = [(32.0, 32.0, 1.0), (8.0, 32.0, 1.0), (16.0, 8.0, 2.0), (16.0, 2.0, 8.0), (4.0, 3.0, 3.0)]


def _divisors(scale_fn, s, bf, bs, lam):
    th = 2 * math.pi / lam
    return th / np.asarray(scale_fn(th, s, bf, bs), dtype=np.float64)


def _wavelength_grid(s, bf, bs):
    lo, hi = min(bf, bs) / 4.0, bs * s * 4.0
    return np.geomspace(lo, hi, 4001)


def _check_bounds(scale_fn, s, bf, bs):
    div = _divisors(scale_fn, s, bf, bs, _wavelength_grid(s, bf, bs))
    return bool(np.all(div >= 1.0 - 1e-12) and np.all(div <= s * (1 + 1e-12)))


def _check_monotone(scale_fn, s, bf, bs):
    div = _divisors(scale_fn, s, bf, bs, _wavelength_grid(s, bf, bs))
    return bool(np.all(np.diff(div) >= -1e-12 * div[1:]))


def _check_upper_edge(scale_fn, s, bf, bs):
    edge = bs * s
    if edge <= bf:  # no band below the edge
        return True
    lam = edge * (1.0 - np.array([1e-3, 1e-6, 1e-9]))
    div = _divisors(scale_fn, s, bf, bs, lam)
    return bool(np.all(np.abs(div - s) <= 4.0 * s * (1.0 - lam / edge) * max(1.0, edge / bs) + 1e-9))


def _check_strict_in_band(scale_fn, s, bf, bs):
    lo, hi = max(bf, bs), bs * s  # the part of the band where 0 <= t <= 1
    if hi <= lo * 1.001:
        return True
    lam = np.geomspace(lo * 1.0005, hi * 0.9995, 200)
    div = _divisors(scale_fn, s, bf, bs, lam)
    return bool(np.all(np.diff(div) > 0))


YARN_CHECKS = (_check_bounds, _check_monotone, _check_upper_edge, _check_strict_in_band)


@pytest.mark.parametrize("s,bf,bs", YARN_CONFIGS)
@pytest.mark.parametrize("check", YARN_CHECKS, ids=lambda f: f.__name__[7:])
def test_yarn_band_properties(check, s, bf, bs):
    assert check(oracle.yarn_scale_theta, s, bf, bs)


def test_yarn_lower_edge_jump_is_the_pages_reading():
    """With the defaults (beta_fast 32, beta_slow 1) the pair just above a
    wavelength of 32 is already fully scaled, the pair just below it not at
    all: the discontinuity the §5.4 formula implies at beta_fast."""
    s = 32.0
    div = _divisors(oracle.yarn_scale_theta, s, 32.0, 1.0, np.array([31.999, 32.001]))
    assert div[0] == 1.0
    assert abs(div[1] - s) <= 1e-3 * s


def test_yarn_pins_catch_planted_mistakes():
    """Plausible misreadings of §5.4 (beta_fast in place of beta_slow in t,
    the divisor written t + (1 - t) s, the clamp of t left out) each fail at
    least one of the band properties above on at least one configuration."""
    def make(t_of, divisor, clamp):
        def scale(th, s, bf, bs):
            th = np.asarray(th, dtype=np.float64)
            lam = 2 * math.pi / th
            t = t_of(lam, s, bf, bs)
            if clamp:
                t = np.clip(t, 0.0, 1.0)
            mid = th / divisor(t, s)
            return np.where(lam < bf, th, np.where(lam > bs * s, th / s, mid))
        return scale

    right_t = lambda lam, s, bf, bs: (lam / bs - 1.0) / (s - 1.0)
    right_div = lambda t, s: t * s + (1.0 - t)
    # the restated rule itself passes every check (so the checks are not vacuous
    # for the mutants below)
    ok = make(right_t, right_div, True)
    assert all(c(ok, *cfg) for c in YARN_CHECKS for cfg in YARN_CONFIGS)
    mutants = {
        "beta_fast in t": make(lambda lam, s, bf, bs: (lam / bf - 1.0) / (s - 1.0), right_div, True),
        "divisor t + (1 - t) s": make(right_t, lambda t, s: t + (1.0 - t) * s, True),
        "no clamp": make(right_t, right_div, False),
    }
    for name, fn in mutants.items():
        failed = [(c.__name__, cfg) for c in YARN_CHECKS for cfg in YARN_CONFIGS if not c(fn, *cfg)]
        assert failed, name
