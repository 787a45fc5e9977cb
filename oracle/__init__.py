"""fp64 CPU oracle for the APEX-1 attention block -- TEST INFRASTRUCTURE ONLY.

The oracle is the yardstick the CUDA library is checked against.  Only the
tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it; the product package never does.  It shares no code
with the CUDA path: the arithmetic lives in ``oracle.c`` (plain C, double
precision), written from the formulas of "APEX-1 Mathematical Reference --
Part 1" (§4 RoPE) and "-- Part 2" (§6 scaled dot-product attention, §8 GQA,
§9.3 decoupled RoPE, §10 sliding window).  This module only compiles that file
and marshals arrays.

Every function here is pinned by ``tests/test_oracle*.py`` against the pages'
worked examples, closed forms, invariants and an independent brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (plain gcc, no -march)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Opts(ctypes.Structure):
    _fields_ = [("yarn_s", ctypes.c_double), ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double),
                ("prefix_len", ctypes.c_int), ("keys_prerotated", ctypes.c_int)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
            vp = ctypes.c_void_p
            lib.oracle_rope_f64.argtypes = [vp, vp, i64, i32, vp, f64]
            lib.oracle_rope_f64.restype = i32
            lib.oracle_rope_theta_f64.argtypes = [i32, f64, vp]
            lib.oracle_rope_theta_f64.restype = i32
            for name in ("oracle_attn_bf16", "oracle_attn_f64"):
                fn = getattr(lib, name)
                fn.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i64, f64, i32,
                               vp, i32, i32]
                fn.restype = i32
            for name in ("oracle_attn_ex_bf16", "oracle_attn_ex_f64"):
                fn = getattr(lib, name)
                fn.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i64, f64, i32,
                               vp, i32, i32, ctypes.POINTER(_Opts)]
                fn.restype = i32
            for name in ("oracle_mla_attn_bf16", "oracle_mla_attn_f64"):
                fn = getattr(lib, name)
                fn.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i64, f64, i32,
                               vp, i32, i32, ctypes.POINTER(_Opts)]
                fn.restype = i32
            lib.oracle_yarn_theta_f64.argtypes = [i32, f64, f64, f64, f64, vp]
            lib.oracle_yarn_theta_f64.restype = i32
            lib.oracle_yarn_scale_theta_f64.argtypes = [vp, i32, f64, f64, f64, vp]
            lib.oracle_yarn_scale_theta_f64.restype = i32
            lib.oracle_yarn_attn_factor.argtypes = [f64]
            lib.oracle_yarn_attn_factor.restype = f64
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def rope_theta(d: int, base: float = 10000.0) -> np.ndarray:
    """theta_i = base^(-2i/d) for i < d/2 (Part 1, §4.3)."""
    out = np.empty(d // 2, dtype=np.float64)
    rc = _load().oracle_rope_theta_f64(d, float(base), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_rope_theta_f64: bad arguments")
    return out


def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """RoPE of the rows of x[..., d] at positions pos (Part 1, §4.2-§4.4)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64), (flat.shape[0],)))
    out = np.empty_like(flat)
    rc = _load().oracle_rope_f64(_ptr(flat), _ptr(out), flat.shape[0], d, _ptr(p), float(base))
    if rc != 0:
        raise ValueError("oracle_rope_f64: bad arguments")
    return out.reshape(x.shape)


def yarn_theta(d: int, base: float = 10000.0, s: float = 1.0, beta_fast: float = 32.0,
               beta_slow: float = 1.0) -> np.ndarray:
    """YaRN-scaled theta'_i (Part 1, §5.3-§5.4)."""
    out = np.empty(d // 2, dtype=np.float64)
    rc = _load().oracle_yarn_theta_f64(d, float(base), float(s), float(beta_fast), float(beta_slow), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_yarn_theta_f64: bad arguments")
    return out


def yarn_scale_theta(theta, s: float, beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """The YaRN rule of Part 1, §5.3-§5.4 applied to given frequencies."""
    th = np.ascontiguousarray(np.asarray(theta, dtype=np.float64).ravel())
    out = np.empty_like(th)
    rc = _load().oracle_yarn_scale_theta_f64(_ptr(th), th.shape[0], float(s), float(beta_fast),
                                             float(beta_slow), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_yarn_scale_theta_f64: bad arguments")
    return out


def yarn_attn_factor(s: float) -> float:
    """Attention temperature 0.1 ln(s) + 1 (Part 1, §5.5); 1 for s <= 1."""
    return float(_load().oracle_yarn_attn_factor(float(s)))


def _as_bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> contiguous uint16 numpy array of its bits."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 tensor")
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def attn(q, k, v, *, window: int = 0, q_pos0: int = 0, rope_base: float = 10000.0,
         causal: bool = True, rows=None, threads: int | None = None, yarn_s: float = 1.0,
         yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0, prefix_len: int = 0,
         keys_prerotated: bool = False) -> np.ndarray:
    """Attention block in fp64.

    q [B, H_q, S_q, d]; k, v [B, H_kv, S_k, d].  bf16 torch tensors are read as
    their exact bf16 values; anything else is taken as float64.  Returns
    out [B, H_q, n_rows, d] (float64), n_rows = S_q or len(rows).
    rope_base <= 0 disables RoPE; causal=False disables the mask (both only for
    the unmasked worked example of Part 2, §6.4).  yarn_s > 1 scales the RoPE
    frequencies and the scores (Part 1, §5); prefix_len > 0 makes positions
    [0, prefix_len) attend to each other bidirectionally (Part 2, §11.1);
    keys_prerotated uses k as already rotated.
    """
    import torch
    bf16 = isinstance(q, torch.Tensor) and q.dtype == torch.bfloat16
    if bf16:
        qa, ka, va = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        fn = _load().oracle_attn_ex_bf16
    else:
        cv = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64))
        qa, ka, va = cv(q), cv(k), cv(v)
        fn = _load().oracle_attn_ex_f64
    opts = _Opts(float(yarn_s), float(yarn_beta_fast), float(yarn_beta_slow), int(prefix_len),
                 1 if keys_prerotated else 0)
    B, H_q, S_q, d = qa.shape
    Bk, H_kv, S_k, dk = ka.shape
    if va.shape != ka.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch between q, k, v")
    if rows is None:
        rows_arr, n_rows, rows_ptr = None, S_q, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n_rows, rows_ptr = int(rows_arr.shape[0]), _ptr(rows_arr)
    out = np.empty((B, H_q, n_rows, d), dtype=np.float64)
    rc = fn(_ptr(qa), _ptr(ka), _ptr(va), _ptr(out), B, H_q, H_kv, S_q, S_k, d, int(window),
            int(q_pos0), float(rope_base), 1 if causal else 0, rows_ptr, n_rows,
            int(threads or default_threads()), ctypes.byref(opts))
    if rc != 0:
        raise ValueError("oracle_attn failed with code %d" % rc)
    return out


def mla_attn(q, k, v, d_rope: int, *, window: int = 0, q_pos0: int = 0, rope_base: float = 10000.0,
             causal: bool = True, rows=None, threads: int | None = None, yarn_s: float = 1.0,
             yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0, prefix_len: int = 0,
             keys_prerotated: bool = False) -> np.ndarray:
    """Multi-head latent attention with decoupled RoPE in fp64 (Part 2, §9.3).

    q [B, H_q, S_q, d_h + d_rope], k [B, H_kv, S_k, d_h + d_rope] hold
    [content | rope part] rows; v [B, H_kv, S_k, d_h].  Only the rope part is
    rotated (a d_rope-dimensional RoPE); scores are divided by
    sqrt(d_h + d_rope).  Returns out [B, H_q, n_rows, d_h] (float64).  The
    other arguments are those of attn(); keys_prerotated means the rope part of
    k is already rotated.
    """
    import torch
    bf16 = isinstance(q, torch.Tensor) and q.dtype == torch.bfloat16
    if bf16:
        qa, ka, va = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        fn = _load().oracle_mla_attn_bf16
    else:
        cv = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64))
        qa, ka, va = cv(q), cv(k), cv(v)
        fn = _load().oracle_mla_attn_f64
    B, H_q, S_q, d_qk = qa.shape
    Bk, H_kv, S_k, dk = ka.shape
    d_h = d_qk - int(d_rope)
    if Bk != B or dk != d_qk or va.shape != (B, H_kv, S_k, d_h) or d_h <= 0:
        raise ValueError("shape mismatch between q, k, v for d_rope=%d" % d_rope)
    opts = _Opts(float(yarn_s), float(yarn_beta_fast), float(yarn_beta_slow), int(prefix_len),
                 1 if keys_prerotated else 0)
    if rows is None:
        rows_arr, n_rows, rows_ptr = None, S_q, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n_rows, rows_ptr = int(rows_arr.shape[0]), _ptr(rows_arr)
    out = np.empty((B, H_q, n_rows, d_h), dtype=np.float64)
    rc = fn(_ptr(qa), _ptr(ka), _ptr(va), _ptr(out), B, H_q, H_kv, S_q, S_k, d_h, int(d_rope), int(window),
            int(q_pos0), float(rope_base), 1 if causal else 0, rows_ptr, n_rows,
            int(threads or default_threads()), ctypes.byref(opts))
    if rc != 0:
        raise ValueError("oracle_mla_attn failed with code %d" % rc)
    return out
