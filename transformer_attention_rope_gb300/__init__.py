"""GB300-native APEX-1 attention block: RoPE + GQA + causal/sliding-window SDPA.

This package is a thin ctypes binding over the C ABI declared in
``include/apex_attn.h`` (``_build/libapex_attn.so``).  It only marshals
arguments: every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback -- if the library is missing, every call raises.

Raw C-ABI names (pointers and sizes):
    apex_attn_fwd, apex_attn_decode, apex_attn_decode_noalloc, apex_attn_decode_workspace_bytes,
    apex_attn_rope_reserve, apex_attn_device_status, apex_attn_status_string,
    apex_attn_fwd_ex, apex_attn_fwd_ws, apex_attn_fwd_workspace_bytes, apex_attn_decode_ex, apex_attn_rope_keys,
    apex_attn_mla_fwd, apex_attn_mla_fwd_ws, apex_attn_mla_fwd_workspace_bytes, apex_attn_mla_decode,
    apex_attn_mla_rope_keys (with an Options struct)
Tensor conveniences (torch, bf16, contiguous, on the current CUDA device):
    fwd(q, k, v, ...), decode(q, k_cache, v_cache, q_pos, ...), rope_keys(k, ...), mla_fwd(q, k, v, d_r, ...),
    mla_decode(q, k_cache, v_cache, q_pos, d_r, ...), mla_rope_keys(k, d_r, ...)
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ApexError", "library_path", "load_library", "apex_attn_fwd", "apex_attn_decode", "apex_attn_decode_noalloc",
    "apex_attn_decode_workspace_bytes", "apex_attn_rope_reserve", "apex_attn_device_status",
    "apex_attn_status_string", "apex_attn_fwd_ex", "apex_attn_fwd_ws", "apex_attn_fwd_workspace_bytes",
    "apex_attn_decode_ex", "apex_attn_rope_keys", "fwd_workspace_bytes",
    "apex_attn_mla_fwd", "apex_attn_mla_fwd_ws", "apex_attn_mla_fwd_workspace_bytes", "apex_attn_mla_decode",
    "apex_attn_mla_rope_keys", "apex_attn_selftest_wait_timeout", "Options", "fwd", "decode",
    "decode_workspace_bytes", "mla_fwd_workspace_bytes",
    "rope_keys", "mla_fwd", "mla_decode", "mla_rope_keys",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libapex_attn.so")
_lock = threading.Lock()
_lib = None

APEX_OK = 0
_STATUS_NAMES = {0: "APEX_OK", 1: "APEX_ERR_INVALID_ARG", 2: "APEX_ERR_UNSUPPORTED", 3: "APEX_ERR_CUDA",
                 4: "APEX_ERR_NO_MEMORY", 5: "APEX_ERR_DEVICE_TIMEOUT"}


class Options(ctypes.Structure):
    """apex_attn_options of include/apex_attn.h (all zeros: the plain block)."""
    _fields_ = [("window", ctypes.c_int), ("q_pos", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("yarn_scale", ctypes.c_float), ("yarn_beta_fast", ctypes.c_float),
                ("yarn_beta_slow", ctypes.c_float), ("prefix_len", ctypes.c_int), ("keys_prerotated", ctypes.c_int)]


class ApexError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (what, _STATUS_NAMES.get(status, status),
                                                 apex_attn_status_string(status)))


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError("libapex_attn.so is not built (run __graft_entry__.build() or "
                                   "python transformer_attention_rope_gb300/build.py); there is no fallback")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.apex_attn_fwd.argtypes = [vp, vp, vp, vp] + [i32] * 8 + [f32, vp]
            lib.apex_attn_fwd.restype = i32
            lib.apex_attn_decode.argtypes = [vp, vp, vp, vp] + [i32] * 7 + [f32, vp, sz, vp]
            lib.apex_attn_decode.restype = i32
            lib.apex_attn_decode_noalloc.argtypes = [vp, vp, vp, vp] + [i32] * 7 + [f32, vp]
            lib.apex_attn_decode_noalloc.restype = i32
            op = ctypes.POINTER(Options)
            lib.apex_attn_fwd_ex.argtypes = [vp, vp, vp, vp] + [i32] * 6 + [op, vp]
            lib.apex_attn_fwd_ex.restype = i32
            lib.apex_attn_fwd_ws.argtypes = [vp, vp, vp, vp] + [i32] * 6 + [op, vp, sz, vp]
            lib.apex_attn_fwd_ws.restype = i32
            lib.apex_attn_fwd_workspace_bytes.argtypes = [i32] * 6 + [op]
            lib.apex_attn_fwd_workspace_bytes.restype = sz
            lib.apex_attn_mla_fwd.argtypes = [vp, vp, vp, vp] + [i32] * 7 + [op, vp]
            lib.apex_attn_mla_fwd.restype = i32
            lib.apex_attn_mla_fwd_ws.argtypes = [vp, vp, vp, vp] + [i32] * 7 + [op, vp, sz, vp]
            lib.apex_attn_mla_fwd_ws.restype = i32
            lib.apex_attn_mla_fwd_workspace_bytes.argtypes = [i32] * 7 + [op]
            lib.apex_attn_mla_fwd_workspace_bytes.restype = sz
            lib.apex_attn_mla_decode.argtypes = [vp, vp, vp, vp] + [i32] * 6 + [op, vp, sz, vp]
            lib.apex_attn_mla_decode.restype = i32
            lib.apex_attn_decode_ex.argtypes = [vp, vp, vp, vp] + [i32] * 5 + [op, vp, sz, vp]
            lib.apex_attn_decode_ex.restype = i32
            lib.apex_attn_rope_keys.argtypes = [vp, vp] + [i32] * 4 + [ctypes.c_longlong] * 2 + [op, vp]
            lib.apex_attn_rope_keys.restype = i32
            lib.apex_attn_mla_rope_keys.argtypes = [vp, vp] + [i32] * 5 + [ctypes.c_longlong] * 2 + [op, vp]
            lib.apex_attn_mla_rope_keys.restype = i32
            lib.apex_attn_decode_workspace_bytes.argtypes = [i32] * 5
            lib.apex_attn_decode_workspace_bytes.restype = sz
            lib.apex_attn_rope_reserve.argtypes = [i32, i32, f32]
            lib.apex_attn_rope_reserve.restype = i32
            lib.apex_attn_selftest_wait_timeout.argtypes = [i32, vp]
            lib.apex_attn_selftest_wait_timeout.restype = i32
            lib.apex_attn_device_status.argtypes = []
            lib.apex_attn_device_status.restype = i32
            lib.apex_attn_status_string.argtypes = [i32]
            lib.apex_attn_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


# ------------------------------------------------------------------ raw C ABI
def apex_attn_fwd(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, window, q_pos0, rope_base, stream) -> int:
    return load_library().apex_attn_fwd(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, window, q_pos0,
                                        rope_base, stream)


def apex_attn_decode(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, window, q_pos, rope_base,
                     workspace, workspace_bytes, stream) -> int:
    return load_library().apex_attn_decode(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, window, q_pos,
                                           rope_base, workspace, workspace_bytes, stream)


def apex_attn_decode_noalloc(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, window, q_pos, rope_base,
                             stream) -> int:
    return load_library().apex_attn_decode_noalloc(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, window,
                                                   q_pos, rope_base, stream)


def apex_attn_fwd_ex(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, opt, stream) -> int:
    return load_library().apex_attn_fwd_ex(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h,
                                           ctypes.byref(opt) if opt is not None else None, stream)


def apex_attn_fwd_ws(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, opt, workspace, workspace_bytes, stream) -> int:
    return load_library().apex_attn_fwd_ws(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h,
                                           ctypes.byref(opt) if opt is not None else None, workspace,
                                           workspace_bytes, stream)


def apex_attn_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, opt) -> int:
    return load_library().apex_attn_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h,
                                                        ctypes.byref(opt) if opt is not None else None)


def apex_attn_mla_fwd(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_r, opt, stream) -> int:
    return load_library().apex_attn_mla_fwd(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_r,
                                            ctypes.byref(opt) if opt is not None else None, stream)


def apex_attn_mla_fwd_ws(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_r, opt, workspace, workspace_bytes,
                         stream) -> int:
    return load_library().apex_attn_mla_fwd_ws(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_r,
                                               ctypes.byref(opt) if opt is not None else None, workspace,
                                               workspace_bytes, stream)


def apex_attn_mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, d_r, opt) -> int:
    return load_library().apex_attn_mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, d_r,
                                                            ctypes.byref(opt) if opt is not None else None)


def apex_attn_mla_decode(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, d_r, opt, workspace,
                         workspace_bytes, stream) -> int:
    return load_library().apex_attn_mla_decode(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, d_r,
                                               ctypes.byref(opt) if opt is not None else None, workspace,
                                               workspace_bytes, stream)


def apex_attn_decode_ex(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, opt, workspace, workspace_bytes,
                        stream) -> int:
    return load_library().apex_attn_decode_ex(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h,
                                              ctypes.byref(opt) if opt is not None else None, workspace,
                                              workspace_bytes, stream)


def apex_attn_rope_keys(k_in, k_out, n_heads, n_pos, d_h, pos0, in_head_stride, out_head_stride, opt,
                        stream) -> int:
    return load_library().apex_attn_rope_keys(k_in, k_out, n_heads, n_pos, d_h, pos0, in_head_stride,
                                              out_head_stride, ctypes.byref(opt) if opt is not None else None,
                                              stream)


def apex_attn_mla_rope_keys(k_in, k_out, n_heads, n_pos, d_h, d_r, pos0, in_head_stride, out_head_stride, opt,
                            stream) -> int:
    return load_library().apex_attn_mla_rope_keys(k_in, k_out, n_heads, n_pos, d_h, d_r, pos0, in_head_stride,
                                                  out_head_stride, ctypes.byref(opt) if opt is not None else None,
                                                  stream)


def apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_h) -> int:
    return load_library().apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_h)


def apex_attn_rope_reserve(max_pos, d_h, rope_base) -> int:
    return load_library().apex_attn_rope_reserve(max_pos, d_h, rope_base)


def apex_attn_selftest_wait_timeout(timeout_ms, stream) -> int:
    return load_library().apex_attn_selftest_wait_timeout(timeout_ms, stream)


def apex_attn_device_status() -> int:
    return load_library().apex_attn_device_status()


def apex_attn_status_string(status: int) -> str:
    return load_library().apex_attn_status_string(int(status)).decode()


# ------------------------------------------------------------------ torch conveniences
def _check(t, name, ndim):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError("%s must be a CUDA bf16 tensor" % name)
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %d-D tensor" % (name, ndim))


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _options(window=0, q_pos=0, rope_base=10000.0, yarn_scale=1.0, yarn_beta_fast=32.0, yarn_beta_slow=1.0,
             prefix_len=0, keys_prerotated=False) -> Options:
    return Options(int(window), int(q_pos), float(rope_base), float(yarn_scale), float(yarn_beta_fast),
                   float(yarn_beta_slow), int(prefix_len), 1 if keys_prerotated else 0)


def fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, *, window: int = 0, q_pos0: int = 0,
                        rope_base: float = 10000.0, yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0,
                        yarn_beta_slow: float = 1.0, prefix_len: int = 0, keys_prerotated: bool = False) -> int:
    """Workspace bytes a prefill with these arguments uses (0: none; see apex_attn_fwd_workspace_bytes)."""
    opt = _options(window, q_pos0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                   keys_prerotated)
    return int(apex_attn_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, opt))


def fwd(q, k, v, *, window: int = 0, q_pos0: int = 0, rope_base: float = 10000.0, out=None, stream=None,
        yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0, prefix_len: int = 0,
        keys_prerotated: bool = False, workspace=None):
    """Prefill. q [B,H_q,S_q,d], k/v [B,H_kv,S_k,d] (bf16, CUDA) -> out [B,H_q,S_q,d].

    workspace: None -- when the library would rotate the keys once before the
    prefill (fwd_workspace_bytes > 0), a buffer for them is taken from torch's
    allocator and apex_attn_fwd_ws runs; a uint8 CUDA tensor -- that buffer;
    False -- no workspace (apex_attn_fwd / apex_attn_fwd_ex)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, 4)
    B, H_q, S_q, d = q.shape
    _, H_kv, S_k, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", 4)
    if workspace is None:
        need = fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d, window=window, q_pos0=q_pos0, rope_base=rope_base,
                                   yarn_scale=yarn_scale, yarn_beta_fast=yarn_beta_fast,
                                   yarn_beta_slow=yarn_beta_slow, prefix_len=prefix_len,
                                   keys_prerotated=keys_prerotated)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    plain = yarn_scale <= 1.0 and prefix_len == 0 and not keys_prerotated
    if workspace is not None and workspace is not False:
        opt = _options(window, q_pos0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                       keys_prerotated)
        st = apex_attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv, S_q, S_k,
                              d, opt, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(stream))
    elif plain:
        st = apex_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv, S_q, S_k, d,
                           int(window), int(q_pos0), float(rope_base), _stream_handle(stream))
    else:
        opt = _options(window, q_pos0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                       keys_prerotated)
        st = apex_attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv, S_q, S_k,
                              d, opt, _stream_handle(stream))
    if st != APEX_OK:
        raise ApexError(st, "apex_attn_fwd")
    return out


def mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, d_r, *, window: int = 0, q_pos0: int = 0,
                            rope_base: float = 10000.0, yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0,
                            yarn_beta_slow: float = 1.0, prefix_len: int = 0, keys_prerotated: bool = False) -> int:
    """Workspace bytes a decoupled-RoPE prefill with these arguments uses (0: none; see
    apex_attn_mla_fwd_workspace_bytes)."""
    opt = _options(window, q_pos0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                   keys_prerotated)
    return int(apex_attn_mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, int(d_r), opt))


def mla_fwd(q, k, v, d_r: int, *, window: int = 0, q_pos0: int = 0, rope_base: float = 10000.0, out=None,
            stream=None, yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0,
            prefix_len: int = 0, keys_prerotated: bool = False, workspace=None):
    """Decoupled-RoPE prefill. q [B,H_q,S_q,d_h+d_r], k [B,H_kv,S_k,d_h+d_r], v [B,H_kv,S_k,d_h]
    (bf16, CUDA; rows [content | rope part]) -> out [B,H_q,S_q,d_h].

    workspace: None -- a buffer from torch's allocator when the library would rotate
    the keys' rope parts once before the prefill (mla_fwd_workspace_bytes > 0); a
    uint8 CUDA tensor -- that buffer; False -- no workspace (apex_attn_mla_fwd)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, 4)
    B, H_q, S_q, d_qk = q.shape
    _, H_kv, S_k, d_h = v.shape
    if d_qk != d_h + d_r or k.shape[-1] != d_qk:
        raise ValueError("q / k rows must hold d_h + d_r entries")
    if out is None:
        out = torch.empty((B, H_q, S_q, d_h), dtype=torch.bfloat16, device=q.device)
    _check(out, "out", 4)
    opt = _options(window, q_pos0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                   keys_prerotated)
    if workspace is None:
        need = int(apex_attn_mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, int(d_r), opt))
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace is not None and workspace is not False:
        st = apex_attn_mla_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv, S_q,
                                  S_k, d_h, int(d_r), opt, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream_handle(stream))
        name = "apex_attn_mla_fwd_ws"
    else:
        st = apex_attn_mla_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv, S_q, S_k,
                               d_h, int(d_r), opt, _stream_handle(stream))
        name = "apex_attn_mla_fwd"
    if st != APEX_OK:
        raise ApexError(st, name)
    return out


def decode_workspace_bytes(B, H_q, H_kv, S_k, d_h) -> int:
    return int(apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_h))


def decode(q, k_cache, v_cache, q_pos: int, *, window: int = 0, rope_base: float = 10000.0, out=None,
           workspace=None, stream=None, yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0,
           yarn_beta_slow: float = 1.0, prefix_len: int = 0, keys_prerotated: bool = False):
    """Decode. q [B,H_q,1,d], caches [B,H_kv,S_k,d] (bf16, CUDA) -> out [B,H_q,1,d]."""
    import torch
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, 4)
    B, H_q, one, d = q.shape
    _, H_kv, S_k, _ = k_cache.shape
    if one != 1:
        raise ValueError("decode takes one query per sequence")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", 4)
    need = decode_workspace_bytes(B, H_q, H_kv, S_k, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    plain = yarn_scale <= 1.0 and prefix_len == 0 and not keys_prerotated
    if plain:
        st = apex_attn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), B, H_q, H_kv,
                              S_k, d, int(window), int(q_pos), float(rope_base), workspace.data_ptr(), ws_bytes,
                              _stream_handle(stream))
    else:
        opt = _options(window, q_pos, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                       keys_prerotated)
        st = apex_attn_decode_ex(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), B, H_q,
                                 H_kv, S_k, d, opt, workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != APEX_OK:
        raise ApexError(st, "apex_attn_decode")
    return out


def mla_decode(q, k_cache, v_cache, q_pos: int, d_r: int, *, window: int = 0, rope_base: float = 10000.0,
               out=None, workspace=None, stream=None, yarn_scale: float = 1.0, yarn_beta_fast: float = 32.0,
               yarn_beta_slow: float = 1.0, prefix_len: int = 0, keys_prerotated: bool = False):
    """Decoupled-RoPE decode. q [B,H_q,1,d_h+d_r], k_cache [B,H_kv,S_k,d_h+d_r], v_cache [B,H_kv,S_k,d_h]
    (bf16, CUDA; rows [content | rope part]) -> out [B,H_q,1,d_h]."""
    import torch
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, 4)
    B, H_q, one, d_qk = q.shape
    _, H_kv, S_k, d_h = v_cache.shape
    if one != 1:
        raise ValueError("decode takes one query per sequence")
    if d_qk != d_h + d_r or k_cache.shape[-1] != d_qk:
        raise ValueError("q / k_cache rows must hold d_h + d_r entries")
    if out is None:
        out = torch.empty((B, H_q, 1, d_h), dtype=torch.bfloat16, device=q.device)
    _check(out, "out", 4)
    need = decode_workspace_bytes(B, H_q, H_kv, S_k, d_h)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    opt = _options(window, q_pos, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow, prefix_len,
                   keys_prerotated)
    st = apex_attn_mla_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), B, H_q, H_kv,
                              S_k, d_h, int(d_r), opt, workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != APEX_OK:
        raise ApexError(st, "apex_attn_mla_decode")
    return out


def rope_keys(k, *, pos0: int = 0, out=None, rope_base: float = 10000.0, yarn_scale: float = 1.0,
              yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0, stream=None):
    """Rotate keys k [B,H,S,d] (bf16, CUDA) to positions pos0 + s: out = RoPE(k) (pre-rotated cache)."""
    import torch
    _check(k, "k", 4)
    B, H, S, d = k.shape
    if out is None:
        out = torch.empty_like(k)
    _check(out, "out", 4)
    if out.shape != k.shape:
        raise ValueError("out must have the shape of k")
    opt = _options(0, 0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow)
    st = apex_attn_rope_keys(k.data_ptr(), out.data_ptr(), B * H, S, d, int(pos0), S * d, S * d, opt,
                             _stream_handle(stream))
    if st != APEX_OK:
        raise ApexError(st, "apex_attn_rope_keys")
    return out


def mla_rope_keys(k, d_r: int, *, pos0: int = 0, out=None, rope_base: float = 10000.0, yarn_scale: float = 1.0,
                  yarn_beta_fast: float = 32.0, yarn_beta_slow: float = 1.0, stream=None):
    """Decoupled-RoPE key rows k [B,H,S,d_h+d_r] (bf16, CUDA; [content | rope part]) with the
    rope part rotated to positions pos0 + s and the content part copied (pre-rotated cache)."""
    import torch
    _check(k, "k", 4)
    B, H, S, d = k.shape
    if out is None:
        out = torch.empty_like(k)
    _check(out, "out", 4)
    if out.shape != k.shape:
        raise ValueError("out must have the shape of k")
    opt = _options(0, 0, rope_base, yarn_scale, yarn_beta_fast, yarn_beta_slow)
    st = apex_attn_mla_rope_keys(k.data_ptr(), out.data_ptr(), B * H, S, d - int(d_r), int(d_r), int(pos0), S * d,
                                 S * d, opt, _stream_handle(stream))
    if st != APEX_OK:
        raise ApexError(st, "apex_attn_mla_rope_keys")
    return out
