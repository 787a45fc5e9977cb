"""The C-ABI library: it builds for sm_103a, exports every declared symbol, and
rejects bad arguments on the host before touching the GPU.  CPU only."""
import ctypes
import os
import re

import pytest

import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "apex_attn.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return apex.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(apex_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("apex_attn_fwd", "apex_attn_decode", "apex_attn_decode_workspace_bytes",
              "apex_attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert hasattr(apex, name), "binding lacks " + name


def test_library_is_in_tree(lib):
    assert os.path.dirname(apex.library_path()).startswith(ROOT)
    assert os.path.exists(apex.library_path())


def test_status_strings(lib):
    for s in range(6):
        assert isinstance(apex.apex_attn_status_string(s), str)
    assert apex.apex_attn_status_string(99) == "unknown status"


# Each call below is rejected by the host-side checks, before any CUDA call.
FAKE = 1 << 20  # a 16-byte aligned non-null address that is never dereferenced


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, 1, 4, 2, 8, 8, 64, 0, 0, 10000.0), 1),        # null q
    ((FAKE + 2, FAKE, FAKE, FAKE, 1, 4, 2, 8, 8, 64, 0, 0, 10000.0), 1),  # misaligned q
    ((FAKE, FAKE, FAKE, FAKE, 1, 3, 2, 8, 8, 64, 0, 0, 10000.0), 1),     # H_q % H_kv != 0
    ((FAKE, FAKE, FAKE, FAKE, 0, 4, 2, 8, 8, 64, 0, 0, 10000.0), 1),     # B = 0
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 8, 8, 96, 0, 0, 10000.0), 2),     # d_h = 96
    ((FAKE, FAKE, FAKE, FAKE, 1, 96, 2, 8, 8, 64, 0, 0, 10000.0), 2),    # G = 48
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 9, 8, 64, 0, 0, 10000.0), 1),     # S_q > S_k
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 4, 8, 64, 0, 5, 10000.0), 1),     # q_pos0 + S_q > S_k
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 4, 8, 64, 0, -1, 10000.0), 1),    # negative q_pos0
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 4, 8, 64, 0, 0, 0.0), 1),         # rope base 0
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 4, 8, 64, 0, 0, float("nan")), 1),
])
def test_fwd_rejects(lib, args, code):
    assert apex.apex_attn_fwd(*args, None) == code


# empty and oversized problems: rejected on the host, nothing launched
@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 0, 8, 64, 0, 0, 10000.0), 1),            # no query rows
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 0, 0, 64, 0, 0, 10000.0), 1),            # no keys
    ((FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 8, (1 << 24) + 1, 64, 0, 0, 10000.0), 2),  # beyond 2^24 keys
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 0, 8, 8, 64, 0, 0, 10000.0), 1),            # no heads
])
def test_fwd_rejects_empty_and_oversized(lib, args, code):
    assert apex.apex_attn_fwd(*args, None) == code


def test_decode_rejects_empty_and_oversized(lib):
    # no keys; beyond 2^24 keys
    assert apex.apex_attn_decode(FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 0, 64, 0, 0, 10000.0, FAKE, 1 << 30, None) == 1
    big = (1 << 24) + 1
    assert apex.apex_attn_decode(FAKE, FAKE, FAKE, FAKE, 1, 8, 2, big, 64, 0, big - 1, 10000.0, FAKE, 1 << 30,
                                 None) == 2
    assert apex.apex_attn_decode_workspace_bytes(1, 8, 2, big, 64) == 0
    assert apex.fwd_workspace_bytes(1, 8, 2, 8, big, 128) == 0


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 63, 10000.0, FAKE, 1 << 30), 1),
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 64, 10000.0, FAKE, 1 << 30), 1),   # q_pos >= S_k
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, -1, 10000.0, FAKE, 1 << 30), 1),
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 63, 10000.0, FAKE, 16), 1),        # workspace too small
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 63, 10000.0, 0, 1 << 30), 1),      # null workspace
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 80, 0, 63, 10000.0, FAKE, 1 << 30), 2),   # d_h = 80
])
def test_decode_rejects(lib, args, code):
    assert apex.apex_attn_decode(*args, None) == code


def test_decode_workspace_bytes(lib):
    n = apex.apex_attn_decode_workspace_bytes(64, 32, 8, 32768, 128)
    assert n > 0 and n % 16 == 0
    # (max, sum) pair + d_h floats for each of at most 64 splits per query head
    assert n <= 64 * 32 * 64 * (128 * 4 + 8) + 16
    assert apex.apex_attn_decode_workspace_bytes(1, 3, 2, 10, 64) == 0
    assert apex.apex_attn_decode_workspace_bytes(1, 4, 2, 10, 96) == 0


def test_rope_reserve_rejects(lib):
    assert apex.apex_attn_rope_reserve(0, 128, 10000.0) == 1
    assert apex.apex_attn_rope_reserve(100, 96, 10000.0) == 2
    assert apex.apex_attn_rope_reserve(100, 128, -1.0) == 1


def _opt(**kw):
    o = dict(window=0, q_pos=0, rope_base=10000.0, yarn_scale=1.0, yarn_beta_fast=32.0, yarn_beta_slow=1.0,
             prefix_len=0, keys_prerotated=False)
    o.update(kw)
    return apex._options(**o)


# prefill with options: (B, H_q, H_kv, S_q, S_k, d_h), options, expected status
@pytest.mark.parametrize("shape,opt,code", [
    ((1, 4, 2, 8, 8, 64), None, 1),                                  # no options
    ((1, 4, 2, 8, 8, 64), dict(prefix_len=-1), 1),
    ((1, 4, 2, 8, 8, 64), dict(prefix_len=9), 1),                    # prefix beyond the keys
    ((1, 4, 2, 8, 8, 64), dict(q_pos=1), 1),                         # q_pos0 + S_q > S_k
    ((1, 4, 2, 8, 8, 64), dict(rope_base=float("inf")), 1),
    ((1, 4, 2, 8, 8, 64), dict(yarn_scale=float("nan")), 1),
    ((1, 4, 2, 8, 8, 64), dict(yarn_scale=4.0, yarn_beta_fast=-1.0), 1),
    ((1, 4, 2, 8, 8, 64), dict(yarn_scale=4.0, yarn_beta_slow=float("inf")), 1),
    ((1, 4, 2, 8, 8, 96), {}, 2),
])
def test_fwd_ex_rejects(lib, shape, opt, code):
    o = None if opt is None else _opt(**opt)
    assert apex.apex_attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, *shape, o, None) == code


# prefill with a workspace: (B, H_q, H_kv, S_q, S_k, d_h), options, workspace, bytes, expected status
@pytest.mark.parametrize("shape,opt,ws,nbytes,code", [
    ((1, 4, 2, 8, 8, 128), None, FAKE, 1 << 20, 1),                 # no options
    ((1, 4, 2, 8, 8, 128), {}, FAKE + 8, 1 << 20, 1),               # misaligned workspace
    ((1, 128, 8, 8192, 8192, 128), {}, FAKE, 8 * 8192 * 128 * 2 - 16, 1),  # one row short of the keys
    ((1, 4, 2, 8, 8, 128), dict(q_pos=1), FAKE, 1 << 20, 1),        # q_pos0 + S_q > S_k
    ((1, 4, 2, 8, 8, 96), {}, FAKE, 1 << 20, 2),                    # d_h = 96
    ((1, 3, 2, 8, 8, 128), {}, FAKE, 1 << 20, 1),                   # H_q % H_kv != 0
])
def test_fwd_ws_rejects(lib, shape, opt, ws, nbytes, code):
    o = None if opt is None else _opt(**opt)
    assert apex.apex_attn_fwd_ws(FAKE, FAKE, FAKE, FAKE, *shape, o, ws, nbytes, None) == code


def test_fwd_workspace_bytes(lib):
    # one bf16 copy of the keys where the pass pays (long windows, wide head groups) ...
    for shape, window in (((4, 32, 8, 4096, 4096, 128), 1024), ((1, 128, 8, 8192, 8192, 128), 0),
                          ((1, 32, 8, 65536, 65536, 128), 4096)):
        B, H_q, H_kv, S_q, S_k, d = shape
        assert apex.fwd_workspace_bytes(*shape, window=window) == B * H_kv * S_k * d * 2
    # ... also on the single-CTA kernel (d_h = 64), ...
    assert apex.fwd_workspace_bytes(1, 128, 8, 8192, 8192, 64) == 8 * 8192 * 64 * 2
    # ... none for small problems, pre-rotated keys or bad sizes
    assert apex.fwd_workspace_bytes(1, 4, 2, 256, 256, 128) == 0
    assert apex.fwd_workspace_bytes(1, 4, 2, 128, 128, 64) == 0          # the tiny workload
    assert apex.fwd_workspace_bytes(4, 32, 8, 4096, 4096, 128, window=1024, keys_prerotated=True) == 0
    assert apex.fwd_workspace_bytes(1, 3, 2, 4096, 4096, 128) == 0
    assert apex.fwd_workspace_bytes(1, 4, 2, 4096, 4000, 128) == 0   # S_q > S_k
    assert apex.apex_attn_fwd_workspace_bytes(4, 32, 8, 4096, 4096, 128, None) == 0


# decoupled-RoPE prefill: (B, H_q, H_kv, S_q, S_k, d_h, d_r), expected status
@pytest.mark.parametrize("shape,code", [
    ((1, 4, 2, 8, 8, 128, 0), 1),
    ((1, 4, 2, 8, 8, 128, 63), 1),       # odd rope part
    ((1, 4, 2, 8, 8, 64, 64), 2),        # only d_h = 128 with d_r = 64 is built
    ((1, 4, 2, 8, 8, 128, 32), 2),
    ((1, 3, 2, 8, 8, 128, 64), 1),       # H_q % H_kv != 0
    ((1, 4, 2, 9, 8, 128, 64), 1),       # S_q > S_k
])
def test_mla_fwd_rejects(lib, shape, code):
    assert apex.apex_attn_mla_fwd(FAKE, FAKE, FAKE, FAKE, *shape, _opt(), None) == code
    assert apex.apex_attn_mla_fwd(0, FAKE, FAKE, FAKE, *shape, _opt(), None) == 1


# decoupled-RoPE prefill with a workspace: (B, H_q, H_kv, S_q, S_k, d_h, d_r), options, workspace, bytes, status
MLA_KEYS = 8 * 8192 * 192 * 2  # one bf16 copy of the key rows of B1 H_kv8 S8192 [128 | 64]


@pytest.mark.parametrize("shape,opt,ws,nbytes,code", [
    ((1, 4, 2, 8, 8, 128, 64), None, FAKE, 1 << 20, 1),                 # no options
    ((1, 128, 8, 8192, 8192, 128, 64), {}, FAKE + 8, MLA_KEYS, 1),      # misaligned workspace
    ((1, 128, 8, 8192, 8192, 128, 64), {}, FAKE, MLA_KEYS - 16, 1),     # one row short of the keys
    ((1, 4, 2, 8, 8, 128, 63), {}, FAKE, 1 << 20, 1),                   # odd rope part
    ((1, 4, 2, 8, 8, 64, 64), {}, FAKE, 1 << 20, 2),                    # only d_h = 128 with d_r = 64
    ((1, 4, 2, 9, 8, 128, 64), {}, FAKE, 1 << 20, 1),                   # S_q > S_k
])
def test_mla_fwd_ws_rejects(lib, shape, opt, ws, nbytes, code):
    o = None if opt is None else _opt(**opt)
    assert apex.apex_attn_mla_fwd_ws(FAKE, FAKE, FAKE, FAKE, *shape, o, ws, nbytes, None) == code


def test_mla_fwd_workspace_bytes(lib):
    # one bf16 copy of the key rows where the pass pays (wide head groups, long windows) ...
    assert apex.mla_fwd_workspace_bytes(1, 128, 8, 8192, 8192, 128, 64) == MLA_KEYS
    assert apex.mla_fwd_workspace_bytes(1, 32, 8, 65536, 65536, 128, 64, window=4096) == 8 * 65536 * 192 * 2
    # ... none where each key tile is visited a few times only (the rope part is a
    # third of the row, so the in-kernel rotation costs less than for plain rows),
    # for pre-rotated keys, and for bad or unsupported sizes
    assert apex.mla_fwd_workspace_bytes(4, 32, 8, 4096, 4096, 128, 64, window=1024) == 0
    assert apex.mla_fwd_workspace_bytes(1, 4, 2, 256, 256, 128, 64) == 0
    assert apex.mla_fwd_workspace_bytes(1, 128, 8, 8192, 8192, 128, 64, keys_prerotated=True) == 0
    assert apex.mla_fwd_workspace_bytes(1, 128, 8, 8192, 8192, 64, 64) == 0
    assert apex.mla_fwd_workspace_bytes(1, 128, 8, 8192, 8192, 128, 0) == 0
    assert apex.mla_fwd_workspace_bytes(1, 128, 8, 8192, 8000, 128, 64) == 0   # S_q > S_k
    assert apex.apex_attn_mla_fwd_workspace_bytes(1, 128, 8, 8192, 8192, 128, 64, None) == 0


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, 2, 8, 128, 0, 0, 1536, 1536), 1),        # no rope part
    ((FAKE, FAKE, 2, 8, 128, 63, 0, 1528, 1528), 1),       # odd rope part
    ((FAKE, FAKE, 2, 8, 64, 64, 0, 1024, 1024), 2),        # only d_h = 128 with d_r = 64
    ((FAKE, FAKE, 2, 8, 128, 32, 0, 1280, 1280), 2),
    ((FAKE, FAKE, 0, 8, 128, 64, 0, 1536, 1536), 1),       # no heads
    ((FAKE, FAKE, 2, 8, 128, 64, -1, 1536, 1536), 1),      # negative first position
    ((FAKE, FAKE, 2, 8, 128, 64, 0, 1024, 1536), 1),       # input heads overlap (stride < 8 rows)
    ((FAKE + 8, FAKE, 2, 8, 128, 64, 0, 1536, 1536), 1),   # misaligned input
])
def test_mla_rope_keys_rejects(lib, args, code):
    assert apex.apex_attn_mla_rope_keys(*args, _opt(), None) == code
    assert apex.apex_attn_mla_rope_keys(FAKE, FAKE, 2, 8, 128, 64, 0, 1536, 1536, None, None) == 1


# decodes with options: (B, H_q, H_kv, S_k, d_h), options, workspace bytes, expected status
@pytest.mark.parametrize("shape,opt,ws,code", [
    ((2, 8, 2, 64, 64), None, 1 << 30, 1),
    ((2, 8, 2, 64, 64), dict(q_pos=64), 1 << 30, 1),      # q_pos >= S_k
    ((2, 8, 2, 64, 64), dict(q_pos=63, prefix_len=65), 1 << 30, 1),
    ((2, 8, 2, 64, 64), dict(q_pos=63), 16, 1),           # workspace too small
    ((2, 8, 2, 64, 96), dict(q_pos=63), 1 << 30, 2),
])
def test_decode_ex_rejects(lib, shape, opt, ws, code):
    o = None if opt is None else _opt(**opt)
    assert apex.apex_attn_decode_ex(FAKE, FAKE, FAKE, FAKE, *shape, o, FAKE, ws, None) == code


@pytest.mark.parametrize("shape,opt,ws,code", [
    ((2, 8, 2, 64, 128, 64), None, 1 << 30, 1),
    ((2, 8, 2, 64, 128, 65), dict(q_pos=63), 1 << 30, 1),
    ((2, 8, 2, 64, 64, 64), dict(q_pos=63), 1 << 30, 2),
    ((2, 8, 2, 64, 128, 64), dict(q_pos=64), 1 << 30, 1),
    ((2, 8, 2, 64, 128, 64), dict(q_pos=63), 16, 1),
])
def test_mla_decode_rejects(lib, shape, opt, ws, code):
    o = None if opt is None else _opt(**opt)
    assert apex.apex_attn_mla_decode(FAKE, FAKE, FAKE, FAKE, *shape, o, FAKE, ws, None) == code


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, 0, 8, 64, 0, 512, 512), 1),          # no heads
    ((FAKE, FAKE, 2, 8, 64, -1, 512, 512), 1),         # negative first position
    ((FAKE, FAKE, 2, 8, 96, 0, 768, 768), 2),          # d_h = 96
    ((FAKE, FAKE, 2, 8, 64, 0, 256, 512), 1),          # input heads overlap
    ((FAKE, FAKE, 2, 8, 64, 0, 516, 512), 1),          # stride not a multiple of 8 elements
    ((FAKE + 8, FAKE, 2, 8, 64, 0, 512, 512), 1),      # misaligned input
])
def test_rope_keys_rejects(lib, args, code):
    assert apex.apex_attn_rope_keys(*args, _opt(), None) == code
    assert apex.apex_attn_rope_keys(FAKE, FAKE, 2, 8, 64, 0, 512, 512, None, None) == 1


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 63, 10000.0), 1),
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 64, 0, 64, 10000.0), 1),       # q_pos >= S_k
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 65536, 64, 0, 63, 10000.0), 2),    # beyond the static scratch
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 64, 96, 0, 63, 10000.0), 2),
    ((FAKE, FAKE, FAKE, FAKE, 2, 6, 2, 64, 64, 0, 63, 10000.0), 2),       # G = 3
])
def test_decode_noalloc_rejects(lib, args, code):
    assert apex.apex_attn_decode_noalloc(*args, None) == code


def test_selftest_rejects_out_of_range_limits(lib):
    assert apex.apex_attn_selftest_wait_timeout(0, None) == 1
    assert apex.apex_attn_selftest_wait_timeout(5001, None) == 1
