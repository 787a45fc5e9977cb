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
