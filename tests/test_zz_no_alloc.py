"""apex_attn_decode_noalloc -- the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory when they call (an engine
whose memory pool owns the whole device, a plugin interface without a
workspace slot, a loop that cannot take an allocation's synchronisation): its
scratch and RoPE table live in the library's own static device arrays.  The
test calls it through the C ABI twice in a row and checks each result against
the fp64 oracle (element by element, at the parity tolerance) and against
apex_attn_decode (which takes a caller-allocated workspace), and checks that
the two calls left free device memory unchanged.  The cases reach the limits
of the static arrays: the last row of the 32768-position RoPE table, and a
batch of query heads so large that the 16 MiB scratch, not the split-count
model, decides how many KV splits run.

This file is collected last on purpose: it must pass both alone in a fresh
process (where its first call also does the one-time set-up) and after the
other GPU tests.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3
SCRATCH_BYTES = 16 << 20


def _call_noalloc(q, k, v, out, q_pos, window):
    B, H_q, _, d = q.shape
    _, H_kv, S_k, _ = k.shape
    return apex.apex_attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H_q, H_kv,
                                         S_k, d, window, q_pos, 10000.0, torch.cuda.current_stream().cuda_stream)


def _close(a, b):
    e = (torch.as_tensor(a).double().cpu() - torch.as_tensor(b).double().cpu()).abs()
    return float(e.max()), float(e.mean())


CASES = [  # B, H_q, H_kv, S_k, d, window, q_pos
    (8, 32, 8, 4096, 128, 0, 4095),
    (3, 16, 4, 777, 64, 100, 700),
    # the whole static table: the query at its last row, every key visible
    (2, 8, 2, 32768, 128, 0, 32767),
    # 512 query heads at d 128: 64 splits would need 512 * 64 * 520 B = 17 MB of
    # partials, so the scratch caps the split count below what the model picks
    (16, 32, 8, 8192, 128, 0, 8191),
]


@pytest.mark.parametrize("B,H_q,H_kv,S_k,d,window,q_pos", CASES)
def test_noalloc_decode_matches_oracle_and_decode_twice(B, H_q, H_kv, S_k, d, window, q_pos):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    q_h = inputs.normal_bf16((B, H_q, 1, d), 300 + S_k, 0)
    k_h = inputs.normal_bf16((B, H_kv, S_k, d), 300 + S_k, 1)
    v_h = inputs.normal_bf16((B, H_kv, S_k, d), 300 + S_k, 2)
    ref = oracle.attn(q_h, k_h, v_h, window=window, q_pos0=q_pos)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    alloc = apex.decode(q, k, v, q_pos, window=window)
    warm = torch.empty_like(q)
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    # the first call on a device may do the one-time set-up; measure after it
    assert _call_noalloc(q, k, v, warm, q_pos, window) == 0
    torch.cuda.synchronize()
    # between the two readings only the library runs (no torch kernels, which
    # could load modules of their own)
    free_before = torch.cuda.mem_get_info(dev)[0]
    for out in outs:
        assert _call_noalloc(q, k, v, out, q_pos, window) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free_before
    assert apex.apex_attn_device_status() == 0
    for out in outs:
        mx, mean = _close(out, ref)
        assert np.isfinite(mx) and mx <= MAX_ERR and mean <= MEAN_ERR, ("vs oracle", mx, mean)
        mx, mean = _close(out, alloc)
        assert np.isfinite(mx) and mx <= MAX_ERR and mean <= MEAN_ERR, ("vs apex_attn_decode", mx, mean)


def test_noalloc_case_list_reaches_the_scratch_limit():
    """The last case needs more partials at the split-count cap than the scratch
    holds (so the scratch, not the cost model's cap, limits it)."""
    B, H_q, H_kv, S_k, d, _, _ = CASES[-1]
    units = B * H_kv
    n_stages = S_k // 64 + 1
    cap = min(32768 // units, n_stages)
    assert B * H_q * cap * (4 * d + 8) > SCRATCH_BYTES


def test_noalloc_rejects_beyond_its_limits():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fake = 1 << 20
    # S_k above the static RoPE table's 32768 positions
    assert apex.apex_attn_decode_noalloc(fake, fake, fake, fake, 1, 8, 2, 40000, 128, 0, 39999, 10000.0, None) == 2
    # one split of partials for B * H_q query heads would not fit the 16 MiB scratch
    assert apex.apex_attn_decode_noalloc(fake, fake, fake, fake, 4096, 16, 16, 1024, 128, 0, 1023, 10000.0,
                                         None) == 2
