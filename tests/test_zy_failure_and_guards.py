"""GPU checks that no test of the parity suites covers: the bounded mbarrier
wait gives up and reports instead of hanging (on a wait that nothing can
complete), the context stays usable afterwards, and no kernel writes outside
its output or workspace (guard regions with a known pattern around them)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

APEX_ERR_DEVICE_TIMEOUT = 5
GUARD = 4096  # bf16 elements on each side
PATTERN = 0x7FA5  # a NaN bit pattern no kernel writes


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _guarded(shape, dev, dtype=torch.bfloat16):
    """A contiguous tensor of `shape` in the middle of a buffer whose GUARD
    elements on both sides hold PATTERN."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.int16, device=dev)
    return buf, buf[GUARD:GUARD + n].view(dtype).view(*shape)


def _guards_intact(buf):
    torch.cuda.synchronize()
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    return bool(torch.all(g == PATTERN).item())


def test_bounded_wait_times_out_and_reports():
    dev = _dev()
    torch.cuda.synchronize()
    assert apex.apex_attn_device_status() == 0
    st = apex.apex_attn_selftest_wait_timeout(50, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert apex.apex_attn_device_status() == APEX_ERR_DEVICE_TIMEOUT
    assert apex.apex_attn_device_status() == 0  # reading clears it
    # the context is still usable
    q, k, v = inputs.workload_inputs(inputs.WORKLOADS["tiny"])
    out = apex.fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    e = np.abs(out.double().cpu().numpy() - oracle.attn(q, k, v))
    assert e.max() <= 2e-2 and apex.apex_attn_device_status() == 0


def test_selftest_rejects_bad_timeouts():
    _dev()
    s = torch.cuda.current_stream().cuda_stream
    assert apex.apex_attn_selftest_wait_timeout(0, s) == 1
    assert apex.apex_attn_selftest_wait_timeout(6000, s) == 1


@pytest.mark.parametrize("kernel,d,B,H_q,H_kv,S,window", [
    ("single", 128, 2, 8, 2, 333, 0),
    ("single", 64, 1, 16, 1, 257, 100),
    ("pair", 128, 1, 8, 2, 333, 64),
    ("mla", 128, 1, 8, 2, 333, 0),
])
def test_prefill_writes_only_its_output(monkeypatch, kernel, d, B, H_q, H_kv, S, window):
    dev = _dev()
    monkeypatch.setenv("APEX_ATTN_PREFILL", "pair" if kernel == "pair" else "single")
    d_r = 64 if kernel == "mla" else 0
    q, k, v = [t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 3000 + S, d_r=d_r)]
    buf, out = _guarded((B, H_q, S, d), dev)
    if kernel == "mla":
        apex.mla_fwd(q, k, v, d_r, window=window, out=out)
    else:
        apex.fwd(q, k, v, window=window, out=out)
    assert _guards_intact(buf)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mla", [False, True])
def test_decode_writes_only_its_output_and_workspace(mla):
    dev = _dev()
    B, H_q, H_kv, S_k, d = 3, 16, 4, 1500, 128
    d_r = 64 if mla else 0
    q, k, v = [t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, 1, S_k, d, 3100, d_r=d_r)]
    obuf, out = _guarded((B, H_q, 1, d), dev)
    nbytes = apex.decode_workspace_bytes(B, H_q, H_kv, S_k, d)
    n_ws = (nbytes + 1) // 2 + 8  # bf16 elements, 16-byte multiple
    n_ws += (-n_ws) % 8
    wbuf, ws = _guarded((n_ws,), dev)
    ws_u8 = ws.view(torch.uint8)
    if mla:
        apex.mla_decode(q, k, v, S_k - 1, d_r, window=700, out=out, workspace=ws_u8)
    else:
        apex.decode(q, k, v, S_k - 1, window=700, out=out, workspace=ws_u8)
    assert _guards_intact(obuf) and _guards_intact(wbuf)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("kernel,d,B,H_q,H_kv,S,window", [
    ("pair", 128, 1, 32, 2, 6000, 0),
    ("single", 64, 2, 8, 2, 8192, 4096),
])
def test_prefill_with_key_pass_writes_only_its_output_and_workspace(monkeypatch, kernel, d, B, H_q, H_kv, S,
                                                                    window):
    """The key-rotation pass writes only inside the workspace, the prefill only
    inside its output (shapes on which the library's cost model runs the pass)."""
    dev = _dev()
    monkeypatch.setenv("APEX_ATTN_PREFILL", kernel)
    nbytes = apex.fwd_workspace_bytes(B, H_q, H_kv, S, S, d, window=window)
    assert nbytes == B * H_kv * S * d * 2
    q, k, v = [t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 3200 + S)]
    obuf, out = _guarded((B, H_q, S, d), dev)
    wbuf, ws = _guarded((nbytes // 2,), dev)
    apex.fwd(q, k, v, window=window, out=out, workspace=ws.view(torch.uint8))
    assert _guards_intact(obuf) and _guards_intact(wbuf)
    assert torch.isfinite(out.float()).all()


def test_mla_prefill_with_key_pass_writes_only_its_output_and_workspace():
    """The same for the decoupled-RoPE prefill: the pass over [content | rope part]
    key rows writes only inside the workspace, the prefill only inside its output."""
    dev = _dev()
    B, H_q, H_kv, S, d, d_r = 1, 32, 2, 6000, 128, 64
    nbytes = apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S, S, d, d_r)
    assert nbytes == B * H_kv * S * (d + d_r) * 2
    q, k, v = [t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 3300 + S, d_r=d_r)]
    obuf, out = _guarded((B, H_q, S, d), dev)
    wbuf, ws = _guarded((nbytes // 2,), dev)
    apex.mla_fwd(q, k, v, d_r, out=out, workspace=ws.view(torch.uint8))
    assert _guards_intact(obuf) and _guards_intact(wbuf)
    assert torch.isfinite(out.float()).all()
    assert apex.apex_attn_device_status() == 0


def test_mla_rope_keys_writes_only_its_rows():
    """apex_attn_mla_rope_keys appending rows into a cache writes only those rows."""
    dev = _dev()
    H, n, d = 3, 200, 192
    src = inputs.normal_bf16((H, n, d), 3301, 1).to(dev)
    obuf, out = _guarded((H, n, d), dev)
    apex.mla_rope_keys(src.view(1, H, n, d), 64, pos0=500, out=out.view(1, H, n, d))
    assert _guards_intact(obuf)
    assert torch.isfinite(out.float()).all()
