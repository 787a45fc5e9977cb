"""GPU: prefill with a workspace (apex_attn_fwd_ws).  Where the library's cost
model rotates the keys once into the workspace, the workspace must then hold
exactly what apex_attn_rope_keys computes and the output must match the fp64
oracle (and the in-kernel-rotation path within the parity tolerance); where it
does not, the workspace is left untouched and the output is bit-identical to
the call without a workspace.  Tolerance: max |err| <= 2e-2, mean |err| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3
NAN_BF16 = -1  # 0xffff as int16: a NaN bf16 pattern no kernel writes


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _errs(got, ref):
    e = np.abs(torch.as_tensor(got).double().cpu().numpy() - np.asarray(ref, dtype=np.float64))
    return float(e.max()), float(e.mean())


def _ws(B, H_kv, S_k, d, dev):
    n = B * H_kv * S_k * d * 2  # one bf16 copy of the keys
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    ws.view(torch.int16).fill_(NAN_BF16)
    return ws


def _rows(S, step):
    return sorted(set(range(0, S, step)) | set(range(S - 64, S)) | set(range(64)))


# shapes on which each key tile is visited often enough for the pass to run
@pytest.mark.parametrize("B,H_q,H_kv,S,window,opts,d", [
    (2, 8, 2, 8192, 4096, {}, 128),                              # G = 4, sliding window
    (1, 32, 2, 8192, 0, {}, 128),                                # G = 16, causal
    (2, 8, 2, 8192, 4096, dict(yarn_scale=8.0), 128),            # YaRN frequencies in the pass
    (1, 16, 4, 6000, 0, dict(prefix_len=700), 128),              # prefix, ragged last tile
    (2, 8, 2, 8192, 4096, {}, 64),                               # d_h = 64: the single-CTA kernel
    (1, 32, 2, 6000, 0, {}, 64),                                 # d_h = 64, G = 16, ragged
])
def test_pass_runs_and_matches_oracle(B, H_q, H_kv, S, window, opts, d):
    dev = _dev()
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S, S, d, 7700 + S + H_q)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    assert apex.fwd_workspace_bytes(B, H_q, H_kv, S, S, d, window=window, **opts) == B * H_kv * S * d * 2
    ws = _ws(B, H_kv, S, d, dev)
    out = apex.fwd(qd, kd, vd, window=window, workspace=ws, **opts)
    torch.cuda.synchronize()
    # the pass ran: the workspace holds the keys as apex_attn_rope_keys rotates them
    rot = apex.rope_keys(kd, **{k_: v_ for k_, v_ in opts.items() if k_.startswith("yarn")})
    held = ws.view(torch.bfloat16).view(B, H_kv, S, d)
    assert torch.equal(held.view(torch.int16), rot.view(torch.int16))
    rows = _rows(S, 7)
    oracle_opts = {("yarn_s" if k_ == "yarn_scale" else k_): v_ for k_, v_ in opts.items()}
    ref = oracle.attn(q, k, v, window=window, rows=rows, **oracle_opts)
    mx, mean = _errs(out[:, :, rows].cpu(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    # and the in-kernel rotation path agrees within the tolerance
    plain = apex.fwd(qd, kd, vd, window=window, workspace=False, **opts)
    mx2, mean2 = _errs(out.cpu(), plain.double().cpu().numpy())
    assert mx2 <= MAX_ERR and mean2 <= MEAN_ERR, (mx2, mean2)
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("B,H_q,H_kv,S,window", [
    (1, 4, 2, 256, 0),
    (2, 8, 2, 1000, 100),
])
def test_small_problem_leaves_workspace_untouched(B, H_q, H_kv, S, window):
    dev = _dev()
    d = 128
    q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 7800 + S))
    assert apex.fwd_workspace_bytes(B, H_q, H_kv, S, S, d, window=window) == 0
    ws = _ws(B, H_kv, S, d, dev)
    out = apex.fwd(q, k, v, window=window, workspace=ws)
    ref = apex.fwd(q, k, v, window=window, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert bool((ws.view(torch.int16) == NAN_BF16).all())


def test_prerotated_keys_never_use_the_workspace():
    dev = _dev()
    B, H_q, H_kv, S, d = 2, 8, 2, 8192, 128
    q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 7900))
    kr = apex.rope_keys(k)
    ws = _ws(B, H_kv, S, d, dev)
    out = apex.fwd(q, kr, v, window=2048, keys_prerotated=True, workspace=ws)
    ref = apex.fwd(q, kr, v, window=2048, keys_prerotated=True, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert bool((ws.view(torch.int16) == NAN_BF16).all())


def test_pass_and_prefill_captured_in_a_graph():
    """The two kernels of a prefill that rotates its keys beforehand (the pass,
    and the prefill launched as its programmatic dependent) captured in one CUDA
    graph, replayed on new inputs copied into the same buffers."""
    dev = _dev()
    B, H_q, H_kv, S, d, W = 2, 8, 2, 8192, 128, 4096
    assert apex.fwd_workspace_bytes(B, H_q, H_kv, S, S, d, window=W) > 0
    q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, d, 8100))
    out = torch.empty_like(q)
    ws = _ws(B, H_kv, S, d, dev)
    apex.fwd(q, k, v, window=W, out=out, workspace=ws)  # table built, module loaded
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            apex.fwd(q, k, v, window=W, out=out, workspace=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    rows = _rows(S, 11)
    for seed in (8101, 8102):
        qh, kh, vh = inputs.make_qkv(B, H_q, H_kv, S, S, d, seed)
        q.copy_(qh)
        k.copy_(kh)
        v.copy_(vh)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.attn(qh, kh, vh, window=W, rows=rows)
        mx, mean = _errs(out[:, :, rows].cpu(), ref)
        assert mx <= MAX_ERR and mean <= MEAN_ERR, (seed, mx, mean)
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("H_q,H_kv,window", [(32, 2, 0), (8, 2, 2500)])
def test_pass_on_a_chunk_of_a_longer_sequence(H_q, H_kv, window):
    """A prefill of rows at positions 3000..6999 against 9001 keys (the last
    2001 never visible): the pass rotates the keys up to the end of the last
    128-key tile any work item reads and leaves the rest of the workspace as
    it was; the output matches the oracle."""
    dev = _dev()
    B, S_q, S_k, q_pos0, d = 1, 4000, 9001, 3000, 128
    assert apex.fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d, window=window, q_pos0=q_pos0) > 0
    q = inputs.normal_bf16((B, H_q, S_q, d), 8300 + H_q, 0)
    k = inputs.normal_bf16((B, H_kv, S_k, d), 8300 + H_q, 1)
    v = inputs.normal_bf16((B, H_kv, S_k, d), 8300 + H_q, 2)
    kd = k.to(dev)
    ws = _ws(B, H_kv, S_k, d, dev)
    out = apex.fwd(q.to(dev), kd, v.to(dev), window=window, q_pos0=q_pos0, workspace=ws)
    torch.cuda.synchronize()
    n_pos = ((q_pos0 + S_q - 1) // 128 + 1) * 128  # 7040
    held = ws.view(torch.int16).view(B, H_kv, S_k, d)
    rot = apex.rope_keys(kd).view(torch.int16)
    assert torch.equal(held[:, :, :n_pos], rot[:, :, :n_pos])
    assert bool((held[:, :, n_pos:] == NAN_BF16).all())
    rows = _rows(S_q, 9)
    ref = oracle.attn(q, k, v, window=window, q_pos0=q_pos0, rows=rows)
    mx, mean = _errs(out[:, :, rows].cpu(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    assert apex.apex_attn_device_status() == 0
