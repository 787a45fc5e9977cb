"""GPU: decoupled-RoPE keys rotated once (APEX-1 Mathematical Reference -- Part 2,
§9.3: rows [content (128) | rope part (64)], only the rope part rotated).

* apex_attn_mla_rope_keys copies the content part bit for bit and rotates the
  rope part as the oracle's 64-dimensional RoPE does, within one bf16 rounding;
* apex_attn_mla_fwd_ws, where the library's cost model rotates the keys into the
  workspace first, leaves there exactly what apex_attn_mla_rope_keys computes and
  matches the fp64 oracle (and the in-kernel-rotation path within the parity
  tolerance); where it does not, the workspace stays untouched and the output is
  bit-identical to the call without one;
* the decoupled-RoPE decode on a cache pre-rotated this way matches the oracle.
Tolerance: max |err| <= 2e-2, mean |err| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_rope_gb300 as apex
from transformer_attention_rope_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3
D_H, D_R = 128, 64
NAN_BF16 = -1  # 0xffff as int16: a NaN bf16 pattern no kernel writes


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _errs(got, ref):
    e = np.abs(torch.as_tensor(got).double().cpu().numpy() - np.asarray(ref, dtype=np.float64))
    return float(e.max()), float(e.mean())


def _ws(B, H_kv, S_k, dev):
    ws = torch.empty(B * H_kv * S_k * (D_H + D_R) * 2, dtype=torch.uint8, device=dev)
    ws.view(torch.int16).fill_(NAN_BF16)
    return ws


def _rows(S, step):
    return sorted(set(range(0, S, step)) | set(range(S - 64, S)) | set(range(64)))


@pytest.mark.parametrize("pos0,yarn", [(0, None), (1000, (16.0, 8.0, 2.0))])
def test_mla_rope_keys_matches_oracle(pos0, yarn):
    dev = _dev()
    B, H, S = 2, 3, 300
    k = inputs.normal_bf16((B, H, S, D_H + D_R), 820 + pos0, 1)
    kw = dict(yarn_scale=yarn[0], yarn_beta_fast=yarn[1], yarn_beta_slow=yarn[2]) if yarn else {}
    got = apex.mla_rope_keys(k.to(dev), D_R, pos0=pos0, **kw).cpu()
    # the content part is copied unchanged
    assert torch.equal(got[..., :D_H].view(torch.int16), k[..., :D_H].view(torch.int16))
    rope = got[..., D_H:].double().numpy()
    # the rope part is rotated exactly as 64-entry key rows are (same table, same arithmetic)
    same = apex.rope_keys(k[..., D_H:].contiguous().to(dev), pos0=pos0, **kw).cpu()
    assert torch.equal(got[..., D_H:].view(torch.int16), same.view(torch.int16))
    if yarn is None:
        # and within one bf16 rounding of the oracle's 64-dimensional RoPE
        pos = np.broadcast_to(np.arange(pos0, pos0 + S)[None, None, :], (B, H, S)).reshape(-1)
        ref = oracle.rope(k[..., D_H:].double().numpy().reshape(-1, D_R), pos).reshape(B, H, S, D_R)
        assert np.all(np.abs(rope - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_mla_rope_keys_append_into_cache():
    """Rotating n new key rows into rows [pos0, pos0 + n) of a larger cache leaves the rest untouched."""
    dev = _dev()
    S_cache, n, pos0, d = 256, 40, 100, D_H + D_R
    cache = torch.zeros((3, S_cache, d), dtype=torch.bfloat16, device=dev)
    new = inputs.normal_bf16((3, n, d), 821, 1).to(dev)
    opt = apex._options()
    st = apex.apex_attn_mla_rope_keys(new.data_ptr(), cache[:, pos0:].data_ptr(), 3, n, D_H, D_R, pos0, n * d,
                                      S_cache * d, opt, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    ref = apex.mla_rope_keys(new.view(1, 3, n, d).contiguous(), D_R, pos0=pos0).view(3, n, d)
    torch.cuda.synchronize()
    assert torch.equal(cache[:, pos0:pos0 + n], ref)
    assert torch.count_nonzero(cache[:, :pos0]) == 0 and torch.count_nonzero(cache[:, pos0 + n:]) == 0


# shapes on which each key tile is visited often enough for the pass to run
@pytest.mark.parametrize("B,H_q,H_kv,S,window,opts", [
    (1, 32, 2, 8192, 0, {}),                                    # G = 16, causal
    (1, 64, 4, 6000, 0, dict(prefix_len=700)),                  # prefix, ragged last tile
    (1, 32, 2, 8192, 0, dict(yarn_scale=8.0)),                  # YaRN frequencies in the pass
    (2, 8, 2, 8192, 6000, {}),                                  # G = 4, long window
])
def test_mla_pass_runs_and_matches_oracle(B, H_q, H_kv, S, window, opts):
    dev = _dev()
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S, S, D_H, 8700 + S + H_q, d_r=D_R)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    need = apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S, S, D_H, D_R, window=window, **opts)
    assert need == B * H_kv * S * (D_H + D_R) * 2
    ws = _ws(B, H_kv, S, dev)
    out = apex.mla_fwd(qd, kd, vd, D_R, window=window, workspace=ws, **opts)
    torch.cuda.synchronize()
    # the pass ran: the workspace holds the keys as apex_attn_mla_rope_keys rotates them
    rot = apex.mla_rope_keys(kd, D_R, **{k_: v_ for k_, v_ in opts.items() if k_.startswith("yarn")})
    held = ws.view(torch.bfloat16).view(B, H_kv, S, D_H + D_R)
    assert torch.equal(held.view(torch.int16), rot.view(torch.int16))
    rows = _rows(S, 13)
    oracle_opts = {("yarn_s" if k_ == "yarn_scale" else k_): v_ for k_, v_ in opts.items()}
    ref = oracle.mla_attn(q, k, v, D_R, window=window, rows=rows, **oracle_opts)
    mx, mean = _errs(out[:, :, rows].cpu(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    # and the in-kernel rotation path agrees within the tolerance
    plain = apex.mla_fwd(qd, kd, vd, D_R, window=window, workspace=False, **opts)
    mx2, mean2 = _errs(out.cpu(), plain.double().cpu().numpy())
    assert mx2 <= MAX_ERR and mean2 <= MEAN_ERR, (mx2, mean2)
    assert apex.apex_attn_device_status() == 0


@pytest.mark.parametrize("B,H_q,H_kv,S,window", [
    (1, 8, 2, 300, 0),
    (4, 32, 8, 4096, 1024),  # the gqa shape: each key tile visited about 9 times
])
def test_mla_small_visits_leave_workspace_untouched(B, H_q, H_kv, S, window):
    dev = _dev()
    q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, D_H, 8800 + S, d_r=D_R))
    assert apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S, S, D_H, D_R, window=window) == 0
    ws = _ws(B, H_kv, S, dev)
    out = apex.mla_fwd(q, k, v, D_R, window=window, workspace=ws)
    ref = apex.mla_fwd(q, k, v, D_R, window=window, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert bool((ws.view(torch.int16) == NAN_BF16).all())


def test_mla_prerotated_cache_prefill_and_decode():
    """Keys rotated by apex_attn_mla_rope_keys and passed with keys_prerotated:
    the prefill uses no workspace (and matches the raw-key call), and the decode
    matches the oracle given the raw keys."""
    dev = _dev()
    B, H_q, H_kv, S = 2, 16, 2, 3000
    q, k, v = inputs.make_qkv(B, H_q, H_kv, S, S, D_H, 8900, d_r=D_R)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kr = apex.mla_rope_keys(kd, D_R)
    assert apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S, S, D_H, D_R, keys_prerotated=True) == 0
    out = apex.mla_fwd(qd, kr, vd, D_R, keys_prerotated=True)
    raw = apex.mla_fwd(qd, kd, vd, D_R, workspace=False)
    torch.cuda.synchronize()
    mx, mean = _errs(out.cpu(), raw.double().cpu().numpy())
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    q1 = q[:, :, -1:].contiguous()
    o1 = apex.mla_decode(q1.to(dev), kr, vd, S - 1, D_R, keys_prerotated=True)
    torch.cuda.synchronize()
    ref = oracle.mla_attn(q1, k, v, D_R, q_pos0=S - 1)
    mx, mean = _errs(o1.cpu(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    assert apex.apex_attn_device_status() == 0


def test_mla_pass_and_prefill_captured_in_a_graph():
    """The decoupled-RoPE pass and the prefill launched as its programmatic
    dependent, captured in one CUDA graph and replayed on new inputs copied into
    the same buffers."""
    dev = _dev()
    B, H_q, H_kv, S = 1, 32, 2, 4096
    assert apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S, S, D_H, D_R) > 0
    q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H_q, H_kv, S, S, D_H, 9100, d_r=D_R))
    out = torch.empty((B, H_q, S, D_H), dtype=torch.bfloat16, device=dev)
    ws = _ws(B, H_kv, S, dev)
    apex.mla_fwd(q, k, v, D_R, out=out, workspace=ws)  # table built, module loaded
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            apex.mla_fwd(q, k, v, D_R, out=out, workspace=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    rows = _rows(S, 11)
    for seed in (9101, 9102):
        qh, kh, vh = inputs.make_qkv(B, H_q, H_kv, S, S, D_H, seed, d_r=D_R)
        q.copy_(qh)
        k.copy_(kh)
        v.copy_(vh)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.mla_attn(qh, kh, vh, D_R, rows=rows)
        mx, mean = _errs(out[:, :, rows].cpu(), ref)
        assert mx <= MAX_ERR and mean <= MEAN_ERR, (seed, mx, mean)
    assert apex.apex_attn_device_status() == 0


def test_mla_pass_on_a_chunk_of_a_longer_sequence():
    """Rows at positions 3000..6999 against 9001 key rows (the last 2001 never
    visible): the pass rotates the key rows up to the end of the last 128-key
    tile any work item reads, leaves the rest of the workspace as it was, and
    the output matches the oracle."""
    dev = _dev()
    B, H_q, H_kv, S_q, S_k, q_pos0 = 1, 32, 2, 4000, 9001, 3000
    assert apex.mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, D_H, D_R, q_pos0=q_pos0) > 0
    q = inputs.normal_bf16((B, H_q, S_q, D_H + D_R), 9200, 0)
    k = inputs.normal_bf16((B, H_kv, S_k, D_H + D_R), 9200, 1)
    v = inputs.normal_bf16((B, H_kv, S_k, D_H), 9200, 2)
    kd = k.to(dev)
    ws = _ws(B, H_kv, S_k, dev)
    out = apex.mla_fwd(q.to(dev), kd, v.to(dev), D_R, q_pos0=q_pos0, workspace=ws)
    torch.cuda.synchronize()
    n_pos = ((q_pos0 + S_q - 1) // 128 + 1) * 128  # 7040
    held = ws.view(torch.int16).view(B, H_kv, S_k, D_H + D_R)
    rot = apex.mla_rope_keys(kd, D_R).view(torch.int16)
    assert torch.equal(held[:, :, :n_pos], rot[:, :, :n_pos])
    assert bool((held[:, :, n_pos:] == NAN_BF16).all())
    rows = _rows(S_q, 9)
    ref = oracle.mla_attn(q, k, v, D_R, q_pos0=q_pos0, rows=rows)
    mx, mean = _errs(out[:, :, rows].cpu(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, (mx, mean)
    assert apex.apex_attn_device_status() == 0
