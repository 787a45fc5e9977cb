"""Benchmark of the APEX-1 attention hot path on GB300.

One step = one pass of the whole hot path on synthetic, seeded bf16 inputs:
  * the prefill call on the GQA prefill workload (B=4, H_q=32, H_kv=8, S=4096,
    d_h=128, causal + window 1024): RoPE, QK^T, mask/skip, online softmax, PV --
    through apex.fwd, i.e. apex_attn_fwd_ws with a workspace from torch, which
    on this workload rotates the keys once (rope_keys kernel) before the
    prefill kernel; the call's time covers both;
  * apex_attn_decode on the decode workload (B=64, H_q=32, H_kv=8, one query at
    position 32767 against a 32768-entry bf16 KV cache, d_h=128): split-KV
    kernel + log-sum-exp combine.

Reported (one JSON line on rank 0):
  value    prefill TFLOP/s over unmasked work, 4 * d_h * visible pairs * B * H_q
           per call, timed with CUDA events around the prefill calls;
  decode   KV GB/s, K + V bytes of the visible keys per call over the decode calls;
  roofline for the kernel that dominates the step (the decode split kernel,
           HBM-bound) and roofline_prefill (tensor-bound), against the measured
           peaks in MEASURED_PEAKS.json;
  e2e      the same two metrics through the same C-ABI calls with the inputs in
           pinned host memory: every step copies the step's inputs host->device
           and the outputs device->host inside the timed region (after the same
           number of untimed warm-up steps), each call type as a serving loop
           runs it: copy-in, compute and copy-out on three streams with two
           buffer sets, so that consecutive steps overlap;
  cpu_baseline  the fp64 oracle, as it stands, on a bounded sample of the same
           workloads on this machine's host cores.

  configs  the other prefill workloads (wide: B1 H_q128 H_kv8 S8192 causal;
           long: B1 H_q32 H_kv8 S65536 W4096; mla: the wide shape with 64-entry
           decoupled RoPE), each timed on its own after the step (same K and
           warm-up, CUDA events around every call) with its ms per call,
           TFLOP/s and fraction of the measured bf16 peak; all three rotate
           their keys (for mla: the rope parts) once before the prefill kernel,
           as the gqa call does, and the time covers both kernels.

With --impl reference the oracle itself is the timed arm (host cores, bounded
sample per step); it prints the same keys with "impl": "reference".
Multi-GPU: every rank runs the same step on its own GPU with its own seed
(independent problems, no collective on the data path): weak scaling.  Under
torchrun the ranks come from the environment; `--gpus N` without it starts N
ranks itself (torch.distributed.run on 127.0.0.1) and refuses to run when fewer
than N GPUs are visible.  `--launcher-check` runs only the ranks' host logic
(gloo, no GPU): each rank reports its seeds and the timings' max-reduction.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and decode KV GB/s on 1×GB300, as % of roofline"
PREFILL = "gqa"
DECODE = "decode"


def visible_range(m, window, prefix_len=0):
    """Keys [lo, hi] a query at position m sees (causal/window; a whole prefix inside it)."""
    if m < prefix_len:
        return 0, prefix_len - 1
    return (max(0, m - window + 1) if window > 0 else 0), m


def visible_pairs(S_q, S_k, window, q_pos0, prefix_len=0):
    """Number of (query, key) pairs the mask leaves visible, per head."""
    total = 0
    for r in range(S_q):
        lo, hi = visible_range(q_pos0 + r, window, prefix_len)
        total += min(hi, S_k - 1) - lo + 1
    return total


def flops_per_pair(w):
    """Tensor FLOPs of one visible (query, key) pair: 2 (d_h + d_r) for the score,
    2 d_h for its share of P V (d_r = 0 for the plain block)."""
    return 2.0 * (w.d_h + w.d_r) + 2.0 * w.d_h


def prefill_flops(w, prefix_len=0):
    return flops_per_pair(w) * visible_pairs(w.S_q, w.S_k, w.window, w.q_pos0, prefix_len) * w.B * w.H_q


def decode_kv_bytes(w, prefix_len=0):
    """K and V bytes a decode call must read: key rows of d_h + d_r, value rows of d_h entries."""
    lo, hi = visible_range(w.q_pos0, w.window, prefix_len)
    return 2.0 * w.B * w.H_kv * (hi - lo + 1) * (2 * w.d_h + w.d_r)


# --feature: the options of the block beyond the plain path, as keyword arguments
# of apex.fwd / apex.decode (YaRN with the pages' s = 32; a 1024-position
# bidirectional prefix; keys pre-rotated once before timing)
FEATURES = {
    "none": {},
    "yarn": {"yarn_scale": 32.0},
    "prefix": {"prefix_len": 1024},
    "prerotated": {"keys_prerotated": True},
}


def rank_workloads(rank, prefill_name=PREFILL, decode_batch=None, decode_name=DECODE):
    """The step's two workloads for one rank: same shapes on every rank, seeds
    offset by rank (independent problems, no data shared between ranks)."""
    from transformer_attention_rope_gb300 import inputs as inp
    wp, wd = inp.WORKLOADS[prefill_name], inp.WORKLOADS[decode_name]
    if decode_batch:
        wd = dataclasses.replace(wd, B=decode_batch)
    return (dataclasses.replace(wp, seed=wp.seed + 1000 * rank),
            dataclasses.replace(wd, seed=wd.seed + 1000 * rank))


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of a list of floats over all ranks of the default
    process group (the slowest rank decides the job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200"]
            if self.bus_id:
                cmd[1:1] = ["-i", self.bus_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        sm = []
        smax = None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
            except ValueError:
                continue
            for n, val in zip(names, r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def bus_id_of(dev_index):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return "%08x:%02x:%02x.0" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id, p.pci_device_id)
    except Exception:
        return None


# ---------------------------------------------------------------- CPU baseline (oracle)
def oracle_sample_prefill(w, q, k, v, budget_rows, batches=1):
    """Oracle on the first `batches` sequences, all heads, an evenly spaced
    subset of rows (all rows when budget_rows >= S_q)."""
    import oracle
    step = max(1, w.S_q // budget_rows)
    rows = list(range(0, w.S_q, step))
    t0 = time.perf_counter()
    if w.d_r:
        oracle.mla_attn(q[:batches], k[:batches], v[:batches], w.d_r, window=w.window, q_pos0=w.q_pos0, rows=rows)
    else:
        oracle.attn(q[:batches], k[:batches], v[:batches], window=w.window, q_pos0=w.q_pos0, rows=rows)
    dt = time.perf_counter() - t0
    pairs = 0
    for r in rows:
        m = w.q_pos0 + r
        lo = max(0, m - w.window + 1) if w.window > 0 else 0
        pairs += m - lo + 1
    flops = flops_per_pair(w) * pairs * w.H_q * batches
    return flops, dt, "prefill %s: %d of %d sequences, all %d heads, %d of %d rows (every %d-th)" % (
        w.name, batches, w.B, w.H_q, len(rows), w.S_q, step)


def oracle_sample_decode(w, q, k, v, n_batch):
    import oracle
    t0 = time.perf_counter()
    if w.d_r:
        oracle.mla_attn(q[:n_batch], k[:n_batch], v[:n_batch], w.d_r, window=w.window, q_pos0=w.q_pos0)
    else:
        oracle.attn(q[:n_batch], k[:n_batch], v[:n_batch], window=w.window, q_pos0=w.q_pos0)
    dt = time.perf_counter() - t0
    m = w.q_pos0
    lo = max(0, m - w.window + 1) if w.window > 0 else 0
    nbytes = 2.0 * n_batch * w.H_kv * (m - lo + 1) * (2 * w.d_h + w.d_r)
    return nbytes, dt, "decode: %d of %d sequences, full cache" % (n_batch, w.B)


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wp, wd, prefill_inputs, decode_inputs, rows=4096):
    fl, dtp, sp = oracle_sample_prefill(wp, *prefill_inputs, rows, batches=wp.B)
    nb, dtd, sd = oracle_sample_decode(wd, *decode_inputs, wd.B)
    return {"value": fl / dtp / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
            "sample": "%s (%.1f s); %s (%.1f s)" % (sp, dtp, sd, dtd),
            "decode_value": nb / dtd / 1e9, "decode_unit": "GB/s", "seconds": dtp + dtd}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from transformer_attention_rope_gb300 import inputs as inp
    wp, wd = inp.WORKLOADS[PREFILL], inp.WORKLOADS[DECODE]
    # inputs: the prefill workload in full, the decode workload for the sampled sequences only
    pin = inp.workload_inputs(wp)
    dq = inp.normal_bf16((wd.B, wd.H_q, 1, wd.d_h), wd.seed, 0)
    n_dec = 2
    dk = inp.normal_bf16((wd.B, wd.H_kv, wd.S_k, wd.d_h), wd.seed, 1)[:n_dec].contiguous()
    dv = inp.normal_bf16((wd.B, wd.H_kv, wd.S_k, wd.d_h), wd.seed, 2)[:n_dec].contiguous()
    rows = 256
    for _ in range(args.warmup):
        oracle_sample_prefill(wp, *pin, rows)
    fl_tot = t_p = nb_tot = t_d = 0.0
    sample = ""
    for _ in range(args.steps):
        fl, dt, sp = oracle_sample_prefill(wp, *pin, rows)
        nb, dt2, sd = oracle_sample_decode(wd, dq[:n_dec].contiguous(), dk, dv, n_dec)
        fl_tot += fl
        t_p += dt
        nb_tot += nb
        t_d += dt2
        sample = sp + "; " + sd
    value = fl_tot / t_p / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": (t_p + t_d) * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill %s + decode %s (oracle sample)" % (PREFILL, DECODE)},
        "decode": {"value": nb_tot / t_d / 1e9, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    import transformer_attention_rope_gb300 as apex
    from transformer_attention_rope_gb300 import inputs as inp

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    apex.load_library()

    wp, wd = rank_workloads(rank, args.prefill_workload, args.decode_batch, args.decode_workload)
    do_pre, do_dec = args.part in ("all", "prefill"), args.part in ("all", "decode")
    stream = torch.cuda.current_stream()

    pin = din = ()
    if do_pre:
        pin = inp.workload_inputs(wp, pin=True)
        pq, pk, pv = (t.to(dev, non_blocking=True) for t in pin)
        pout = torch.empty((wp.B, wp.H_q, wp.S_q, wp.d_h), dtype=torch.bfloat16, device=dev)
        pout_h = torch.empty(pout.shape, dtype=pout.dtype, pin_memory=True)
        apex.apex_attn_rope_reserve(wp.S_k, wp.d_r or wp.d_h, wp.rope_base)
    if do_dec:
        din = inp.workload_inputs(dataclasses.replace(wd, S_q=1), pin=True)
        dq, dk, dv = (t.to(dev, non_blocking=True) for t in din)
        dout = torch.empty((wd.B, wd.H_q, 1, wd.d_h), dtype=torch.bfloat16, device=dev)
        dout_h = torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)
        ws = torch.empty(apex.decode_workspace_bytes(wd.B, wd.H_q, wd.H_kv, wd.S_k, wd.d_h), dtype=torch.uint8,
                         device=dev)
        apex.apex_attn_rope_reserve(wd.S_k, wd.d_r or wd.d_h, wd.rope_base)
    torch.cuda.synchronize()

    feat = FEATURES[args.feature]
    if feat.get("keys_prerotated"):
        # the caches hold RoPE(k_j, j) (decoupled RoPE: the rope part rotated):
        # rotate the keys once, outside the timing
        if do_pre:
            pk = apex.mla_rope_keys(pk, wp.d_r) if wp.d_r else apex.rope_keys(pk)
        if do_dec:
            dk = apex.mla_rope_keys(dk, wd.d_r) if wd.d_r else apex.rope_keys(dk)
        torch.cuda.synchronize()

    def prefill():
        if wp.d_r:
            apex.mla_fwd(pq, pk, pv, wp.d_r, window=wp.window, q_pos0=wp.q_pos0, rope_base=wp.rope_base, out=pout,
                         **feat)
        else:
            apex.fwd(pq, pk, pv, window=wp.window, q_pos0=wp.q_pos0, rope_base=wp.rope_base, out=pout, **feat)

    def decode():
        if wd.d_r:
            apex.mla_decode(dq, dk, dv, wd.q_pos0, wd.d_r, window=wd.window, rope_base=wd.rope_base, out=dout,
                            workspace=ws, **feat)
        else:
            apex.decode(dq, dk, dv, wd.q_pos0, window=wd.window, rope_base=wd.rope_base, out=dout, workspace=ws,
                        **feat)

    warm = max(3, args.warmup)
    for _ in range(warm):
        if do_pre:
            prefill()
        if do_dec:
            decode()
    torch.cuda.synchronize()
    st = apex.apex_attn_device_status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)

    # ---- device-resident timed region: events before, between and after the two calls
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(bus_id_of(local))
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        ev[i][0].record(stream)
        if do_pre:
            prefill()
        ev[i][1].record(stream)
        if do_dec:
            decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    t_pre = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    t_all = ev[0][0].elapsed_time(ev[-1][2]) / 1e3
    st = apex.apex_attn_device_status()
    if st != 0:
        raise RuntimeError("device status %d after the timed region" % st)

    # ---- end to end through the C ABI with pinned host buffers.  Each call type
    # runs its steps as a serving loop would: three streams (copy in, compute,
    # copy out) and two sets of device buffers, so that step i + 1's inputs move
    # in while step i computes and step i - 1's result moves out.  Every step
    # still copies its own inputs in and its result out.
    h2d = sum(t.numel() * t.element_size() for t in (*pin, *din))
    if feat.get("keys_prerotated"):  # the pre-rotated key caches stay on the device
        h2d -= sum(t.numel() * t.element_size() for t in (pin[1:2] + din[1:2]))
    d2h = (pout.numel() * 2 if do_pre else 0) + (dout.numel() * 2 if do_dec else 0)

    def e2e_run(host_in, dev_sets, dev_outs, host_outs, call, keep):
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def step(i):
            b = i % 2
            if i >= 2:
                s_in.wait_event(comp_done[b])  # step i - 2 has consumed this input set
            with torch.cuda.stream(s_in):
                for j, (dst, src) in enumerate(zip(dev_sets[b], host_in)):
                    if j not in keep:
                        dst.copy_(src, non_blocking=True)
            in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if i >= 2:
                stream.wait_event(out_done[b])  # step i - 2's result has been read back
            call(*dev_sets[b], dev_outs[b])
            comp_done[b].record(stream)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                host_outs[b].copy_(dev_outs[b], non_blocking=True)
            out_done[b].record(s_out)

        # the first copies from (and into) freshly pinned buffers run several times
        # slower than later ones: warm up as the device-resident leg does
        for i in range(warm):
            step(i)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(warm, warm + K):
            step(i)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3

    te_pre = te_dec = 0.0
    if do_pre:
        keep = (1,) if feat.get("keys_prerotated") else ()
        sets = [(pq, pk, pv), tuple(t if j in keep else torch.empty_like(t) for j, t in enumerate((pq, pk, pv)))]
        outs = [pout, torch.empty_like(pout)]
        houts = [pout_h, torch.empty(pout.shape, dtype=pout.dtype, pin_memory=True)]

        def pre_call(q_, k_, v_, o_):
            if wp.d_r:
                apex.mla_fwd(q_, k_, v_, wp.d_r, window=wp.window, q_pos0=wp.q_pos0, rope_base=wp.rope_base, out=o_,
                             **feat)
            else:
                apex.fwd(q_, k_, v_, window=wp.window, q_pos0=wp.q_pos0, rope_base=wp.rope_base, out=o_, **feat)
        te_pre = e2e_run(pin, sets, outs, houts, pre_call, keep)
        del sets, outs
    if do_dec:
        keep = (1,) if feat.get("keys_prerotated") else ()
        sets = [(dq, dk, dv), tuple(t if j in keep else torch.empty_like(t) for j, t in enumerate((dq, dk, dv)))]
        outs = [dout, torch.empty_like(dout)]
        houts = [dout_h, torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)]

        def dec_call(q_, k_, v_, o_):
            if wd.d_r:
                apex.mla_decode(q_, k_, v_, wd.q_pos0, wd.d_r, window=wd.window, rope_base=wd.rope_base, out=o_,
                                workspace=ws, **feat)
            else:
                apex.decode(q_, k_, v_, wd.q_pos0, window=wd.window, rope_base=wd.rope_base, out=o_, workspace=ws,
                            **feat)
        te_dec = e2e_run(din, sets, outs, houts, dec_call, keep)
        del sets, outs

    # ---- the other prefill workloads, each timed on its own
    cfg_res, cfg_clocks = {}, None
    if args.config_names:
        cs = ClockSampler(bus_id_of(local))
        cs.start()
        cfg_res = time_prefill_configs(args.config_names, rank, K, warm, stream, dev)
        cfg_clocks = cs.stop()
    cfg_t = max_over_ranks([t for _, t in cfg_res.values()], pg, dev)

    flops = prefill_flops(wp, feat.get("prefix_len", 0))
    kvb = decode_kv_bytes(wd, feat.get("prefix_len", 0))
    t_pre, t_dec, t_all, te_pre, te_dec = max_over_ranks([t_pre, t_dec, t_all, te_pre, te_dec], pg, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and do_pre and do_dec and args.feature == "none":
        cpu = cpu_baseline(wp, wd, pin, din)

    if rank == 0:
        peaks = load_peaks()
        traffic = load_traffic()
        line = {"metric": METRIC, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": warm,
                "ms_per_step": t_all * 1e3 / K, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
        desc = []
        if do_pre:
            desc.append("prefill %s (B%d Hq%d Hkv%d S%d d%d%s W%d)" % (
                wp.name, wp.B, wp.H_q, wp.H_kv, wp.S_q, wp.d_h, ("+%d decoupled RoPE" % wp.d_r) if wp.d_r else "",
                wp.window))
        if do_dec:
            desc.append("decode %s(B%d Hq%d Hkv%d Sk%d d%d%s q_pos %d)" % (
                (wd.name + " ") if wd.d_r else "", wd.B, wd.H_q, wd.H_kv, wd.S_k, wd.d_h,
                ("+%d decoupled RoPE" % wd.d_r) if wd.d_r else "", wd.q_pos0))
        if args.feature != "none":
            desc.append("feature %s %s" % (args.feature, json.dumps(feat)))
        line["config"] = {
            "workload": " + ".join(desc),
            "l2": "inputs larger than L2 (prefill Q+K+V >= 201 MB; decode K+V 8.6 GB streamed every step)",
            "parallelism": "replica per GPU (independent problems)" if world > 1 else "1 GPU",
        }
        e2e = {"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        if do_pre:
            pre_launch_s = t_pre / K
            pre_achieved = flops / pre_launch_s / 1e12
            line["value"] = world * K * flops / t_pre / 1e12
            line["config"]["prefill_tflop_per_call"] = flops / 1e12
            line["prefill"] = {"value": line["value"], "unit": "TFLOP/s", "ms_per_call": pre_launch_s * 1e3,
                               "frac_of_bf16": pre_achieved / peaks["bf16_tflops"],
                               "frac_of_bf16_sustained": pre_achieved / peaks["bf16_tflops_sustained"]}
            kname, prerot = prefill_kernel_name(wp, feat)
            line["roofline_prefill"] = {"kernel": kernel_label(kname, prerot), "bound": "tensor",
                                        "achieved": pre_achieved,
                                        "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                        "frac": pre_achieved / peaks["bf16_tflops"],
                                        "traffic": call_traffic(traffic, "prefill_" + wp.name +
                                                                ("_single" if kname == "prefill_kernel" else ""),
                                                                prerot),
                                        "peak_source": peaks["source"] + " (burst)"}
            e2e.update({"value": world * K * flops / te_pre / 1e12, "unit": "TFLOP/s"})
        if do_dec:
            dec_launch_s = t_dec / K
            dec_achieved = kvb / dec_launch_s / 1e9
            line["config"]["decode_kv_bytes_per_call"] = kvb
            line["decode"] = {"value": world * K * kvb / t_dec / 1e9, "unit": "GB/s",
                              "ms_per_call": dec_launch_s * 1e3, "frac_of_hbm": dec_achieved / peaks["hbm_gbs"]}
            line["roofline_decode"] = {"kernel": "decode_split_kernel (+ its combine kernel, timed together)",
                                       "bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": dec_achieved / peaks["hbm_gbs"],
                                       "traffic": traffic.get(wd.name), "peak_source": peaks["source"]}
            e2e.update({"decode_value": world * K * kvb / te_dec / 1e9, "decode_unit": "GB/s"})
            if not do_pre:
                line["value"], line["unit"] = line["decode"]["value"], "GB/s"
                e2e.update({"value": e2e["decode_value"], "unit": "GB/s"})
        if cfg_res:
            configs = {}
            for (name, (w, _)), t in zip(cfg_res.items(), cfg_t):
                fl = prefill_flops(w)
                ach = fl / t / 1e12
                kname, prerot = prefill_kernel_name(w)
                configs[name] = {
                    "workload": "B%d Hq%d Hkv%d S%d d%d%s W%d" % (
                        w.B, w.H_q, w.H_kv, w.S_q, w.d_h, ("+%d decoupled RoPE" % w.d_r) if w.d_r else "",
                        w.window),
                    "ms_per_call": t * 1e3, "tflop_per_call": fl / 1e12,
                    "value": world * fl / t / 1e12, "unit": "TFLOP/s", "calls": K,
                    "roofline": {"kernel": kernel_label(kname, prerot), "bound": "tensor", "achieved": ach,
                                 "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                                 "frac_of_bf16_sustained": ach / peaks["bf16_tflops_sustained"],
                                 "traffic": call_traffic(traffic, "prefill_" + name +
                                                         ("_single" if kname == "prefill_kernel" else ""), prerot),
                                 "peak_source": peaks["source"] + " (burst)"}}
            line["configs"] = configs
            line["configs_clocks"] = cfg_clocks
        # the kernel that dominates the step's time carries the roofline key
        if do_dec and (not do_pre or t_dec >= t_pre):
            line["roofline"] = line["roofline_decode"]
        else:
            line["roofline"] = line["roofline_prefill"]
        line["e2e"] = e2e
        pre_launches = (2 if prefill_kernel_name(wp, feat)[1] else 1) if do_pre else 0
        line["gpu_launches"] = K * (pre_launches + (2 if do_dec else 0))
        line["clocks"] = clocks
        line["wall_s_timed"] = t_wall
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def prefill_call(apex, w, q, k, v, out, feat):
    if w.d_r:
        return apex.mla_fwd(q, k, v, w.d_r, window=w.window, q_pos0=w.q_pos0, rope_base=w.rope_base, out=out,
                            **feat)
    return apex.fwd(q, k, v, window=w.window, q_pos0=w.q_pos0, rope_base=w.rope_base, out=out, **feat)


def prefill_kernel_name(w, feat=None):
    """The prefill kernel a call runs, and whether the keys are rotated once by
    rope_keys_kernel before it (the call's time covers both)."""
    import transformer_attention_rope_gb300 as apex
    opts = {k: v for k, v in (feat or {}).items()}
    if w.d_r:
        prerot = apex.mla_fwd_workspace_bytes(w.B, w.H_q, w.H_kv, w.S_q, w.S_k, w.d_h, w.d_r, window=w.window,
                                              q_pos0=w.q_pos0, rope_base=w.rope_base, **opts) > 0
        return "prefill_pair_kernel", prerot
    name = ("prefill_kernel" if (w.d_h != 128 or os.environ.get("APEX_ATTN_PREFILL") == "single")
            else "prefill_pair_kernel")
    prerot = apex.fwd_workspace_bytes(w.B, w.H_q, w.H_kv, w.S_q, w.S_k, w.d_h, window=w.window, q_pos0=w.q_pos0,
                                      rope_base=w.rope_base, **opts) > 0
    return name, prerot


def call_traffic(traffic, key, prerot):
    """DRAM bytes of one call: the prefill kernel's, plus the key-rotation pass's
    when it runs (null when either capture is missing or stale)."""
    a = traffic.get(key)
    if not prerot:
        return a
    b = traffic.get(key + "_rope_keys")
    return a + b if (a is not None and b is not None) else None


def kernel_label(name, prerot):
    return ("rope_keys_kernel + %s (keys rotated once into the workspace, then the prefill; timed together)" % name
            if prerot else name)


def time_prefill_configs(names, rank, K, warm, stream, dev):
    """Each named prefill workload on its own: W warm-up calls, then K calls with
    CUDA events around each on the launching stream; returns seconds per call."""
    import torch

    import transformer_attention_rope_gb300 as apex
    from transformer_attention_rope_gb300 import inputs as inp
    res = {}
    for name in names:
        w = inp.WORKLOADS[name]
        w = dataclasses.replace(w, seed=w.seed + 1000 * rank)
        q, k, v = (t.to(dev) for t in inp.workload_inputs(w))
        out = torch.empty((w.B, w.H_q, w.S_q, w.d_h), dtype=torch.bfloat16, device=dev)
        apex.apex_attn_rope_reserve(w.S_k, w.d_r or w.d_h, w.rope_base)
        for _ in range(warm):
            prefill_call(apex, w, q, k, v, out, {})
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b in ev:
            a.record(stream)
            prefill_call(apex, w, q, k, v, out, {})
            b.record(stream)
        torch.cuda.synchronize()
        res[name] = (w, sum(a.elapsed_time(b) for a, b in ev) / 1e3 / K)
        del q, k, v, out
        torch.cuda.empty_cache()
    st = apex.apex_attn_device_status()
    if st != 0:
        raise RuntimeError("device status %d after the prefill configs" % st)
    return res


def free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n, argv):
    """Start n ranks of this script under torch.distributed.run (one node,
    rendezvous on 127.0.0.1) and return the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def run_launcher_check(args):
    """Host logic of the N-rank bench without a GPU: gloo process group, the
    per-rank seeds, and the max-over-ranks reduction of the timings."""
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    wp, wd = rank_workloads(rank, args.prefill_workload, args.decode_batch, args.decode_workload)
    timings = max_over_ranks([1.0 + rank, 2.0 * (world - rank)], dist if world > 1 else None)
    seeds = [[wp.seed, wd.seed]]
    if world > 1:
        gathered = [None] * world
        dist.all_gather_object(gathered, [wp.seed, wd.seed])
        seeds = gathered
    if rank == 0:
        print(json.dumps({"launcher_check": True, "n_ranks": world, "gpus_flag": args.gpus, "seeds": seeds,
                          "max_over_ranks": timings, "local_rank": local}))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def load_traffic():
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    only for kernels whose source is unchanged since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for key, rec in d.items():
        if not isinstance(rec, dict):
            continue
        try:
            with open(os.path.join(ROOT, rec["source"]), "rb") as f:
                same = hashlib.sha256(f.read()).hexdigest() == rec["sha256"]
        except (OSError, KeyError):
            same = False
        out[key] = rec.get("dram_bytes_per_launch") if same else None
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--part", choices=["all", "prefill", "decode"], default="all",
                    help="run only one of the two calls per step (profiling)")
    ap.add_argument("--prefill-workload", choices=["tiny", "gqa", "wide", "long", "mla"], default=PREFILL)
    ap.add_argument("--decode-workload", choices=["decode", "mla_decode"], default=DECODE)
    ap.add_argument("--feature", choices=sorted(FEATURES), default="none",
                    help="run the step with one of the block's options")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="decode batch size (profiling a smaller case; default: the workload's 64)")
    ap.add_argument("--configs", default=None,
                    help="comma list of further prefill workloads timed after the step (wide, long, mla) or "
                         "'none'; default: all three with --part all and --feature none, else none")
    ap.add_argument("--launcher-check", action="store_true",
                    help="start the ranks and run only their host logic (gloo, no GPU)")
    args = ap.parse_args()
    if args.configs is None:
        args.configs = "wide,long,mla" if (args.part == "all" and args.feature == "none") else "none"
    names = [c for c in args.configs.split(",") if c and c != "none"]
    for c in names:
        if c not in ("tiny", "gqa", "wide", "long", "mla"):
            ap.error("unknown prefill workload in --configs: %s" % c)
    args.config_names = names
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if "WORLD_SIZE" in os.environ:
        if int(os.environ["WORLD_SIZE"]) != args.gpus:
            print("bench.py: WORLD_SIZE=%s but --gpus %d" % (os.environ["WORLD_SIZE"], args.gpus), file=sys.stderr)
            return 2
    elif args.gpus > 1:
        # no launcher around us: start the N ranks ourselves
        if not args.launcher_check and args.impl == "ours":
            import torch
            have = torch.cuda.device_count()
            if have < args.gpus:
                print("bench.py: --gpus %d but %d GPU(s) visible" % (args.gpus, have), file=sys.stderr)
                return 2
        return launch_ranks(args.gpus, sys.argv[1:])
    if args.launcher_check:
        return run_launcher_check(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
