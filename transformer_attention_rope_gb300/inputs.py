"""Seeded synthetic inputs for the attention block.

This module holds no attention arithmetic: it only draws N(0, 1) numbers and
rounds them to bf16, so both the CUDA library's tests/bench and the fp64 oracle
can be fed the very same tensors.

Recipe (deterministic for a given seed, independent of the thread count):
  * tensors are drawn in the order Q, K, V (stream ids 0, 1, 2);
  * each tensor is cut into chunks of ``CHUNK`` elements; chunk c of stream s is
    filled by numpy's PCG64 seeded with SeedSequence([seed, s, c]) drawing
    float32 standard normals;
  * each float32 is rounded to bf16 (round-to-nearest-even).

The named workloads below are the five synthetic configurations of the
APEX-1 attention block (shapes from the pages' symbol table ranges: batch
1-64, sequence 2K-131K, head dim 64-128, 8-128 query heads, 2-8 KV heads,
window 512-4096).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    S_q: int
    S_k: int
    d_h: int
    window: int          # <= 0: causal only
    q_pos0: int          # position of query row 0 (decode: the query position)
    seed: int
    decode: bool = False
    rope_base: float = 10000.0
    d_r: int = 0         # > 0: decoupled RoPE; q / k rows hold d_h + d_r entries, v rows d_h

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv


WORKLOADS = {
    # B=1, H_q=4, H_kv=2, S=128, d_h=64, causal; seed 0
    "tiny": Workload("tiny", 1, 4, 2, 128, 128, 64, 0, 0, 0),
    # GQA prefill with a 1024-token sliding window
    "gqa": Workload("gqa", 4, 32, 8, 4096, 4096, 128, 1024, 0, 1),
    # wide-group (G=16) global causal prefill
    "wide": Workload("wide", 1, 128, 8, 8192, 8192, 128, 0, 0, 2),
    # long-context sliding window
    "long": Workload("long", 1, 32, 8, 65536, 65536, 128, 4096, 0, 3),
    # single-query decode at position 32767 against a 32768-entry KV cache
    "decode": Workload("decode", 64, 32, 8, 1, 32768, 128, 0, 32767, 4, decode=True),
    # global-layer prefill of multi-head latent attention with a 64-entry decoupled RoPE part
    "mla": Workload("mla", 1, 128, 8, 8192, 8192, 128, 0, 0, 5, d_r=64),
    # the decode cache shape with decoupled-RoPE key rows (128 + 64 entries)
    "mla_decode": Workload("mla_decode", 64, 32, 8, 1, 32768, 128, 0, 32767, 6, decode=True, d_r=64),
}


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def normal_bf16(shape, seed: int, stream: int, *, pin: bool = False) -> torch.Tensor:
    """Seeded N(0,1) draw rounded to bf16, as a CPU tensor of ``shape``."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, pin_memory=pin)
    n_chunks = (n + CHUNK - 1) // CHUNK

    def fill(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, c])))
        a = rng.standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi].copy_(torch.from_numpy(a))

    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.view(*shape)


def make_qkv(B: int, H_q: int, H_kv: int, S_q: int, S_k: int, d_h: int, seed: int,
             *, pin: bool = False, d_r: int = 0):
    """Q [B,H_q,S_q,d_h+d_r], K [B,H_kv,S_k,d_h+d_r], V [B,H_kv,S_k,d_h], bf16 on the CPU
    (drawn Q, K, V)."""
    q = normal_bf16((B, H_q, S_q, d_h + d_r), seed, 0, pin=pin)
    k = normal_bf16((B, H_kv, S_k, d_h + d_r), seed, 1, pin=pin)
    v = normal_bf16((B, H_kv, S_k, d_h), seed, 2, pin=pin)
    return q, k, v


def workload_inputs(w: Workload, *, pin: bool = False):
    return make_qkv(w.B, w.H_q, w.H_kv, w.S_q, w.S_k, w.d_h, w.seed, pin=pin, d_r=w.d_r)
