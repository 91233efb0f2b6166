"""Seeded synthetic inputs for the GDN layer (shared by the tests and the benchmark).

This module holds no arithmetic of the layer: it only draws random numbers and
rounds them to the io dtype.  Both the CUDA library and the fp64 oracle are fed
from here.

Every draw comes from numpy's Philox counter-based generator keyed by
(workload id, layer, sequence/slot id, stream tag), so any one sequence can be
regenerated on its own for an isolated run.  Distributions (the workloads'
recipe): q, k, v, z, a, b ~ N(0, 1) rounded to the io dtype; A_log ~ U(0, ln 16);
dt_bias = 0; conv weights ~ N(0, 0.25) (variance 0.25, std 0.5); RMSNorm weight 1;
initial states ~ N(0, 0.1) (variance 0.1) where a workload asks for a random state.
"""
from __future__ import annotations

import math

import numpy as np

# stream tags: which tensor family a draw belongs to
_TAGS = {"params": 1, "prefill": 2, "decode": 3, "state": 4, "schedule": 5, "slots": 6}


def _gen(workload: int, layer: int, ident: int, tag: str, sub: int = 0) -> np.random.Generator:
    key0 = (int(workload) & 0xFFFF) << 48 | (int(layer) & 0xFFFF) << 32 | (_TAGS[tag] & 0xFFFF) << 16
    key1 = (int(ident) & 0xFFFFFFFF) << 32 | (int(sub) & 0xFFFFFFFF)
    return np.random.Generator(np.random.Philox(key=[key0, key1]))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The uint16 bit patterns of float32 values that are exactly bfloat16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def to_io(x: np.ndarray, io_dtype: str) -> np.ndarray:
    """float32 values rounded to the io dtype ('f32' or 'bf16'), kept as float32."""
    if io_dtype == "bf16":
        return bf16_round(x)
    if io_dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(io_dtype)


def layer_params(workload: int, layer: int, hqk: int, hv: int, dk: int, dv: int, conv_w: int):
    """Per-layer parameters: conv weights [C][W], A_log [Hv], dt_bias [Hv], norm weight [dv] (fp32)."""
    C = 2 * hqk * dk + hv * dv
    g = _gen(workload, layer, 0, "params")
    w = (g.standard_normal((C, conv_w)) * 0.5).astype(np.float32)
    A_log = g.uniform(0.0, math.log(16.0), size=hv).astype(np.float32)
    return {
        "conv_w": w,
        "A_log": A_log,
        "dt_bias": np.zeros(hv, dtype=np.float32),
        "norm_w": np.ones(dv, dtype=np.float32),
    }


def token_inputs(workload: int, layer: int, ident: int, L: int, hqk: int, hv: int, dk: int, dv: int,
                 io_dtype: str, tag: str = "prefill", sub: int = 0):
    """Inputs for L tokens of one sequence: q, k [L][Hqk*dk]; v, z [L][Hv*dv]; a, b [L][Hv].

    ``ident`` is the sequence (or slot) id, ``sub`` the decode step for tag 'decode'."""
    g = _gen(workload, layer, ident, tag, sub)
    out = {}
    for name, width in (("q", hqk * dk), ("k", hqk * dk), ("v", hv * dv), ("z", hv * dv), ("a", hv), ("b", hv)):
        out[name] = to_io(g.standard_normal((L, width), dtype=np.float32), io_dtype)
    return out


def batch_inputs(workload: int, layer: int, idents, L: int, hqk: int, hv: int, dk: int, dv: int,
                 io_dtype: str, tag: str = "prefill", sub: int = 0):
    """token_inputs for several sequences of equal length, stacked row-wise in the given order."""
    parts = [token_inputs(workload, layer, i, L, hqk, hv, dk, dv, io_dtype, tag, sub) for i in idents]
    return {k: np.ascontiguousarray(np.concatenate([p[k] for p in parts], axis=0)) for k in parts[0]}


def varlen_inputs(workload: int, layer: int, lengths, hqk: int, hv: int, dk: int, dv: int, io_dtype: str,
                  first_id: int = 0):
    """Packed inputs of sequences with the given lengths (ids first_id, first_id+1, ...) and cu_seqlens."""
    parts = [token_inputs(workload, layer, first_id + i, L, hqk, hv, dk, dv, io_dtype) for i, L in enumerate(lengths)]
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    packed = {k: np.ascontiguousarray(np.concatenate([p[k] for p in parts], axis=0)) for k in parts[0]}
    return packed, cu


def initial_state(workload: int, layer: int, slot: int, hv: int, dv: int, dk: int, var: float = 0.1):
    """A random recurrent state [Hv][dv][dk] ~ N(0, var) (fp32)."""
    g = _gen(workload, layer, slot, "state")
    return (g.standard_normal((hv, dv, dk), dtype=np.float32) * np.float32(math.sqrt(var))).astype(np.float32)


def initial_convbuf(workload: int, layer: int, slot: int, conv_w: int, C: int, io_dtype: str):
    """A random conv buffer [W-1][C] ~ N(0, 1) in the io dtype (for tests that need a non-zero one)."""
    g = _gen(workload, layer, slot, "state", 1)
    return to_io(g.standard_normal((conv_w - 1, C), dtype=np.float32), io_dtype)


def distinct_slots(workload: int, m: int, num_slots: int, sub: int = 0) -> np.ndarray:
    """m distinct pool indices drawn at random (fixed per workload, m and sub)."""
    g = _gen(workload, 0, m, "slots", sub)
    return g.permutation(num_slots)[:m].astype(np.int32)


def rng(workload: int, tag: str = "schedule", sub: int = 0) -> np.random.Generator:
    """A generator for schedule decisions (admit/finish choices) of a workload."""
    return _gen(workload, 0, 0, tag, sub)


def device_token_inputs(workload: int, layer: int, ident: int, L: int, hqk: int, hv: int, dk: int, dv: int,
                        io_dtype: str, tag: str = "prefill", sub: int = 0, device: str = "cuda"):
    """Large inputs drawn on the device with torch's seeded counter-based (Philox) CUDA generator, keyed
    like token_inputs: q, k [L][Hqk*dk]; v, z [L][Hv*dv]; a, b [L][Hv] ~ N(0, 1) in the io dtype.
    For workloads too large to draw on the host; the same tensors (copied to the host) feed the oracle."""
    import torch

    seed = ((int(workload) & 0xFF) << 56) | ((int(layer) & 0xFF) << 48) | ((_TAGS[tag] & 0xFF) << 40) | \
           ((int(ident) & 0xFFFFF) << 20) | (int(sub) & 0xFFFFF)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if io_dtype == "bf16" else torch.float32
    out = {}
    for name, width in (("q", hqk * dk), ("k", hqk * dk), ("v", hv * dv), ("z", hv * dv), ("a", hv), ("b", hv)):
        out[name] = torch.randn((L, width), generator=g, device=device, dtype=torch.float32).to(dt)
    return out
