"""Shared helpers of the GPU parity tests: run the CUDA library through its C ABI and
the fp64 oracle on the same seeded inputs, and compare.

Tolerances (normwise relative error ||gpu - oracle||_inf / ||oracle||_inf, per output
tensor and per final-state tensor):
  decode  <= 1e-3     prefill  <= 5e-3
fp32 outputs are compared against those bounds; bf16 outputs element-wise against
1e-3 * ||ref||_inf + half a bf16 ulp of the reference element (the output rounding
alone is up to 2^-9 relative, above the decode bound).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as oracle_pkg
from gated_deltanet_linear_rule_gb300 import binding, synth

DECODE_TOL = 1e-3
PREFILL_TOL = 5e-3


def dev(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device="cuda", dtype=dtype)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def relerr(a, b) -> float:
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / den) if den > 0 else float(np.abs(a - b).max())


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1e-38)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def check_out(gpu: np.ndarray, ref: np.ndarray, out_dtype: str, tol: float, what: str):
    if out_dtype == "f32":
        r = relerr(gpu, ref)
        assert r <= tol, f"{what}: relative error {r:.3e} > {tol:.1e}"
        return r
    bound = tol * np.abs(ref).max() + bf16_half_ulp(ref)
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} bf16 elements outside tol*|ref|max + ulp/2"
    return relerr(gpu, ref)


class Layer:
    """One GDN layer shape with seeded parameters, a pool, and the matching oracle shape."""

    def __init__(self, workload: int, hqk: int, hv: int, d: int, conv_w: int = 4, io: str = "bf16",
                 out: str | None = None, num_slots: int = 8, num_layers: int = 1, chunk: int = 0,
                 max_prefill_tokens: int = 0, layer_ids=(0,)):
        self.workload, self.hqk, self.hv, self.d, self.W = workload, hqk, hv, d, conv_w
        self.io, self.out = io, out or io
        self.C = 2 * hqk * d + hv * d
        self.pool = binding.Pool(hqk, hv, d, d, num_slots, num_layers, conv_w, io, self.out, chunk,
                                 max_prefill_tokens)
        self.params = {}
        for layer in layer_ids:
            p = synth.layer_params(workload, layer, hqk, hv, d, d, conv_w)
            self.params[layer] = p
            self.pool.layer_params(layer, torch.from_numpy(p["conv_w"]), torch.from_numpy(p["A_log"]),
                                   torch.from_numpy(p["dt_bias"]), torch.from_numpy(p["norm_w"]))
        self.oshape = {"hqk": hqk, "hv": hv, "dk": d, "dv": d, "conv_w": conv_w, "l2_eps": 1e-6, "norm_eps": 1e-6}
        self.oracle = oracle_pkg.load()

    def close(self):
        self.pool.close()

    # -- state -------------------------------------------------------------
    def set_state(self, layer, slot, S=None, conv=None):
        Sv, Cv = self.pool.state_views(layer, slot)
        if S is not None:
            Sv.copy_(dev(S))
        if conv is not None:
            Cv.copy_(dev(conv, Cv.dtype))
        torch.cuda.synchronize()

    def get_state(self, layer, slot):
        Sv, Cv = self.pool.state_views(layer, slot)
        torch.cuda.synchronize()
        return host(Sv), host(Cv)

    # -- inputs ------------------------------------------------------------
    def to_dev(self, inp):
        dt = self.pool.torch_io
        return {k: (v.contiguous() if isinstance(v, torch.Tensor) else dev(v, dt)) for k, v in inp.items()}

    def decode_inputs(self, idents, step, layer=0):
        return synth.batch_inputs(self.workload, layer, idents, 1, self.hqk, self.hv, self.d, self.d, self.io,
                                  tag="decode", sub=step)

    # -- runs --------------------------------------------------------------
    def gpu_decode(self, layer, slot_ids, inp, stream=None):
        m = len(slot_ids)
        ids = torch.tensor(np.asarray(slot_ids, dtype=np.int32), device="cuda")
        ptrs = self.pool.slot_ptrs(layer, ids, stream=stream)
        d = self.to_dev(inp)
        out = torch.empty((m, self.hv * self.d), dtype=self.pool.torch_out, device="cuda")
        self.pool.decode_step(layer, ptrs, m, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out, stream=stream)
        return out

    def gpu_prefill(self, layer, slot_ids, inp, cu, stream=None):
        T = int(cu[-1])
        d = self.to_dev(inp)
        out = torch.empty((T, self.hv * self.d), dtype=self.pool.torch_out, device="cuda")
        cu_d = torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")
        ids = torch.tensor(np.asarray(slot_ids, dtype=np.int32), device="cuda")
        self.pool.prefill_varlen(layer, cu_d, ids, len(slot_ids), T, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"],
                                 out, stream=stream)
        return out

    def oracle_run(self, layer, cu, inp, S, conv, head_mask=None, threads=0):
        """S [n][Hv][d][d], conv [n][W-1][C]: the states the sequences start from."""
        p = self.params[layer]
        return self.oracle.layer(self.oshape, np.asarray(cu, dtype=np.int64), inp["q"], inp["k"], inp["v"], inp["a"],
                                 inp["b"], inp["z"], p["conv_w"], p["A_log"], p["dt_bias"], p["norm_w"], S, conv,
                                 head_mask=head_mask, threads=threads)


def oracle_heads(L: "Layer", layer, cu, inp, S0, conv0, heads, threads=0, workers=None):
    """The oracle for selected v-heads only, each on a head-sliced problem (1 q/k head, 1 v head):
    heads are independent apart from the q/k head they read, so the slice is the same computation.
    The heads run concurrently on host threads (the oracle's C call releases the interpreter lock).
    inp: host arrays (or device tensors) as for Layer.oracle_run; S0 [n][Hv][d][d]; conv0 [n][W-1][C].
    Returns {h: (out [T][d], S [n][d][d])}."""
    import concurrent.futures as cf
    import os

    d, r, W = L.d, L.hv // L.hqk, L.W
    Cq = L.hqk * d
    p = L.params[layer]
    shape = dict(L.oshape, hqk=1, hv=1)

    def slice_head(h):
        hk = h // r
        qs, ks, vs = slice(hk * d, (hk + 1) * d), slice(hk * d, (hk + 1) * d), slice(h * d, (h + 1) * d)
        sub = {"q": inp["q"][:, qs], "k": inp["k"][:, ks], "v": inp["v"][:, vs], "z": inp["z"][:, vs],
               "a": inp["a"][:, h:h + 1], "b": inp["b"][:, h:h + 1]}
        # device tensors are sliced on the device and only the head's columns come to the host
        return {k: (host(v) if isinstance(v, torch.Tensor) else np.asarray(v)) for k, v in sub.items()}

    def run(h, sub):
        hk = h // r
        ch = np.concatenate([np.arange(hk * d, (hk + 1) * d), Cq + np.arange(hk * d, (hk + 1) * d),
                             2 * Cq + np.arange(h * d, (h + 1) * d)])
        o = L.oracle.layer(shape, np.asarray(cu, dtype=np.int64), sub["q"], sub["k"], sub["v"], sub["a"], sub["b"],
                           sub["z"], p["conv_w"][ch], p["A_log"][h:h + 1], p["dt_bias"][h:h + 1], p["norm_w"],
                           np.ascontiguousarray(S0[:, h:h + 1]), np.ascontiguousarray(conv0[:, :, ch]),
                           threads=threads)
        return h, (o["out"], o["S"][:, 0])

    subs = {h: slice_head(h) for h in heads}
    n = workers or min(len(heads), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        return dict(ex.map(lambda h: run(h, subs[h]), heads))


def random_states(workload, layer, slots, hv, d, var=0.1):
    return np.stack([synth.initial_state(workload, layer, s, hv, d, d, var) for s in slots]).astype(np.float64)


def gib(x):
    return x / 2 ** 30


__all__ = ["Layer", "dev", "host", "relerr", "check_out", "DECODE_TOL", "PREFILL_TOL", "random_states", "math"]
