"""The method's edge cases driven through the kernels, against the fp64 oracle.

The oracle's pins fix what these cases compute (pure decay at beta = 0, the undecayed
delta rule at alpha = 1, a reset at alpha = 0); here the same inputs go through the
CUDA path: the chunked tensor-core prefill (d = 128) and the batched decode kernel.

  beta_zero        b = -30 on every token: beta = sigmoid(-30) ~ 9e-14, S_t = alpha_t S_{t-1}
  beta_zero_mixed  b = -30 on a random half of the tokens
  alpha_one        A_log = -30: exp(A_log) ~ 9e-14, so g ~ 0 and alpha = 1 to fp32 precision
  alpha_zero       a = +30 on a random quarter of the tokens with A_log = ln 16: g = -480, so
                   alpha underflows to 0 within a step; the chunk's decay prefix G then spans
                   thousands, the case where exp(G_i - G_j) loses precision
  large_v          v scaled by 10^4 (|v| up to ~4e4): past fp16's 65504 once convolved and
                   multiplied through the triangular solve
  large_z          z scaled by 10^5: the output gate silu(z) w_n past fp16's range
  large_state      the slots start from a state scaled by 10^4
  huge_v           v scaled by 10^15 with the state scaled to match: far past any 16-bit
                   range, still well inside fp32 (the outputs' sums of squares stay finite)
"""
import math

import numpy as np
import pytest

from gated_deltanet_linear_rule_gb300 import synth
from gdn_harness import DECODE_TOL, PREFILL_TOL, Layer, host, relerr

pytestmark = pytest.mark.gpu

CASES = ["beta_zero", "beta_zero_mixed", "alpha_one", "alpha_zero", "large_v", "large_z", "large_state", "huge_v"]


def _edit_inputs(case, inp, io, seed):
    """A copy of the inputs with the case's edit, rounded back to the io dtype."""
    r = np.random.default_rng(seed)
    out = {k: v.copy() for k, v in inp.items()}
    T, hv = out["a"].shape
    if case == "beta_zero":
        out["b"][:] = -30.0
    elif case == "beta_zero_mixed":
        out["b"][r.random((T, hv)) < 0.5] = -30.0
    elif case == "alpha_zero":
        out["a"][r.random((T, hv)) < 0.25] = 30.0
    elif case == "large_v":
        out["v"] = out["v"] * 1e4
    elif case == "large_z":
        out["z"] = out["z"] * 1e5
    elif case == "huge_v":
        out["v"] = out["v"] * 1e15
    return {k: synth.to_io(v, io) for k, v in out.items()}


def _state_scale(case):
    return {"large_state": 1e4, "huge_v": 1e15}.get(case, 1.0)


def _layer(case, io):
    L = Layer(31, 1, 2, 128, io=io, out="f32", num_slots=8, max_prefill_tokens=256)
    p = L.params[0]
    if case == "alpha_one":
        p["A_log"] = np.full_like(p["A_log"], -30.0)
    elif case == "alpha_zero":
        p["A_log"] = np.full_like(p["A_log"], math.log(16.0))
    if case in ("alpha_one", "alpha_zero"):
        import torch
        L.pool.layer_params(0, torch.from_numpy(p["conv_w"]), torch.from_numpy(p["A_log"]),
                            torch.from_numpy(p["dt_bias"]), torch.from_numpy(p["norm_w"]))
    return L


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("case", CASES)
def test_edge_case_chunked_prefill_then_decode(case, io):
    """Chunked prefill (d = 128, GQA 2, lengths around the 64-token chunk) from random states, then four
    decode steps whose inputs carry the same edit: outputs and final states against the oracle."""
    L = _layer(case, io)
    lengths = [130, 64, 7, 1]
    n = len(lengths)
    slots = [L.pool.alloc() for _ in range(n)]
    sc = _state_scale(case)
    S0 = np.stack([synth.initial_state(31, 0, j, 2, 128, 128) * sc for j in range(n)]).astype(np.float64)
    conv0 = np.stack([synth.initial_convbuf(31, 0, j, 4, L.C, io) for j in range(n)]).astype(np.float64)
    for j, s in enumerate(slots):
        L.set_state(0, s, S0[j], conv0[j])
    inp, cu = synth.varlen_inputs(31, 0, lengths, 1, 2, 128, 128, io)
    inp = _edit_inputs(case, inp, io, 1)
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, S0, conv0)
    assert np.isfinite(o).all(), f"{case}: non-finite prefill output"
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    print(f"{case} {io}: prefill out {r_out:.2e}, S {r_S:.2e}")
    assert r_out <= PREFILL_TOL and r_S <= PREFILL_TOL, f"{case}: prefill out {r_out:.2e}, S {r_S:.2e}"
    for j, s in enumerate(slots):
        assert np.array_equal(L.get_state(0, s)[1], ref["convbuf"][j])
    S, conv = ref["S"], ref["convbuf"]
    for step in range(4):
        dinp = _edit_inputs(case, L.decode_inputs(list(range(n)), step), io, 100 + step)
        og = host(L.gpu_decode(0, slots, dinp))
        r = L.oracle_run(0, np.arange(n + 1), dinp, S, conv)
        S, conv = r["S"], r["convbuf"]
        e = relerr(og, r["out"])
        assert np.isfinite(og).all() and e <= DECODE_TOL, f"{case}: decode step {step} out {e:.2e}"
    for j, s in enumerate(slots):
        e = relerr(L.get_state(0, s)[0], S[j])
        assert e <= DECODE_TOL, f"{case}: final S of slot {s} after decode: {e:.2e}"
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("case", ["beta_zero", "alpha_zero", "large_v", "large_z"])
def test_edge_case_recurrent_prefill_d64(case):
    """The same edits through the d < 128 prefill path (d = 64, fp32 io), against the oracle."""
    L = Layer(32, 2, 4, 64, io="f32", out="f32", num_slots=4, max_prefill_tokens=256)
    if case == "alpha_zero":
        import torch
        p = L.params[0]
        p["A_log"] = np.full_like(p["A_log"], math.log(16.0))
        L.pool.layer_params(0, torch.from_numpy(p["conv_w"]), torch.from_numpy(p["A_log"]),
                            torch.from_numpy(p["dt_bias"]), torch.from_numpy(p["norm_w"]))
    lengths = [90, 33]
    slots = [L.pool.alloc() for _ in lengths]
    S0 = np.stack([synth.initial_state(32, 0, j, 4, 64, 64) for j in range(2)]).astype(np.float64)
    for j, s in enumerate(slots):
        L.set_state(0, s, S0[j])
    inp, cu = synth.varlen_inputs(32, 0, lengths, 2, 4, 64, 64, "f32")
    inp = _edit_inputs(case, inp, "f32", 2)
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, S0, np.zeros((2, 3, L.C)))
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    assert r_out <= PREFILL_TOL and r_S <= PREFILL_TOL, f"{case}: out {r_out:.2e}, S {r_S:.2e}"
    L.close()
