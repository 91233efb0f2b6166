"""One whole GDN layer through the C ABI -- gdn_in_proj -> gdn_prefill_varlen -> gdn_out_proj over
three prompts, then decode steps gdn_in_proj -> gdn_decode_step -> gdn_out_proj on the same slots --
against the oracle's composition of the same maps: its projections in fp64, the layer's io rounded
to bf16 at each boundary (the layer's inputs q, k, v, z, a, b and its output o are bf16 values by
the boundary's definition), its recurrence on those values.

Tolerance: normwise 1e-2 on y.  The GPU's projection accumulates in fp32, so an output whose exact
value lies within that accumulation error of a bf16 rounding boundary can round to the
neighbouring bf16 value (one ulp, 2^-8 relative); such single-ulp input differences move the
affected rows of the layer's output by about the same relative amount, which the normwise bound
covers together with the layer's own prefill bound (5e-3) and the bf16 rounding of o.  A layout
mismatch between the three calls (a swapped segment, a transposed head, a wrong stride) gives
errors of order one."""
import numpy as np
import pytest
import torch

import oracle as oracle_pkg
from gated_deltanet_linear_rule_gb300 import binding
from gdn_harness import Layer, host, relerr

pytestmark = pytest.mark.gpu

HQK, HV, D, HID = 2, 4, 128, 256  # d = 128 takes the chunked tensor-core prefill
LENGTHS = [5, 130, 64]
TOL = 1e-2


def _round_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def _shape():
    return binding.GdnShape(hqk=HQK, hv=HV, dk=D, dv=D, conv_w=4, chunk=64, io_dtype=1, out_dtype=1, l2_eps=1e-6,
                            norm_eps=1e-6, max_prefill_tokens=0)


def _gpu_in_proj(x, w_in):
    T = x.shape[0]
    o = {n: torch.empty((T, w), dtype=torch.bfloat16, device="cuda")
         for n, w in (("q", HQK * D), ("k", HQK * D), ("v", HV * D), ("z", HV * D), ("a", HV), ("b", HV))}
    binding.in_proj(_shape(), HID, T, x, w_in, o["q"], o["k"], o["v"], o["z"], o["a"], o["b"])
    return o


def _gpu_out_proj(o, w_out):
    y = torch.empty((o.shape[0], HID), dtype=torch.bfloat16, device="cuda")
    binding.out_proj(_shape(), HID, o.shape[0], o, w_out, y)
    return y


def test_layer_prefill_then_decode_through_projections():
    L = Layer(51, HQK, HV, D, io="bf16", out="bf16", num_slots=len(LENGTHS) + 1, max_prefill_tokens=sum(LENGTHS))
    orc = oracle_pkg.load()
    n, T = len(LENGTHS), sum(LENGTHS)
    N = 2 * HQK * D + 2 * HV * D + 2 * HV
    g = torch.Generator().manual_seed(51)
    x = torch.randn((T, HID), generator=g).to(torch.bfloat16)
    w_in = (torch.randn((N, HID), generator=g) * HID ** -0.5).to(torch.bfloat16)
    w_out = (torch.randn((HID, HV * D), generator=g) * (HV * D) ** -0.5).to(torch.bfloat16)
    wi, wo = w_in.cuda(), w_out.cuda()
    w_in64, w_out64 = w_in.double().numpy(), w_out.double().numpy()
    cu = np.concatenate([[0], np.cumsum(LENGTHS)]).astype(np.int64)

    slots = [L.pool.alloc() for _ in LENGTHS]
    o = L.gpu_prefill(0, slots, _gpu_in_proj(x.cuda(), wi), cu)
    y = host(_gpu_out_proj(o, wo))

    pr = {k: _round_bf16(v) for k, v in orc.in_proj(x.double().numpy(), w_in64, HQK, HV, D, D).items()}
    ref = L.oracle_run(0, cu, pr, np.zeros((n, HV, D, D)), np.zeros((n, L.W - 1, L.C)))
    y_ref = orc.out_proj(_round_bf16(ref["out"]), w_out64)
    r = relerr(y, y_ref)
    print(f"layer prefill: y relative error {r:.2e}")
    assert r <= TOL, f"prefill layer output: relative error {r:.3e}"
    assert L.pool.device_status() == 0

    S, conv = ref["S"], ref["convbuf"]
    for step in range(3):
        xd = torch.randn((n, HID), generator=g).to(torch.bfloat16)
        od = L.gpu_decode(0, slots, _gpu_in_proj(xd.cuda(), wi))
        yd = host(_gpu_out_proj(od, wo))
        prd = {k: _round_bf16(v) for k, v in orc.in_proj(xd.double().numpy(), w_in64, HQK, HV, D, D).items()}
        rd = L.oracle_run(0, np.arange(n + 1), prd, S, conv)
        S, conv = rd["S"], rd["convbuf"]
        yd_ref = orc.out_proj(_round_bf16(rd["out"]), w_out64)
        r = relerr(yd, yd_ref)
        print(f"layer decode step {step}: y relative error {r:.2e}")
        assert r <= TOL, f"decode step {step} layer output: relative error {r:.3e}"
    assert L.pool.device_status() == 0
    L.close()
