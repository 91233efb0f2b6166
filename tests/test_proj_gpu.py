"""gdn_in_proj / gdn_out_proj (tcgen05 GEMMs with a routing epilogue) against the oracle's products.

bf16 operands, fp32 accumulation, bf16 outputs: each output element must lie within half a bf16
ulp of the fp64 product of the same bf16 inputs, plus an accumulation allowance of 1e-5 of the
largest |output| (fp32 sums of up to 4096 products)."""
import numpy as np
import pytest
import torch

import oracle as oracle_pkg
from gated_deltanet_linear_rule_gb300 import binding
from gdn_harness import bf16_half_ulp, host

pytestmark = pytest.mark.gpu


def _shape(hqk, hv, d):
    return binding.GdnShape(hqk=hqk, hv=hv, dk=d, dv=d, conv_w=4, chunk=64, io_dtype=1, out_dtype=1, l2_eps=1e-6,
                            norm_eps=1e-6, max_prefill_tokens=0)


def _bf16(t):
    return t.to(torch.bfloat16)


def _check(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    # half an ulp of the larger of the two (a value at a power of two may round up into the next
    # binade) plus the accumulation allowance
    bound = bf16_half_ulp(np.maximum(np.abs(ref), np.abs(gpu))) + 1e-5 * np.abs(ref).max()
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside the bound (max err {np.abs(gpu - ref).max():.3e})"


def _in_proj_case(hqk, hv, d, hidden, T, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    Dq, Dv = hqk * d, hv * d
    N = 2 * Dq + 2 * Dv + 2 * hv
    x = _bf16(torch.randn((T, hidden), generator=g, device="cuda"))
    w = _bf16(torch.randn((N, hidden), generator=g, device="cuda") * hidden ** -0.5)
    outs = {n: torch.full((T, wd), float("nan"), dtype=torch.bfloat16, device="cuda")
            for n, wd in (("q", Dq), ("k", Dq), ("v", Dv), ("z", Dv), ("a", hv), ("b", hv))}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.in_proj(_shape(hqk, hv, d), hidden, T, x, w, outs["q"], outs["k"], outs["v"], outs["z"], outs["a"],
                    outs["b"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle_pkg.load().in_proj(host(x), host(w), hqk, hv, d, d)
    for n in ref:
        _check(host(outs[n]), ref[n], f"in_proj {n} (Hqk {hqk}, Hv {hv}, d {d}, hidden {hidden}, T {T})")


@pytest.mark.parametrize("hqk,hv,d,hidden,T", [
    (2, 4, 16, 128, 300),     # N = 200: one partial N tile; 3 M tiles, the last partial; narrow a / b
    (1, 2, 32, 64, 1),        # one row, K = 64 (a single K slice)
    (4, 8, 64, 192, 129),     # GQA 2, d = 64, K = 3 slices
])
def test_in_proj_small_shapes(hqk, hv, d, hidden, T):
    _in_proj_case(hqk, hv, d, hidden, T, seed=hidden + T)


@pytest.mark.parametrize("T", [256, 300, 1100, 2100])
def test_in_proj_35b_layer_shape(T):
    """16 q/k and 32 v heads, d = 128, hidden 2048: N = 12 352 columns, K = 32 slices.  T = 256 (the
    decode batch) runs on CTA pairs with 256 x 192 tiles (one round), 2100 on pairs with 256 x 256
    tiles (each pair takes several in turn, and the last tile's second CTA holds no valid row); 300
    and 1100 fall a few rows past a multiple of 256 and run on single CTAs (128-row tiles, at 1100
    several per CTA).  The small shapes above take split-K clusters or 192-wide pairs."""
    _in_proj_case(16, 32, 128, 2048, T, seed=T)


@pytest.mark.parametrize("hidden,T", [(2048, 300), (256, 77), (2048, 2100)])
def test_out_proj(hidden, T):
    hqk, hv, d = 16, 32, 128
    Dv = hv * d
    g = torch.Generator(device="cuda").manual_seed(hidden + T)
    o = _bf16(torch.randn((T, Dv), generator=g, device="cuda"))
    w = _bf16(torch.randn((hidden, Dv), generator=g, device="cuda") * Dv ** -0.5)
    y = torch.full((T, hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.out_proj(_shape(hqk, hv, d), hidden, T, o, w, y)
    torch.cuda.synchronize()
    ref = oracle_pkg.load().out_proj(host(o), host(w))
    _check(host(y), ref, f"out_proj (hidden {hidden}, T {T})")


def test_projection_calls_reject_bad_arguments():
    sh = _shape(16, 32, 128)
    x = torch.zeros((8, 2048), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((12352, 2048), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((8, 2048), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((8, 4096), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((8, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.GdnError):  # hidden not a multiple of 64
        binding.in_proj(sh, 2000, 8, x, w, q, q, v, v, a, a)
    with pytest.raises(binding.GdnError):  # misaligned output
        binding.in_proj(sh, 2048, 8, x, w, q, q, v, v, a.view(-1)[1:].view(1, -1), a)
    bad = _shape(16, 32, 128)
    bad.io_dtype = 0
    with pytest.raises(binding.GdnError):  # fp32 io is not built
        binding.in_proj(bad, 2048, 8, x, w, q, q, v, v, a, a)
    binding.in_proj(sh, 2048, 0, x, w, q, q, v, v, a, a)  # T = 0: nothing to do
