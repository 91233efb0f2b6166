"""Bounds checks in place of a device memory checker: every output buffer of a call sits between
canary regions that must come back untouched, and every slot a call does not name must come back
bit for bit.  Shapes with partial tiles, partial chunks, empty sequences and several kernel paths.
Also: an allocation the device cannot satisfy is reported, and the context keeps working."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import Layer

pytestmark = pytest.mark.gpu

PAD = 64  # canary elements before and after each output (a multiple of 16 B for bf16 and fp32)
_CANARY = {torch.bfloat16: (torch.int16, 0x7FA5), torch.float32: (torch.int32, 0x7FC0A5A5)}  # NaN payloads


def _boxed(shape, dtype):
    """A buffer of `shape` inside canary padding: (the whole buffer, the view passed to a call)."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
    it, val = _CANARY[dtype]
    buf.view(it).fill_(val)
    return buf, buf[PAD:PAD + n].view(shape)


def _intact(buf) -> bool:
    it, val = _CANARY[buf.dtype]
    raw = buf.view(it)
    return bool((raw[:PAD] == val).all()) and bool((raw[-PAD:] == val).all())


def _fill_slots(L, slots, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    for s in slots:
        Sv, Cv = L.pool.state_views(0, s)
        Sv.copy_(torch.randn(Sv.shape, generator=g, device="cuda") * 0.3)
        Cv.copy_(torch.randn(Cv.shape, generator=g, device="cuda").to(Cv.dtype))
    torch.cuda.synchronize()


def _snap(L, slots):
    return [tuple(t.clone() for t in L.pool.state_views(0, s)) for s in slots]


def _same(a, b):
    return all(torch.equal(x, y) for p, q in zip(a, b) for x, y in zip(p, q))


@pytest.mark.parametrize("hqk,hv,d", [(2, 4, 128), (2, 4, 32)])
def test_decode_writes_only_its_slots_and_output(hqk, hv, d):
    L = Layer(61, hqk, hv, d, io="bf16", out="bf16", num_slots=8)
    slots = [L.pool.alloc() for _ in range(8)]
    _fill_slots(L, slots, 61)
    used, idle = [slots[1], slots[4], slots[6]], [slots[0], slots[2], slots[3], slots[5], slots[7]]
    before = _snap(L, idle)
    inp = L.to_dev(L.decode_inputs([0, 1, 2], 0))
    buf, out = _boxed((3, hv * d), torch.bfloat16)
    ptrs = L.pool.slot_ptrs(0, torch.tensor(used, dtype=torch.int32, device="cuda"))
    L.pool.decode_step(0, ptrs, 3, inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"], out)
    torch.cuda.synchronize()
    assert _intact(buf), "decode wrote outside its output"
    assert _same(before, _snap(L, idle)), "decode touched a slot it was not given"
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("hqk,hv,d,lengths", [(1, 2, 128, [70, 5, 0, 64]), (2, 4, 32, [9, 1, 0])])
def test_prefill_writes_only_its_slots_and_output(hqk, hv, d, lengths):
    """d = 128 runs the chunked tensor-core path (a partial second chunk, a short and an empty
    prompt); d = 32 the recurrent path."""
    T = sum(lengths)
    L = Layer(62, hqk, hv, d, io="bf16", out="f32", num_slots=len(lengths) + 3, max_prefill_tokens=T)
    slots = [L.pool.alloc() for _ in range(len(lengths) + 3)]
    _fill_slots(L, slots, 62)
    used, idle = slots[:len(lengths)], slots[len(lengths):]
    before = _snap(L, idle)
    inp, cu = synth.varlen_inputs(62, 0, lengths, hqk, hv, d, d, "bf16")
    dv = L.to_dev(inp)
    buf, out = _boxed((T, hv * d), torch.float32)
    L.pool.prefill_varlen(0, torch.tensor(cu, dtype=torch.int32, device="cuda"),
                          torch.tensor(used, dtype=torch.int32, device="cuda"), len(lengths), T, dv["q"], dv["k"],
                          dv["v"], dv["a"], dv["b"], dv["z"], out)
    torch.cuda.synchronize()
    assert _intact(buf), "prefill wrote outside its output"
    assert _same(before, _snap(L, idle)), "prefill touched a slot it was not given"
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("hqk,hv,d,hidden,T", [
    (2, 4, 16, 128, 300),     # split-K clusters of 2, partial N and M tiles, narrow a / b
    (1, 2, 32, 64, 1),        # 256 x 192 CTA pairs, one row
    (16, 32, 128, 2048, 300),  # single CTAs, a partial M tile
    (16, 32, 128, 2048, 256),  # 256 x 192 CTA pairs
])
def test_projections_write_only_their_outputs(hqk, hv, d, hidden, T):
    sh = binding.GdnShape(hqk=hqk, hv=hv, dk=d, dv=d, conv_w=4, chunk=64, io_dtype=1, out_dtype=1, l2_eps=1e-6,
                          norm_eps=1e-6, max_prefill_tokens=0)
    Dq, Dv = hqk * d, hv * d
    N = 2 * Dq + 2 * Dv + 2 * hv
    g = torch.Generator(device="cuda").manual_seed(hidden + T)
    x = torch.randn((T, hidden), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((N, hidden), generator=g, device="cuda") * hidden ** -0.5).to(torch.bfloat16)
    boxes = {n: _boxed((T, wd), torch.bfloat16)
             for n, wd in (("q", Dq), ("k", Dq), ("v", Dv), ("z", Dv), ("a", hv), ("b", hv))}
    o = {n: bx[1] for n, bx in boxes.items()}
    binding.in_proj(sh, hidden, T, x, w, o["q"], o["k"], o["v"], o["z"], o["a"], o["b"])
    wo = (torch.randn((hidden, Dv), generator=g, device="cuda") * Dv ** -0.5).to(torch.bfloat16)
    ybuf, y = _boxed((T, hidden), torch.bfloat16)
    if Dv % 64 == 0:
        binding.out_proj(sh, hidden, T, o["v"], wo, y)
    torch.cuda.synchronize()
    for n, (buf, _) in boxes.items():
        assert _intact(buf), f"in_proj wrote outside {n}"
    assert _intact(ybuf), "out_proj wrote outside y"


def test_pool_allocation_failure_is_reported_and_the_context_keeps_working():
    """A pool larger than the device (an allocation that must fail) is refused with a CUDA status,
    leaves no error behind for later calls, and a normal pool then computes as usual."""
    with pytest.raises(binding.GdnError):
        binding.Pool(16, 32, 128, 128, num_slots=200_000, num_layers=1)  # ~410 GB of state
    L = Layer(63, 2, 4, 128, io="bf16", out="bf16", num_slots=2)
    s = L.pool.alloc()
    o = L.gpu_decode(0, [s], L.decode_inputs([0], 0))
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert L.pool.device_status() == 0
    L.close()
