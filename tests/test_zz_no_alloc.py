"""The allocation-free prefill entry point (gdn_prefill_varlen_noalloc) against the pool entry point.

Some callers cannot call cudaMalloc: their device memory is owned and budgeted by a host
framework or allocator of their own, or they run in a phase that must not allocate.  They
cannot create a pool, so the no-alloc entry point runs the same prefill kernels on slots the
caller already owns, with the library's fixed static scratch.  Its results must equal the pool
entry point's bit for bit (the same kernels on the same inputs), and the oracle's.  This file
is collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import PREFILL_TOL, Layer, check_out, host, relerr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize(
    "hqk,hv,d,io,lengths",
    [
        (16, 32, 128, "bf16", [5, 300, 64, 129]),  # the chunked tensor-core path (d = 128)
        (2, 4, 64, "f32", [37, 1, 90]),  # the d < 128 path, whose per-token workspace is the larger one
    ],
)
def test_noalloc_prefill_matches_pool_prefill_on_two_calls_in_a_row(hqk, hv, d, io, lengths):
    W = 4
    n, T = len(lengths), sum(lengths)
    L = Layer(11, hqk, hv, d, io=io, out=io, num_slots=n, max_prefill_tokens=T)
    pool_slots = [L.pool.alloc() for _ in lengths]

    # caller-owned slots for the no-alloc call, laid out like one pool layer (allocated here by the test)
    nslots = n + 2
    sb = binding.slot_bytes(hqk, hv, d, d, W, io)
    state_bytes = hv * d * d * 4
    conv_bytes = (W - 1) * L.C * (2 if io == "bf16" else 4)
    states = torch.zeros(nslots * sb, dtype=torch.uint8, device="cuda")
    assert states.data_ptr() % 256 == 0
    own_slots = [nslots - 1, 0, 3, 1][:n]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    params = [t.cuda() for t in L.pool._params[0]]
    out_dt = torch.bfloat16 if io == "bf16" else torch.float32

    S_ref, conv_ref = np.zeros((n, hv, d, d)), np.zeros((n, W - 1, L.C))
    for call in range(2):
        inp, cu = synth.varlen_inputs(11, 0, lengths, hqk, hv, d, d, io, first_id=10 * call)
        ref = L.gpu_prefill(0, pool_slots, inp, cu)
        dv = L.to_dev(inp)
        out = torch.empty((T, hv * d), dtype=out_dt, device="cuda")
        binding.prefill_varlen_noalloc(L.pool.shape, *params, states, nslots,
                                       torch.tensor(cu, dtype=torch.int32, device="cuda"),
                                       torch.tensor(own_slots, dtype=torch.int32, device="cuda"),
                                       n, T, dv["q"], dv["k"], dv["v"], dv["a"], dv["b"], dv["z"], out,
                                       status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref), f"call {call}: output differs from the pool entry point's"
        for j, s in enumerate(own_slots):
            S_pool, C_pool = L.pool.state_views(0, pool_slots[j])
            S_own = states[s * sb:s * sb + state_bytes]
            C_own = states[s * sb + state_bytes:s * sb + state_bytes + conv_bytes]
            assert torch.equal(S_own, S_pool.reshape(-1).view(torch.uint8)), f"call {call}: S of sequence {j}"
            assert torch.equal(C_own, C_pool.reshape(-1).view(torch.uint8)), f"call {call}: conv buffer of sequence {j}"
        # and the oracle, continuing from the states the previous call left
        r = L.oracle_run(0, cu, inp, S_ref, conv_ref)
        S_ref, conv_ref = r["S"], r["convbuf"]
        check_out(host(out), r["out"], io, PREFILL_TOL, f"call {call} output vs the oracle")
        for j, s in enumerate(own_slots):
            S_own = states[s * sb:s * sb + state_bytes].view(torch.float32).reshape(hv, d, d)
            assert relerr(host(S_own), S_ref[j]) <= PREFILL_TOL, f"call {call}: S of sequence {j} vs the oracle"
    L.close()


def test_noalloc_rejects_calls_beyond_the_static_scratch():
    hqk, hv, d, W = 16, 32, 128, 4
    shape = binding.GdnShape(hqk, hv, d, d, W, 64, 1, 1, 1e-6, 1e-6, 0)
    sb = binding.slot_bytes(hqk, hv, d, d, W, "bf16")
    states = torch.zeros(sb, dtype=torch.uint8, device="cuda")
    dummy = torch.zeros(16, device="cuda")
    cu = torch.tensor([0, 4096], dtype=torch.int32, device="cuda")
    ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.GdnError) as e:
        binding.prefill_varlen_noalloc(shape, dummy, dummy, dummy, dummy, states, 1, cu, ids, 1, 4096,
                                       dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert e.value.code == -6
