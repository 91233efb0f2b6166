"""The allocation-free prefill entry point (gdn_prefill_varlen_noalloc) against the pool entry point.

Some callers cannot call cudaMalloc (their device memory is owned and budgeted elsewhere,
or they run in a phase that must not allocate), so they cannot create a pool; the
no-alloc entry point runs the same prefill kernels on slots the caller already owns, with
the library's static scratch.  This file is collected last on purpose: if it fails, a run
that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import PREFILL_TOL, Layer, host, relerr

pytestmark = pytest.mark.gpu


def test_noalloc_prefill_matches_pool_prefill_on_two_calls_in_a_row():
    hqk, hv, d, W = 16, 32, 128, 4
    lengths = [5, 300, 64, 129]
    T = sum(lengths)
    L = Layer(11, hqk, hv, d, io="bf16", out="bf16", num_slots=4, max_prefill_tokens=T)
    pool_slots = [L.pool.alloc() for _ in lengths]

    # caller-owned slots for the no-alloc call, laid out like one pool layer (allocated here by the test)
    nslots = 6
    sb = binding.slot_bytes(hqk, hv, d, d, W, "bf16")
    states = torch.zeros(nslots * sb, dtype=torch.uint8, device="cuda")
    assert states.data_ptr() % 256 == 0
    own_slots = [5, 0, 3, 1]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    params = [t.cuda() for t in L.pool._params[0]]

    for call in range(2):
        inp, cu = synth.varlen_inputs(11, 0, lengths, hqk, hv, d, d, "bf16", first_id=10 * call)
        ref = L.gpu_prefill(0, pool_slots, inp, cu)
        dv = L.to_dev(inp)
        out = torch.empty((T, hv * d), dtype=torch.bfloat16, device="cuda")
        binding.prefill_varlen_noalloc(L.pool.shape, *params, states, nslots,
                                       torch.tensor(cu, dtype=torch.int32, device="cuda"),
                                       torch.tensor(own_slots, dtype=torch.int32, device="cuda"),
                                       len(lengths), T, dv["q"], dv["k"], dv["v"], dv["a"], dv["b"], dv["z"], out,
                                       status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r = relerr(host(out), host(ref))
        assert r <= PREFILL_TOL, f"call {call}: output relative error {r:.3e}"
        for j, s in enumerate(own_slots):
            S_own = states[s * sb:s * sb + hv * d * d * 4].view(torch.float32)
            S_pool, C_pool = L.get_state(0, pool_slots[j])
            C_own = states[s * sb + hv * d * d * 4:s * sb + hv * d * d * 4 + (W - 1) * L.C * 2].view(torch.bfloat16)
            assert relerr(host(S_own).reshape(S_pool.shape), S_pool) <= PREFILL_TOL, f"call {call}: S of seq {j}"
            assert np.array_equal(host(C_own).reshape(C_pool.shape), C_pool), f"call {call}: conv buffer of seq {j}"
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
