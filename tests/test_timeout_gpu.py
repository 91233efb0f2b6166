"""A pipeline wait that runs out ends the kernel with a status bit, not a hang or a fault.

A pool created with GDN_DEBUG_FLAGS=1 has a decode kernel whose producer fills no stage, so
each consumer's bounded wait gives up after its 1 s limit; the launch sets GDN_DEV_TIMEOUT,
writes no output, and the context stays usable for a normal pool afterwards.  With
GDN_DEBUG_FLAGS=2 the chunked prefill's state pass never fetches its first chunk's record: both
CTAs of each cluster give up on it, leave the chunk loop, drain the copies they did issue and
meet at the closing cluster barrier."""
import os
import time

import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import DECODE_TOL, PREFILL_TOL, Layer, check_out, host, random_states

pytestmark = pytest.mark.gpu


def test_decode_wait_timeout_sets_status_and_context_survives(monkeypatch):
    monkeypatch.setenv("GDN_DEBUG_FLAGS", "1")
    L = Layer(31, 2, 2, 16, io="f32", num_slots=2)
    monkeypatch.delenv("GDN_DEBUG_FLAGS")
    slots = [L.pool.alloc(), L.pool.alloc()]
    inp = L.to_dev(L.decode_inputs([0, 1], 0))
    out = torch.full((2, 32), 5.0, device="cuda")
    ptrs = L.pool.slot_ptrs(0, torch.tensor(slots, dtype=torch.int32, device="cuda"))
    t0 = time.time()
    L.pool.decode_step(0, ptrs, 2, inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"], out)
    st = L.pool.device_status()
    elapsed = time.time() - t0
    assert st & binding.DEV_TIMEOUT, f"status {st}"
    assert elapsed < 30, "the bounded waits should end the kernel within seconds"
    assert torch.all(out == 5.0)
    L.close()
    # a normal pool on the same context still computes correct results
    N = Layer(31, 2, 2, 16, io="f32", num_slots=2)
    s = N.pool.alloc()
    S0 = random_states(31, 0, [s], 2, 16)
    N.set_state(0, s, S0[0])
    dinp = N.decode_inputs([0], 0)
    o = host(N.gpu_decode(0, [s], dinp))
    ref = N.oracle_run(0, [0, 1], dinp, S0, np.zeros((1, 3, N.C)))
    check_out(o, ref["out"], "f32", DECODE_TOL, "decode after a timed-out launch")
    assert N.pool.device_status() == 0
    N.close()


def test_prefill_state_wait_timeout_sets_status_and_context_survives(monkeypatch):
    monkeypatch.setenv("GDN_DEBUG_FLAGS", "2")
    L = Layer(32, 1, 2, 128, io="bf16", out="f32", num_slots=2, max_prefill_tokens=256)
    monkeypatch.delenv("GDN_DEBUG_FLAGS")
    slot = L.pool.alloc()
    inp, cu = synth.varlen_inputs(32, 0, [150], 1, 2, 128, 128, "bf16")
    d = L.to_dev(inp)
    out = torch.full((150, 2 * 128), 5.0, device="cuda")
    cu_d = torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")
    ids = torch.tensor([slot], dtype=torch.int32, device="cuda")
    t0 = time.time()
    L.pool.prefill_varlen(0, cu_d, ids, 1, 150, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out)
    st = L.pool.device_status()
    elapsed = time.time() - t0
    assert st & binding.DEV_TIMEOUT, f"status {st}"
    assert elapsed < 30, "the bounded waits should end the kernel within seconds"
    assert torch.all(out == 5.0), "no output row is written after the failed wait"
    S, _ = L.get_state(0, slot)
    assert not S.any(), "the slot's state is not written after the failed wait"
    L.close()
    # a normal pool on the same context still computes correct results
    N = Layer(32, 1, 2, 128, io="bf16", out="f32", num_slots=2, max_prefill_tokens=256)
    s = N.pool.alloc()
    o = host(N.gpu_prefill(0, [s], inp, cu))
    ref = N.oracle_run(0, cu, inp, np.zeros((1, 2, 128, 128)), np.zeros((1, 3, N.C)))
    check_out(o, ref["out"], "f32", PREFILL_TOL, "prefill after a timed-out state pass")
    assert N.pool.device_status() == 0
    N.close()
