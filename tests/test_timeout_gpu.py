"""A pipeline wait that runs out ends the kernel with a status bit, not a hang or a fault.

A pool created with GDN_DEBUG_FLAGS=1 has a decode kernel whose producer fills no stage, so
each consumer's bounded wait gives up after its 1 s limit; the launch sets GDN_DEV_TIMEOUT,
writes no output, and the context stays usable for a normal pool afterwards."""
import os
import time

import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding
from gdn_harness import DECODE_TOL, Layer, check_out, host, random_states

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
