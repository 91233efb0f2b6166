"""CUDA-graph decode (issue #5279 phase P8) and slot snapshot / restore (phase P7, prefix reuse)."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import DECODE_TOL, PREFILL_TOL, Layer, check_out, host, relerr

pytestmark = pytest.mark.gpu


def test_graph_replay_of_decode_equals_eager_bitwise():
    """Eight decode steps at m = 64 captured into one CUDA graph keyed by the slot-pointer array: the
    replayed outputs and final states equal the eager run from the same states, bit for bit, and
    every row of every replayed step and every final state agrees with the oracle."""
    L = Layer(21, 16, 32, 128, io="bf16", out="bf16", num_slots=96)
    slots = [L.pool.alloc() for _ in range(64)]
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    blk = L.pool.state_block(0)
    g = torch.Generator(device="cuda").manual_seed(3)
    init = torch.randn(blk.shape, generator=g, device="cuda") * 0.3
    host_steps = [L.decode_inputs(list(range(64)), s) for s in range(8)]
    steps = [L.to_dev(h) for h in host_steps]
    outs = [torch.empty((64, 32 * 128), dtype=torch.bfloat16, device="cuda") for _ in steps]
    ptrs = L.pool.slot_ptrs(0, ids)

    def run_steps(stream=None):
        for d, o in zip(steps, outs):
            L.pool.decode_step(0, ptrs, 64, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], o, stream=stream)

    blk.copy_(init)
    for s in slots:
        L.pool.state_views(0, s)[1].zero_()
    run_steps()  # eager (also the warm-up call before capture)
    torch.cuda.synchronize()
    eager_out = [o.clone() for o in outs]
    eager_S = blk.clone()

    blk.copy_(init)
    for s in slots:
        L.pool.state_views(0, s)[1].zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            run_steps(stream=cap)
    # capture records the launches without running them: the states are still the initial ones
    assert torch.equal(blk, init)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager_out):
        assert torch.equal(a, b)
    assert torch.equal(blk, eager_S)
    assert L.pool.device_status() == 0

    # the replayed steps against the oracle, from the same initial states and zero conv buffers
    S = host(init[slots])
    conv = np.zeros((64, 3, L.C))
    for j, (hs, o) in enumerate(zip(host_steps, outs)):
        r = L.oracle_run(0, np.arange(65), hs, S, conv)
        S, conv = r["S"], r["convbuf"]
        check_out(host(o), r["out"], "bf16", DECODE_TOL, f"replayed step {j}")
    e = max(relerr(host(blk[s]), S[i]) for i, s in enumerate(slots))
    assert e <= DECODE_TOL, f"final states after the replay: {e:.3e}"
    L.close()


@pytest.mark.parametrize("prefix", [128, 100])
def test_snapshot_restore_prefix_reuse(prefix):
    """A prompt prefix is prefilled once and snapshotted; restoring it into other slots and prefilling
    different suffixes equals prefilling each full prompt from scratch (within the prefill tolerance:
    the restored call picks its fp16 operand scales from the restored state's measured maximum, the
    uninterrupted one from a bound carried across the chunk boundary, so values far below a chunk's
    largest can round differently) and the oracle's run of the full prompt; a host round trip restores
    the same bytes."""
    hqk, hv, d = 2, 4, 128
    suffix = 77
    L = Layer(22, hqk, hv, d, io="bf16", out="f32", num_slots=8, num_layers=2, layer_ids=(0, 1),
              max_prefill_tokens=prefix + suffix)
    base = L.pool.alloc()
    pre = synth.token_inputs(22, 0, 0, prefix, hqk, hv, d, d, "bf16")
    L.gpu_prefill(0, [base], pre, [0, prefix])
    snap_dev = L.pool.snapshot(base)
    snap_host = torch.empty(L.pool.snapshot_bytes(), dtype=torch.uint8).pin_memory()
    L.pool.snapshot(base, snap_host)
    torch.cuda.synchronize()
    assert torch.equal(snap_host.cuda(), snap_dev)
    for branch in (1, 2):
        suf = synth.token_inputs(22, 0, branch, suffix, hqk, hv, d, d, "bf16")
        reuse = L.pool.alloc()
        L.pool.restore(reuse, snap_dev if branch == 1 else snap_host)
        out_reuse = host(L.gpu_prefill(0, [reuse], suf, [0, suffix]))
        full = {k: np.concatenate([pre[k], suf[k]]) for k in pre}
        fresh = L.pool.alloc()
        out_full = host(L.gpu_prefill(0, [fresh], full, [0, prefix + suffix]))[prefix:]
        S_r, C_r = L.get_state(0, reuse)
        S_f, C_f = L.get_state(0, fresh)
        assert np.array_equal(C_r, C_f)
        assert relerr(out_reuse, out_full) <= PREFILL_TOL and relerr(S_r, S_f) <= PREFILL_TOL
        ref = L.oracle_run(0, [0, prefix + suffix], full, np.zeros((1, hv, d, d)), np.zeros((1, 3, L.C)))
        check_out(out_reuse, ref["out"][prefix:], "f32", PREFILL_TOL, "restored continuation")
        assert relerr(S_r, ref["S"][0]) <= PREFILL_TOL
        assert np.array_equal(C_r, ref["convbuf"][0])
        # layer 1 was never touched: the restore copied its zeros too
        assert not L.get_state(1, reuse)[0].any()
    with pytest.raises(binding.GdnError):
        L.pool.restore(7, snap_dev)  # slot 7 is free
    L.close()
