"""gdn_mixed_step: decode rows and prefill sequences of one layer in one call (a continuous-batching
step).  Its results are those of gdn_decode_step followed by gdn_prefill_varlen, bit for bit, both
run eagerly and replayed from a CUDA graph, and each part is checked against the oracle."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import synth
from gdn_harness import PREFILL_TOL, Layer, check_out, host, random_states, relerr

pytestmark = pytest.mark.gpu

HQK, HV, D = 4, 8, 128
M_DEC = 12
PRE_LENGTHS = [300, 1, 129, 64]


def _setup(workload: int, lengths=PRE_LENGTHS):
    """A pool with M_DEC decode slots holding random states and len(lengths) fresh prefill slots,
    plus one step of decode inputs and one set of packed prefill inputs."""
    T = sum(lengths)
    L = Layer(workload, HQK, HV, D, io="bf16", out="bf16", num_slots=M_DEC + len(lengths) + 2,
              max_prefill_tokens=T)
    dec_slots = [L.pool.alloc() for _ in range(M_DEC)]
    pre_slots = [L.pool.alloc() for _ in lengths]
    g = torch.Generator(device="cuda").manual_seed(workload)
    for s in dec_slots:
        Sv, Cv = L.pool.state_views(0, s)
        Sv.copy_(torch.randn(Sv.shape, generator=g, device="cuda") * 0.3)
        Cv.copy_((torch.randn(Cv.shape, generator=g, device="cuda")).to(Cv.dtype))
    torch.cuda.synchronize()
    dec_in = L.to_dev(L.decode_inputs(list(range(M_DEC)), 0))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pre_in = synth.token_inputs(workload, 0, 0, T, HQK, HV, D, D, "bf16")
    return L, dec_slots, pre_slots, dec_in, pre_in, cu


def _states(L, slots):
    out = []
    for s in slots:
        Sv, Cv = L.pool.state_views(0, s)
        out.append((Sv.clone(), Cv.clone()))
    return out


def _restore(L, slots, saved):
    for s, (S, C) in zip(slots, saved):
        Sv, Cv = L.pool.state_views(0, s)
        Sv.copy_(S)
        Cv.copy_(C)
    torch.cuda.synchronize()


@pytest.mark.parametrize("lengths", [PRE_LENGTHS, [40] * 10], ids=["decode_beside_state_pass", "decode_from_start"])
def test_mixed_step_equals_decode_then_prefill_bitwise(lengths):
    """With 4 prompts the state pass (2 CTAs per (sequence, v-head): 64) leaves SMs idle, and the
    decode runs beside it once the pre-pass is done; with 10 it fills the GPU (160 CTAs), and the
    decode runs beside the whole prefill.  Either way the results equal the two separate calls."""
    L, dec_slots, pre_slots, dec_in, pre_in, cu = _setup(41, lengths)
    all_slots = dec_slots + pre_slots
    init = _states(L, all_slots)
    T = int(cu[-1])
    ids_dec = torch.tensor(dec_slots, dtype=torch.int32, device="cuda")
    ptrs = L.pool.slot_ptrs(0, ids_dec)
    cu_d = torch.tensor(cu, device="cuda")
    ids_pre = torch.tensor(pre_slots, dtype=torch.int32, device="cuda")
    p = L.to_dev(pre_in)
    d = dec_in

    # separate calls, decode then prefill
    out_d1 = torch.empty((M_DEC, HV * D), dtype=torch.bfloat16, device="cuda")
    out_p1 = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")
    L.pool.decode_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_d1)
    L.pool.prefill_varlen(0, cu_d, ids_pre, len(pre_slots), T, p["q"], p["k"], p["v"], p["a"], p["b"], p["z"],
                          out_p1)
    torch.cuda.synchronize()
    sep = _states(L, all_slots)

    # one mixed call from the same states
    _restore(L, all_slots, init)
    out_d2 = torch.empty_like(out_d1)
    out_p2 = torch.empty_like(out_p1)
    L.pool.mixed_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_d2, cu_d, ids_pre,
                      len(pre_slots), T, p["q"], p["k"], p["v"], p["a"], p["b"], p["z"], out_p2)
    torch.cuda.synchronize()
    assert torch.equal(out_d1, out_d2)
    assert torch.equal(out_p1, out_p2)
    for (S1, C1), (S2, C2) in zip(sep, _states(L, all_slots)):
        assert torch.equal(S1, S2) and torch.equal(C1, C2)
    assert L.pool.device_status() == 0

    # the prefill part against the oracle (fresh slots)
    n = len(lengths)
    ref = L.oracle_run(0, cu, pre_in, np.zeros((n, HV, D, D)), np.zeros((n, L.W - 1, L.C)))
    check_out(host(out_p2), ref["out"], "bf16", PREFILL_TOL, "mixed step prefill out")
    L.close()


def test_mixed_step_graph_replay_equals_eager_bitwise():
    """The fork to the pool's internal stream and the join back are captured into a CUDA graph; the
    replay gives the eager results bit for bit."""
    L, dec_slots, pre_slots, dec_in, pre_in, cu = _setup(42)
    all_slots = dec_slots + pre_slots
    init = _states(L, all_slots)
    T = int(cu[-1])
    ptrs = L.pool.slot_ptrs(0, torch.tensor(dec_slots, dtype=torch.int32, device="cuda"))
    cu_d = torch.tensor(cu, device="cuda")
    ids_pre = torch.tensor(pre_slots, dtype=torch.int32, device="cuda")
    p = L.to_dev(pre_in)
    d = dec_in
    out_d = torch.empty((M_DEC, HV * D), dtype=torch.bfloat16, device="cuda")
    out_p = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")

    def step(stream=None):
        L.pool.mixed_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_d, cu_d, ids_pre,
                          len(pre_slots), T, p["q"], p["k"], p["v"], p["a"], p["b"], p["z"], out_p, stream=stream)

    step()  # eager, also the first call that creates the internal stream
    torch.cuda.synchronize()
    eager = (out_d.clone(), out_p.clone(), _states(L, all_slots))

    _restore(L, all_slots, init)
    out_d.zero_()
    out_p.zero_()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step(stream=cap)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_d, eager[0])
    assert torch.equal(out_p, eager[1])
    for (S1, C1), (S2, C2) in zip(eager[2], _states(L, all_slots)):
        assert torch.equal(S1, S2) and torch.equal(C1, C2)
    assert L.pool.device_status() == 0
    L.close()


def test_mixed_step_with_a_segmented_prefill():
    """A mixed step whose prefill part is one 33 000-token prompt: more chunk records than the
    workspace's 512, so the prefill runs in pipelined segments on the pool's second stream while the
    decode runs on the mixed step's own stream.  Results equal the two separate calls bit for bit;
    the prefill output and final state against the oracle."""
    hqk, hv, d, m = 1, 2, 128, 12
    T = 33000
    L = Layer(45, hqk, hv, d, io="bf16", out="f32", num_slots=m + 2, max_prefill_tokens=T)
    dec_slots = [L.pool.alloc() for _ in range(m)]
    pre_slot = L.pool.alloc()
    S0 = random_states(45, 0, dec_slots, hv, d)
    for s_, Si in zip(dec_slots, S0):
        L.set_state(0, s_, Si)
    dec = L.to_dev(L.decode_inputs(list(range(m)), 0))
    inp, cu = synth.varlen_inputs(45, 0, [T], hqk, hv, d, d, "bf16")
    p = L.to_dev(inp)
    cu_d = torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")
    ids = torch.tensor([pre_slot], dtype=torch.int32, device="cuda")
    ptrs = L.pool.slot_ptrs(0, torch.tensor(dec_slots, dtype=torch.int32, device="cuda"))
    all_slots = dec_slots + [pre_slot]
    init = _states(L, all_slots)
    out_d1 = torch.empty((m, hv * d), dtype=torch.float32, device="cuda")
    out_p1 = torch.empty((T, hv * d), dtype=torch.float32, device="cuda")
    L.pool.decode_step(0, ptrs, m, dec["q"], dec["k"], dec["v"], dec["a"], dec["b"], dec["z"], out_d1)
    L.pool.prefill_varlen(0, cu_d, ids, 1, T, p["q"], p["k"], p["v"], p["a"], p["b"], p["z"], out_p1)
    torch.cuda.synchronize()
    sep = _states(L, all_slots)
    _restore(L, all_slots, init)
    out_d2 = torch.empty_like(out_d1)
    out_p2 = torch.empty_like(out_p1)
    L.pool.mixed_step(0, ptrs, m, dec["q"], dec["k"], dec["v"], dec["a"], dec["b"], dec["z"], out_d2, cu_d, ids, 1, T,
                      p["q"], p["k"], p["v"], p["a"], p["b"], p["z"], out_p2)
    torch.cuda.synchronize()
    assert torch.equal(out_d1, out_d2)
    assert torch.equal(out_p1, out_p2)
    for (S1, C1), (S2, C2) in zip(sep, _states(L, all_slots)):
        assert torch.equal(S1, S2) and torch.equal(C1, C2)
    assert L.pool.device_status() == 0
    ref = L.oracle_run(0, cu, inp, np.zeros((1, hv, d, d)), np.zeros((1, L.W - 1, L.C)))
    check_out(host(out_p2), ref["out"], "f32", PREFILL_TOL, "segmented prefill in a mixed step")
    Sg, _ = L.get_state(0, pre_slot)
    assert relerr(Sg, ref["S"][0]) <= PREFILL_TOL
    L.close()


def test_mixed_step_with_one_part_empty():
    """m = 0 or n_seqs = 0 runs the other part alone (no fork), with the same results as its own call."""
    L, dec_slots, pre_slots, dec_in, pre_in, cu = _setup(43)
    T = int(cu[-1])
    ptrs = L.pool.slot_ptrs(0, torch.tensor(dec_slots, dtype=torch.int32, device="cuda"))
    init = _states(L, dec_slots)
    d = dec_in
    out_a = torch.empty((M_DEC, HV * D), dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    L.pool.decode_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_a)
    torch.cuda.synchronize()
    _restore(L, dec_slots, init)
    L.pool.mixed_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_b, None, None, 0, 0,
                      *([None] * 7))
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    cu_d = torch.tensor(cu, device="cuda")
    ids_pre = torch.tensor(pre_slots, dtype=torch.int32, device="cuda")
    p = L.to_dev(pre_in)
    out_p = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")
    L.pool.mixed_step(0, None, 0, *([None] * 7), cu_d, ids_pre, len(pre_slots), T, p["q"], p["k"], p["v"], p["a"],
                      p["b"], p["z"], out_p)
    torch.cuda.synchronize()
    n = len(PRE_LENGTHS)
    ref = L.oracle_run(0, cu, pre_in, np.zeros((n, HV, D, D)), np.zeros((n, L.W - 1, L.C)))
    check_out(host(out_p), ref["out"], "bf16", PREFILL_TOL, "mixed step prefill-only out")
    assert L.pool.device_status() == 0
    L.close()


def test_mixed_step_with_overlapping_slots_does_nothing():
    """A slot named by a decode row and by a prefill sequence: the device check sets
    GDN_DEV_SLOT_OVERLAP and neither part runs -- no output, state or conv buffer changes; the next
    call with disjoint slots runs normally."""
    L, dec_slots, pre_slots, dec_in, pre_in, cu = _setup(44)
    T = int(cu[-1])
    all_slots = dec_slots + pre_slots
    init = _states(L, all_slots)
    clash = list(pre_slots)
    clash[1] = dec_slots[5]  # the second prefill sequence names the sixth decode row's slot
    ptrs = L.pool.slot_ptrs(0, torch.tensor(dec_slots, dtype=torch.int32, device="cuda"))
    cu_d = torch.tensor(cu, device="cuda")
    p = L.to_dev(pre_in)
    d = dec_in
    out_d = torch.full((M_DEC, HV * D), 7.0, dtype=torch.bfloat16, device="cuda")
    out_p = torch.full((T, HV * D), 7.0, dtype=torch.bfloat16, device="cuda")
    L.pool.mixed_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_d, cu_d,
                      torch.tensor(clash, dtype=torch.int32, device="cuda"), len(clash), T, p["q"], p["k"], p["v"],
                      p["a"], p["b"], p["z"], out_p)
    torch.cuda.synchronize()
    assert L.pool.device_status() & 0x10
    assert torch.all(out_d == 7.0) and torch.all(out_p == 7.0)
    for (S0, C0), (S1, C1) in zip(init, _states(L, all_slots)):
        assert torch.equal(S0, S1) and torch.equal(C0, C1)
    # disjoint slots: the step runs (and clears the gate for the calls after it)
    L.pool.mixed_step(0, ptrs, M_DEC, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out_d, cu_d,
                      torch.tensor(pre_slots, dtype=torch.int32, device="cuda"), len(pre_slots), T, p["q"], p["k"],
                      p["v"], p["a"], p["b"], p["z"], out_p)
    torch.cuda.synchronize()
    assert L.pool.device_status() == 0
    n = len(PRE_LENGTHS)
    ref = L.oracle_run(0, cu, pre_in, np.zeros((n, HV, D, D)), np.zeros((n, L.W - 1, L.C)))
    check_out(host(out_p), ref["out"], "bf16", PREFILL_TOL, "mixed step prefill out after an overlap")
    L.close()
