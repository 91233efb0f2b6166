"""Slot pool behaviour on the GPU: allocation, recycling (zeroing), exhaustion, contamination."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import binding, synth
from gdn_harness import PREFILL_TOL, Layer, check_out, host, relerr

pytestmark = pytest.mark.gpu


def test_alloc_recycle_exhaustion():
    L = Layer(3, 2, 2, 16, io="f32", num_slots=3)
    p = L.pool
    ids = [p.alloc() for _ in range(3)]
    assert ids == [0, 1, 2]
    with pytest.raises(binding.GdnError) as e:
        p.alloc()
    assert e.value.code == -2
    p.recycle(1)
    with pytest.raises(binding.GdnError) as e:
        p.recycle(1)  # already free
    assert e.value.code == -3
    with pytest.raises(binding.GdnError) as e:
        p.recycle(7)
    assert e.value.code == -3
    assert p.info().free_slots == 1
    assert p.alloc() == 1
    p.reset()
    assert p.info().free_slots == 3 and p.alloc() == 0
    L.close()


def test_recycle_zeroes_every_layer_of_the_slot():
    L = Layer(3, 2, 4, 32, io="bf16", num_slots=4, num_layers=3, layer_ids=(0, 1, 2), max_prefill_tokens=64)
    a, b = L.pool.alloc(), L.pool.alloc()
    for layer in range(3):
        for s in (a, b):
            Sv, Cv = L.pool.state_views(layer, s)
            Sv.normal_()
            Cv.normal_()
    L.pool.recycle(a)
    torch.cuda.synchronize()
    for layer in range(3):
        Sa, Ca = L.get_state(layer, a)
        Sb, Cb = L.get_state(layer, b)
        assert not Sa.any() and not Ca.any(), f"layer {layer} of the recycled slot is not zero"
        assert Sb.any() and Cb.any(), "recycling one slot touched another"
    L.close()


def test_pool_sizes_match_the_layout():
    L = Layer(2, 16, 32, 128, io="bf16", num_slots=4, num_layers=2, layer_ids=(0, 1))
    inf = L.pool.info()
    assert inf.state_bytes == 32 * 128 * 128 * 4
    assert inf.conv_bytes == 3 * (2 * 16 * 128 + 32 * 128) * 2
    assert inf.slot_bytes % 256 == 0 and inf.slot_bytes >= inf.state_bytes + inf.conv_bytes
    assert L.pool.slot_addr(1, 2) - L.pool.slot_addr(0, 0) == (2 * 2 + 1) * inf.slot_bytes
    L.close()


def test_contamination_reused_slots_equal_isolated_runs():
    """Mixed batch with slot reuse (a small version of the 512-slot continuous-batching workload): each
    iteration finishes some sequences (recycle), admits new prefills into the freed slots and decodes every
    active slot.  Every admitted sequence's outputs equal an isolated run of the same sequence in a fresh
    pool, bit for bit."""
    hqk, hv, d = 2, 4, 64
    plen = 40
    L = Layer(4, hqk, hv, d, io="bf16", num_slots=6, max_prefill_tokens=2 * plen)
    rng = synth.rng(4)
    active = {}  # slot -> (sequence id, decode steps done)
    record = {}  # sequence id -> list of output rows (prefill block, then decode rows)
    next_id = 0
    for it in range(6):
        if len(active) >= 4:
            for s in rng.choice(sorted(active), size=2, replace=False):
                del active[int(s)]
                L.pool.recycle(int(s))
        new = []
        while len(active) + len(new) < 6 and len(new) < 2:
            new.append((L.pool.alloc(), next_id))
            next_id += 1
        if new:
            parts = [synth.token_inputs(4, 0, sid, plen, hqk, hv, d, d, "bf16") for _, sid in new]
            inp = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
            cu = np.arange(len(new) + 1) * plen
            out = host(L.gpu_prefill(0, [s for s, _ in new], inp, cu))
            for j, (s, sid) in enumerate(new):
                active[s] = (sid, 0)
                record[sid] = [out[j * plen:(j + 1) * plen]]
        slots = sorted(active)
        dinp = [synth.token_inputs(4, 0, active[s][0], 1, hqk, hv, d, d, "bf16", tag="decode", sub=active[s][1])
                for s in slots]
        inp = {k: np.concatenate([p[k] for p in dinp]) for k in dinp[0]}
        out = host(L.gpu_decode(0, slots, inp))
        for j, s in enumerate(slots):
            sid, n = active[s]
            record[sid].append(out[j:j + 1])
            active[s] = (sid, n + 1)
    assert L.pool.device_status() == 0
    L.close()
    # isolated runs: a fresh pool per sequence, same kernels at n = 1 / m = 1
    for sid, rows in record.items():
        I = Layer(4, hqk, hv, d, io="bf16", num_slots=1, max_prefill_tokens=plen)
        s = I.pool.alloc()
        inp = synth.token_inputs(4, 0, sid, plen, hqk, hv, d, d, "bf16")
        got = [host(I.gpu_prefill(0, [s], inp, [0, plen]))]
        for step in range(len(rows) - 1):
            dinp = synth.token_inputs(4, 0, sid, 1, hqk, hv, d, d, "bf16", tag="decode", sub=step)
            got.append(host(I.gpu_decode(0, [s], dinp)))
        for a, b in zip(got, rows):
            assert np.array_equal(a, b), f"sequence {sid} differs from its isolated run"
        I.close()


def test_recycle_and_reset_are_ordered_after_work_queued_on_their_stream():
    """gdn_slot_recycle and gdn_pool_reset clear the device allocation flags on the stream they are
    given: a prefill queued earlier on that (non-blocking) stream still finds its slot allocated and
    runs, and the zeroing follows it."""
    L = Layer(3, 2, 2, 16, io="f32", num_slots=2, max_prefill_tokens=64)
    inp, cu = synth.varlen_inputs(3, 0, [20], 2, 2, 16, 16, "f32")
    d = L.to_dev(inp)
    cu_d = torch.tensor(cu, device="cuda")
    st = torch.cuda.Stream()
    for how in ("recycle", "reset"):
        s = L.pool.alloc()
        ids = torch.tensor([s], dtype=torch.int32, device="cuda")
        out = torch.full((20, 32), 7.0, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            torch.cuda._sleep(20_000_000)  # keeps the prefill queued while the host goes on
            L.pool.prefill_varlen(0, cu_d, ids, 1, 20, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out, stream=st)
            if how == "recycle":
                L.pool.recycle(s, stream=st)
            else:
                L.pool.reset(stream=st)
        st.synchronize()
        assert L.pool.device_status(stream=st) == 0, how
        assert not torch.any(out == 7.0), f"{how}: the queued prefill did not run"
        Sg, Cg = L.get_state(0, s)
        assert not Sg.any() and not Cg.any(), f"{how}: the slot was not zeroed after the prefill"
    L.close()


@pytest.mark.parametrize("lengths", [[1] * 95 + [900], [150] * 4 + [4] * 85, [4] * 40 + [150, 600] + [2] * 50],
                         ids=["one_long", "four_of_three_chunks", "two_long_among_short"])
def test_chunked_prefill_in_segments(lengths):
    """At d = 128 a pool for 1 024-token calls holds 96 chunk records; a call with more chunks runs in
    segments of 48 (the state pass of one overlapping the pre-pass of the next), each continuing from
    the states the one before left in the slots.  Records are numbered chunk-index-major (every
    sequence's chunk 0, then chunk 1, ...), so with these mixes the long prompts' chunks fall into
    two or three segments, some of which hold no chunk of a given sequence.  Outputs, final states and
    conv buffers against the oracle, then two decode steps from those states."""
    L = Layer(33, 1, 2, 128, io="bf16", out="f32", num_slots=96, max_prefill_tokens=1024)
    assert L.pool.info().workspace_bytes < 16 * 2 ** 20  # 96 records of 2 x 57 KB + 32 KB, and small tables
    n = len(lengths)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(33, 0, lengths, 1, 2, 128, 128, "bf16")
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, np.zeros((n, 2, 128, 128)), np.zeros((n, 3, L.C)))
    check_out(o, ref["out"], "f32", PREFILL_TOL, "segmented prefill out")
    assert L.pool.device_status() == 0
    S, conv = ref["S"], ref["convbuf"]
    for j in range(n):
        Sg, Cg = L.get_state(0, slots[j])
        assert relerr(Sg, S[j]) <= PREFILL_TOL, f"final S of sequence {j}"
        assert np.array_equal(Cg, conv[j]), f"conv buffer of sequence {j}"
    pick = [0, n // 2, n - 1]
    S, conv = S[pick].copy(), conv[pick].copy()
    for step in range(2):
        dinp = L.decode_inputs(pick, step)
        out = host(L.gpu_decode(0, [slots[j] for j in pick], dinp))
        ref = L.oracle_run(0, np.arange(len(pick) + 1), dinp, S, conv)
        S, conv = ref["S"], ref["convbuf"]
        check_out(out, ref["out"], "f32", PREFILL_TOL, f"decode step {step} after the segmented prefill")
    L.close()


@pytest.mark.parametrize("lengths", [[4] * 600, [3] * 300 + [700] + [5] * 299], ids=["600_short", "one_long_among_600"])
def test_prefill_many_sequences(lengths):
    """More than 512 sequences in a call: the validation checks distinct slot ids with per-slot marks
    and ranks the lengths by a histogram instead of pairwise, and the call runs in segments whose
    state passes take only the sequences with records in them (with one long prompt among the short
    ones, a segment's sequences are two runs of ranks).  Outputs against the oracle, final states
    and conv buffers of a sample; then a call naming one slot twice is refused on the device with
    nothing written, and the marks are clear again for a valid call."""
    n = len(lengths)
    T = sum(lengths)
    L = Layer(36, 1, 2, 128, io="bf16", out="f32", num_slots=n, max_prefill_tokens=T)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(36, 0, lengths, 1, 2, 128, 128, "bf16")
    o = host(L.gpu_prefill(0, slots, inp, cu))
    assert L.pool.device_status() == 0
    ref = L.oracle_run(0, cu, inp, np.zeros((n, 2, 128, 128)), np.zeros((n, 3, L.C)))
    check_out(o, ref["out"], "f32", PREFILL_TOL, "many-sequence prefill out")
    for j in sorted({0, 1, n // 2, n // 2 + 1, n - 1}):
        Sg, Cg = L.get_state(0, slots[j])
        assert relerr(Sg, ref["S"][j]) <= PREFILL_TOL, f"final S of sequence {j}"
        assert np.array_equal(Cg, ref["convbuf"][j]), f"conv buffer of sequence {j}"
    # one slot named twice: refused on the device, nothing written
    d = L.to_dev(inp)
    cu_d = torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")
    dup = list(slots)
    dup[-1] = dup[n // 3]
    out = torch.full((T, 2 * 128), 7.0, device="cuda")
    before = L.get_state(0, slots[n // 3])
    L.pool.prefill_varlen(0, cu_d, torch.tensor(dup, dtype=torch.int32, device="cuda"), n, T, d["q"], d["k"], d["v"],
                          d["a"], d["b"], d["z"], out)
    assert L.pool.device_status() & binding.DEV_BAD_SLOT_ID
    assert torch.all(out == 7.0)
    after = L.get_state(0, slots[n // 3])
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    # the marks were cleared: the same valid call runs again (from the states the first one left)
    o2 = host(L.gpu_prefill(0, slots, inp, cu))
    assert L.pool.device_status() == 0
    ref2 = L.oracle_run(0, cu, inp, ref["S"], ref["convbuf"])
    check_out(o2, ref2["out"], "f32", PREFILL_TOL, "second many-sequence prefill out")
    L.close()


@pytest.mark.parametrize("d,chunk", [(16, 0), (32, 8)], ids=["recurrent_d16", "chunked_d32"])
def test_prefill_many_sequences_small_d(d, chunk):
    """More than 512 sequences at d < 128 (fp32): the validation's per-slot marks and length
    histogram feed the recurrent and the fp32 chunked kernels too.  Outputs and a sample of final
    states against the oracle; a repeated slot id is refused on the device."""
    lengths = [1, 2, 3, 5] * 150
    n, T = len(lengths), sum(lengths)
    L = Layer(37, 2, 4, d, io="f32", num_slots=n, chunk=chunk, max_prefill_tokens=T)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(37, 0, lengths, 2, 4, d, d, "f32")
    o = host(L.gpu_prefill(0, slots, inp, cu))
    assert L.pool.device_status() == 0
    ref = L.oracle_run(0, cu, inp, np.zeros((n, 4, d, d)), np.zeros((n, 3, L.C)))
    check_out(o, ref["out"], "f32", PREFILL_TOL, "many-sequence small-d prefill out")
    for j in (0, n // 2, n - 1):
        Sg, Cg = L.get_state(0, slots[j])
        assert relerr(Sg, ref["S"][j]) <= PREFILL_TOL
        assert np.array_equal(Cg, ref["convbuf"][j])
    dup = list(slots)
    dup[5] = dup[400]
    L.gpu_prefill(0, dup, inp, cu)
    assert L.pool.device_status() & binding.DEV_BAD_SLOT_ID
    L.close()


def test_segmented_prefill_graph_replay_equals_eager_bitwise():
    """A prefill that runs in pipelined segments forks work onto the pool's second stream and joins
    it back; captured into a CUDA graph, its replay gives the eager results bit for bit (outputs,
    states and conv buffers), twice in a row from the same starting states."""
    L = Layer(35, 1, 2, 128, io="bf16", out="f32", num_slots=96, max_prefill_tokens=1024)
    lengths = [4] * 40 + [150, 600] + [2] * 50
    n = len(lengths)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(35, 0, lengths, 1, 2, 128, 128, "bf16")
    T = int(cu[-1])
    d = L.to_dev(inp)
    cu_d = torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    out = torch.empty((T, 2 * 128), dtype=torch.float32, device="cuda")

    def call(stream=None):
        L.pool.prefill_varlen(0, cu_d, ids, n, T, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], out, stream=stream)

    def states():
        return [tuple(t.clone() for t in L.pool.state_views(0, s)) for s in slots]

    call()
    torch.cuda.synchronize()
    eager_out, eager_states = out.clone(), states()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    for s in slots:
        L.pool.recycle(s)
        L.pool.alloc()
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            call(stream=cap)
    for _ in range(2):
        for s in slots:  # the same zero starting states before each replay
            for t in L.pool.state_views(0, s):
                t.zero_()
        out.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager_out)
        for (S1, C1), (S2, C2) in zip(eager_states, states()):
            assert torch.equal(S1, S2) and torch.equal(C1, C2)
    assert L.pool.device_status() == 0
    L.close()


def test_chunked_prefill_workspace_is_bounded():
    """A pool for 80 000-token prefills holds 512 chunk records (1.2 GB at 16/32 heads), not one per
    chunk of the longest call."""
    L = Layer(34, 16, 32, 128, io="bf16", num_slots=1, max_prefill_tokens=80000)
    assert L.pool.info().workspace_bytes < 1.3e9
    L.close()
