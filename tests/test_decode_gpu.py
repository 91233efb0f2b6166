"""GPU parity of the batched decode kernel against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import synth
from gdn_harness import DECODE_TOL, Layer, check_out, host, random_states, relerr

pytestmark = pytest.mark.gpu


def _decode_run(L: Layer, layer, slots, steps, S0, conv0, sample=None, idents=None):
    """Run `steps` decode steps on the GPU at m = len(slots); compare rows `sample` with the oracle."""
    idents = list(range(len(slots))) if idents is None else idents
    sample = list(range(len(slots))) if sample is None else sample
    S = S0[sample].copy()
    conv = conv0[sample].copy()
    worst = 0.0
    for step in range(steps):
        inp = L.decode_inputs(idents, step, layer)
        out = host(L.gpu_decode(layer, slots, inp))
        sub = {k: v[sample] for k, v in inp.items()}
        ref = L.oracle_run(layer, np.arange(len(sample) + 1), sub, S, conv)
        S, conv = ref["S"], ref["convbuf"]
        worst = max(worst, check_out(out[sample], ref["out"], L.out, DECODE_TOL, f"decode out step {step}"))
    for j, row in enumerate(sample):
        Sg, Cg = L.get_state(layer, slots[row])
        r = relerr(Sg, S[j])
        assert r <= DECODE_TOL, f"final S of slot {slots[row]}: {r:.3e}"
        assert np.array_equal(Cg, conv[j]), f"conv buffer of slot {slots[row]}"
        worst = max(worst, r)
    return worst


def test_decode_tiny_fp32():
    """2 slots, 2 q/k + 2 v heads, d = 16, conv 4, fp32 io: 8 steps from a random state and conv buffer."""
    L = Layer(1, 2, 2, 16, io="f32", num_slots=4)
    slots = [L.pool.alloc(), L.pool.alloc()]
    S0 = random_states(1, 0, slots, 2, 16)
    conv0 = np.stack([synth.initial_convbuf(1, 0, s, 4, L.C, "f32") for s in slots]).astype(np.float64)
    for s, Si, ci in zip(slots, S0, conv0):
        L.set_state(0, s, Si, ci)
    worst = _decode_run(L, 0, slots, 8, S0, conv0)
    assert worst < 2e-5, f"fp32 decode should be near fp32 rounding, got {worst:.3e}"
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("hqk,hv,d,W", [(2, 4, 32, 4), (4, 4, 64, 3), (1, 8, 16, 2), (2, 2, 128, 1)])
def test_decode_shapes_fp32(hqk, hv, d, W):
    """Other head dims, GQA ratios and conv widths (fp32 io)."""
    L = Layer(7, hqk, hv, d, conv_w=W, io="f32", num_slots=3)
    slots = [L.pool.alloc() for _ in range(3)]
    S0 = random_states(7, 0, slots, hv, d)
    conv0 = np.stack([synth.initial_convbuf(7, 0, s, W, L.C, "f32") for s in slots]).astype(np.float64)
    for s, Si, ci in zip(slots, S0, conv0):
        L.set_state(0, s, Si, ci)
    worst = _decode_run(L, 0, slots, 3, S0, conv0)
    assert worst < 2e-5
    L.close()


@pytest.fixture(scope="module")
def pool256_35b():
    """The 35B-A3B-shaped GDN layer: 16 q/k heads, 32 v heads, d = 128, conv 4, bf16 io, a 256-slot
    pool whose states are N(0, 0.1)."""
    L = Layer(2, 16, 32, 128, io="bf16", out="bf16", num_slots=256)
    slots = [L.pool.alloc() for _ in range(256)]
    S0 = np.empty((256, 32, 128, 128), dtype=np.float32)
    for s in slots:
        S0[s] = synth.initial_state(2, 0, s, 32, 128, 128, 0.1)
    base = L.pool.slot_addr(0, 0)
    info = L.pool.info()
    for s in slots:
        Sv, _ = L.pool.state_views(0, s)
        Sv.copy_(torch.from_numpy(S0[s]).cuda())
    torch.cuda.synchronize()
    yield L, S0
    L.close()


def _reset_states(L, S0, slots):
    for s in slots:
        Sv, Cv = L.pool.state_views(0, s)
        Sv.copy_(torch.from_numpy(S0[s]).cuda())
        Cv.zero_()
    torch.cuda.synchronize()


@pytest.mark.parametrize("m", [1, 4, 8, 16, 256])
def test_decode_35b_layer_parity(pool256_35b, m):
    """m active slots at random distinct pool indices; bf16 out vs the oracle on sampled rows (m = 1,
    4, 8: one item per SM with an 8-stage ring; m = 16: 6 stages, 2 CTAs per SM; m = 256: 4 stages,
    3 CTAs per SM taking several items each)."""
    L, S0 = pool256_35b
    slots = [int(s) for s in synth.distinct_slots(2, m, 256)]
    _reset_states(L, S0, slots)
    sample = sorted(set([0, m // 2, m - 1]))
    conv0 = np.zeros((m, 3, L.C))
    _decode_run(L, 0, slots, 3, S0[slots].astype(np.float64), conv0, sample=sample)
    assert L.pool.device_status() == 0


def test_decode_35b_layer_100_steps_fp32_out(pool256_35b):
    """100 steps at m = 4 with the state checked at the end (bf16 in, fp32 out for the 1e-3 bound)."""
    L0, S0 = pool256_35b
    L = Layer(2, 16, 32, 128, io="bf16", out="f32", num_slots=8)
    slots = [L.pool.alloc() for _ in range(4)]
    init = np.stack([S0[s] for s in range(4)]).astype(np.float64)
    for s, Si in zip(slots, init):
        L.set_state(0, s, Si)
    worst = _decode_run(L, 0, slots, 100, init, np.zeros((4, 3, L.C)))
    assert worst <= DECODE_TOL
    L.close()


def test_decode_steps_back_to_back_without_sync():
    """12 decode steps at m = 8 queued on one stream with no host synchronisation between them (inputs
    uploaded first, one output buffer per step, the slot-pointer array formed by a kernel right before
    the first step).  A decode launch may be scheduled while the previous kernel on the stream ends
    (programmatic launch), so this checks that every step still sees the state and conv buffer that
    the step before it wrote: all outputs and the final states against the oracle."""
    L = Layer(2, 16, 32, 128, io="bf16", out="f32", num_slots=16)
    slots = [L.pool.alloc() for _ in range(8)]
    init = random_states(2, 0, slots, 32, 128)
    conv0 = np.stack([synth.initial_convbuf(2, 0, s, 4, L.C, "bf16") for s in slots]).astype(np.float64)
    for s, Si, ci in zip(slots, init, conv0):
        L.set_state(0, s, Si, ci)
    steps = 12
    idents = list(range(len(slots)))
    inputs = [L.decode_inputs(idents, step) for step in range(steps)]
    dev_inputs = [L.to_dev(inp) for inp in inputs]
    outs = [torch.empty((len(slots), 32 * 128), dtype=torch.float32, device="cuda") for _ in range(steps)]
    torch.cuda.synchronize()
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    ptrs = L.pool.slot_ptrs(0, ids)
    for step in range(steps):
        d = dev_inputs[step]
        L.pool.decode_step(0, ptrs, len(slots), d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], outs[step])
    torch.cuda.synchronize()
    S, conv = init.copy(), conv0.copy()
    for step in range(steps):
        ref = L.oracle_run(0, np.arange(len(slots) + 1), inputs[step], S, conv)
        S, conv = ref["S"], ref["convbuf"]
        check_out(host(outs[step]), ref["out"], "f32", DECODE_TOL, f"decode out step {step}")
    for j, s in enumerate(slots):
        Sg, Cg = L.get_state(0, s)
        assert relerr(Sg, S[j]) <= DECODE_TOL, f"final S of slot {s}"
        assert np.array_equal(Cg, conv[j]), f"conv buffer of slot {s}"
    assert L.pool.device_status() == 0
    L.close()


def test_decode_batched_equals_single_bitwise(pool256_35b):
    """Each slot's output and state in a batch equal the same slot run alone (m = 1), bit for bit, for
    64 slots.
    The launches differ in shape: m = 1 runs one item per SM with an 8-stage ring, m = 64 two CTAs
    per SM with 6 stages, m = 256 three CTAs per SM with 4 stages, each CTA taking several items."""
    L, S0 = pool256_35b
    slots = [int(s) for s in synth.distinct_slots(2, 256, 256, sub=1)]
    N = 64  # slots run alone: every row of the m = 64 batch and the first 64 rows of the m = 256 one
    blk = L.pool.state_block(0)
    batched = {}
    for m in (256, 64):
        _reset_states(L, S0, slots)
        outs = []
        for step in range(2):
            inp = L.decode_inputs(list(range(m)), step)
            outs.append(L.gpu_decode(0, slots[:m], inp).clone())
        batched[m] = (outs, blk[slots[:N]].clone(), [L.pool.state_views(0, s)[1].clone() for s in slots[:N]])
    _reset_states(L, S0, slots)
    for j, s in enumerate(slots[:N]):
        for step in range(2):
            inp = L.decode_inputs([j], step)
            o = L.gpu_decode(0, [s], inp)
            for m, (outs, _, _) in batched.items():
                assert torch.equal(o[0], outs[step][j]), f"slot {s} step {step} output differs from the m = {m} batch"
    torch.cuda.synchronize()
    alone = blk[slots[:N]]
    for m, (_, states, convs) in batched.items():
        assert torch.equal(alone, states), f"states of the slots run alone vs the m = {m} batch"
        for j, s in enumerate(slots[:N]):
            assert torch.equal(L.pool.state_views(0, s)[1], convs[j]), f"slot {s} conv buffer vs m = {m}"


def test_decode_m256_every_row_against_oracle(pool256_35b):
    """One step of the headline batch (m = 256 slots at random pool indices): every row's output and
    every slot's final state and conv buffer against the oracle."""
    L, S0 = pool256_35b
    slots = [int(s) for s in synth.distinct_slots(2, 256, 256)]
    _reset_states(L, S0, slots)
    _decode_run(L, 0, slots, 1, S0[slots].astype(np.float64), np.zeros((256, 3, L.C)))
    assert L.pool.device_status() == 0


def test_decode_deterministic(pool256_35b):
    """The same step twice from the same state gives identical bits."""
    L, S0 = pool256_35b
    slots = [int(s) for s in synth.distinct_slots(2, 32, 256, sub=2)]
    res = []
    for _ in range(2):
        _reset_states(L, S0, slots)
        inp = L.decode_inputs(list(range(32)), 0)
        res.append((L.gpu_decode(0, slots, inp).clone(), L.get_state(0, slots[5])[0]))
    assert torch.equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


def test_decode_bad_slot_pointer_is_skipped_not_faulted():
    """A pointer outside the layer's slots (or to another layer) skips that row and sets a status bit;
    the other rows are still computed and no memory outside the pool is touched."""
    L = Layer(3, 2, 2, 16, io="f32", num_slots=4, num_layers=2, layer_ids=(0, 1))
    a, b = L.pool.alloc(), L.pool.alloc()
    good = L.pool.slot_addr(0, a)
    wrong_layer = L.pool.slot_addr(1, b)
    misaligned = L.pool.slot_addr(0, b) + 64
    ptrs = torch.tensor([good, wrong_layer, misaligned, 0], dtype=torch.int64, device="cuda")
    inp = L.to_dev(L.decode_inputs([0, 1, 2, 3], 0))
    out = torch.full((4, 2 * 16), 7.0, device="cuda")
    L.pool.decode_step(0, ptrs, 4, inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"], out)
    st = L.pool.device_status()
    assert st & 0x1
    o = host(out)
    assert np.all(o[1:] == 7.0) and not np.all(o[0] == 7.0)
    assert L.pool.device_status() == 0  # reading clears the word
    L.close()


def test_slot_ptrs_rejects_freed_and_repeated_ids():
    L = Layer(3, 2, 2, 16, io="f32", num_slots=4)
    a, b = L.pool.alloc(), L.pool.alloc()
    ids = torch.tensor([a, 3, b, a, -1, 9], dtype=torch.int32, device="cuda")
    p = L.pool.slot_ptrs(0, ids).cpu().numpy()
    assert p[0] == L.pool.slot_addr(0, a) and p[2] == L.pool.slot_addr(0, b)
    assert p[1] == 0 and p[3] == 0 and p[4] == 0 and p[5] == 0
    assert L.pool.device_status() & 0x2
    L.close()
