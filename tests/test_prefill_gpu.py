"""GPU parity of the varlen prefill against the fp64 oracle, and its hand-off to decode."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import synth
from gdn_harness import DECODE_TOL, PREFILL_TOL, Layer, check_out, host, relerr

pytestmark = pytest.mark.gpu


def _prefill_then_decode(L, lengths, decode_steps, tol_p, sample_heads=None, S_init=None):
    n = len(lengths)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(L.workload, 0, lengths, L.hqk, L.hv, L.d, L.d, L.io)
    S0 = np.zeros((n, L.hv, L.d, L.d)) if S_init is None else S_init
    if S_init is not None:
        for s, Si in zip(slots, S_init):
            L.set_state(0, s, Si)
    conv0 = np.zeros((n, L.W - 1, L.C))
    out = host(L.gpu_prefill(0, slots, inp, cu))
    mask = None
    if sample_heads is not None:
        mask = np.zeros(L.hv, dtype=np.int32)
        mask[sample_heads] = 1
    ref = L.oracle_run(0, cu, inp, S0, conv0, head_mask=mask)
    cols = np.concatenate([np.arange(h * L.d, (h + 1) * L.d) for h in (sample_heads or range(L.hv))])
    check_out(out[:, cols], ref["out"][:, cols], L.out, tol_p, "prefill out")
    heads = list(sample_heads or range(L.hv))
    for j, s in enumerate(slots):
        Sg, Cg = L.get_state(0, s)
        if lengths[j] > 0:
            r = relerr(Sg[heads], ref["S"][j][heads])
            assert r <= tol_p, f"prefill final S seq {j} (len {lengths[j]}): {r:.3e}"
        assert np.array_equal(Cg, ref["convbuf"][j]), f"conv buffer seq {j}"
    S, conv = ref["S"], ref["convbuf"]
    for step in range(decode_steps):
        dinp = L.decode_inputs(list(range(n)), step)
        o = host(L.gpu_decode(0, slots, dinp))
        r = L.oracle_run(0, np.arange(n + 1), dinp, S, conv, head_mask=mask)
        S, conv = r["S"], r["convbuf"]
        check_out(o[:, cols], r["out"][:, cols], L.out, tol_p, f"decode after prefill step {step}")
    assert L.pool.device_status() == 0
    return slots


def test_prefill_tiny_fp32():
    """2 sequences of 32 tokens, 2 q/k and 2 v heads, d = 16, chunk 8, then 8 decode steps (fp32)."""
    L = Layer(1, 2, 2, 16, io="f32", num_slots=4, chunk=8, max_prefill_tokens=64)
    _prefill_then_decode(L, [32, 32], 8, 2e-5)
    L.close()


def test_prefill_ragged_small_fp32():
    """Ragged and empty sequences, lengths shorter than the conv window, GQA ratio 2, d = 32."""
    L = Layer(4, 2, 4, 32, io="f32", num_slots=8, max_prefill_tokens=512)
    _prefill_then_decode(L, [1, 0, 2, 3, 17, 70, 130], 3, 2e-5)
    L.close()


def test_prefill_from_nonzero_state_and_split_calls():
    """Prefill continues from the slot's state: one call over L tokens equals two calls over the halves."""
    L = Layer(5, 2, 4, 64, io="bf16", out="f32", num_slots=4, max_prefill_tokens=256)
    a, b = L.pool.alloc(), L.pool.alloc()
    inp, cu = synth.varlen_inputs(5, 0, [90], 2, 4, 64, 64, "bf16")
    S0 = synth.initial_state(5, 0, 0, 4, 64, 64)
    L.set_state(0, a, S0)
    L.set_state(0, b, S0)
    whole = host(L.gpu_prefill(0, [a], inp, cu))
    first = {k: v[:37] for k, v in inp.items()}
    second = {k: v[37:] for k, v in inp.items()}
    o1 = host(L.gpu_prefill(0, [b], first, [0, 37]))
    o2 = host(L.gpu_prefill(0, [b], second, [0, 53]))
    assert relerr(np.concatenate([o1, o2]), whole) <= PREFILL_TOL
    Sa, Ca = L.get_state(0, a)
    Sb, Cb = L.get_state(0, b)
    assert relerr(Sb, Sa) <= PREFILL_TOL and np.array_equal(Ca, Cb)
    ref = L.oracle_run(0, cu, inp, S0[None].astype(np.float64), np.zeros((1, 3, L.C)))
    check_out(whole, ref["out"], "f32", PREFILL_TOL, "prefill from a random state")
    L.close()


def test_prefill_8_sequences_15998_tokens_35b_layer():
    """Lengths {1,17,300,4095,1024,2048,513,8000} (15 998 tokens), 16/32 heads, d = 128, chunk 64, bf16 io,
    zero initial state; final states handed to 16 decode steps.  Every head of every sequence against
    the oracle."""
    lengths = [1, 17, 300, 4095, 1024, 2048, 513, 8000]
    L = Layer(3, 16, 32, 128, io="bf16", out="bf16", num_slots=16, max_prefill_tokens=sum(lengths))
    _prefill_then_decode(L, lengths, 16, PREFILL_TOL)
    L.close()


def test_prefill_batch_equals_sequences_alone_bitwise():
    """A sequence prefilled inside a varlen batch equals the same sequence prefilled alone, bit for bit."""
    lengths = [5, 300, 64, 129]
    L = Layer(6, 4, 8, 128, io="bf16", num_slots=8, max_prefill_tokens=sum(lengths))
    inp, cu = synth.varlen_inputs(6, 0, lengths, 4, 8, 128, 128, "bf16")
    slots = [L.pool.alloc() for _ in lengths]
    out_b = L.gpu_prefill(0, slots, inp, cu).clone()
    states = [L.get_state(0, s) for s in slots]
    for j, s in enumerate(slots):
        L.pool.recycle(s)
        assert L.pool.alloc() == s
        part = {k: v[cu[j]:cu[j + 1]] for k, v in inp.items()}
        o = L.gpu_prefill(0, [s], part, [0, lengths[j]])
        assert torch.equal(o, out_b[cu[j]:cu[j + 1]]), f"sequence {j} output differs"
        Sg, Cg = L.get_state(0, s)
        assert np.array_equal(Sg, states[j][0]) and np.array_equal(Cg, states[j][1])
    L.close()


def test_prefill_rejects_bad_metadata_on_device():
    """Non-monotone cu_seqlens or a repeated / freed slot id: nothing is written, a status bit is set."""
    L = Layer(3, 2, 2, 16, io="f32", num_slots=4, max_prefill_tokens=64)
    a, b = L.pool.alloc(), L.pool.alloc()
    inp, _ = synth.varlen_inputs(3, 0, [6, 4], 2, 2, 16, 16, "f32")
    d = L.to_dev(inp)
    res = torch.full((10, 32), 3.0, device="cuda")
    for cu, ids, bit in (([0, 7, 6], [a, b], 0x4), ([0, 6, 10], [a, a], 0x2), ([0, 6, 10], [a, 3], 0x2)):
        L.pool.prefill_varlen(0, torch.tensor(cu, dtype=torch.int32, device="cuda"),
                              torch.tensor(ids, dtype=torch.int32, device="cuda"), 2, 10,
                              d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], res)
        assert L.pool.device_status() & bit
        assert torch.all(res == 3.0)
        Sa, Ca = L.get_state(0, a)
        assert not Sa.any() and not Ca.any()
    L.close()


@pytest.mark.parametrize("io,out", [("bf16", "f32"), ("f32", "f32")])
def test_prefill_chunked_d128_ragged(io, out):
    """d = 128 runs the chunked tensor-core kernel: lengths around the 64-token chunk boundary and an
    empty sequence (its slot keeps its state and conv buffer), GQA 2, then 4 decode steps from the
    handed-off states."""
    lengths = [1, 5, 63, 0, 64, 65, 130, 200, 7]
    L = Layer(8, 1, 2, 128, io=io, out=out, num_slots=len(lengths), max_prefill_tokens=sum(lengths))
    n = len(lengths)
    slots = [L.pool.alloc() for _ in range(n)]
    inp, cu = synth.varlen_inputs(8, 0, lengths, 1, 2, 128, 128, io)
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, np.zeros((n, 2, 128, 128)), np.zeros((n, 3, L.C)))
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    print(f"chunked d128 io={io}: out {r_out:.2e}, S {r_S:.2e}")
    assert r_out <= PREFILL_TOL and r_S <= PREFILL_TOL
    for j, s in enumerate(slots):
        assert np.array_equal(L.get_state(0, s)[1], ref["convbuf"][j])
    S, conv = ref["S"], ref["convbuf"]
    for step in range(4):
        dinp = L.decode_inputs(list(range(n)), step)
        og = host(L.gpu_decode(0, slots, dinp))
        r = L.oracle_run(0, np.arange(n + 1), dinp, S, conv)
        S, conv = r["S"], r["convbuf"]
        assert relerr(og, r["out"]) <= PREFILL_TOL
    assert L.pool.device_status() == 0
    L.close()


def test_prefill_chunked_d128_random_state_weak_decay_split():
    """d = 128 from a random N(0, 0.1) state, with A_log shifted so the decay is weak (the state matters
    across chunks), one call vs two calls split at a non-chunk boundary, and the oracle."""
    hqk, hv, d = 2, 4, 128
    L = Layer(12, hqk, hv, d, io="bf16", out="f32", num_slots=4, max_prefill_tokens=512)
    p = L.params[0]
    p["A_log"] = (p["A_log"] - 4.0).astype(np.float32)  # alpha ~ exp(-e^{A_log} softplus(a)) closer to 1
    L.pool.layer_params(0, torch.from_numpy(p["conv_w"]), torch.from_numpy(p["A_log"]),
                        torch.from_numpy(p["dt_bias"]), torch.from_numpy(p["norm_w"]))
    a, b = L.pool.alloc(), L.pool.alloc()
    inp, cu = synth.varlen_inputs(12, 0, [300], hqk, hv, d, d, "bf16")
    S0 = synth.initial_state(12, 0, 0, hv, d, d)
    L.set_state(0, a, S0)
    L.set_state(0, b, S0)
    whole = host(L.gpu_prefill(0, [a], inp, cu))
    o1 = host(L.gpu_prefill(0, [b], {k: v[:100] for k, v in inp.items()}, [0, 100]))
    o2 = host(L.gpu_prefill(0, [b], {k: v[100:] for k, v in inp.items()}, [0, 200]))
    ref = L.oracle_run(0, cu, inp, S0[None].astype(np.float64), np.zeros((1, 3, L.C)))
    r1 = relerr(whole, ref["out"])
    r2 = relerr(np.concatenate([o1, o2]), ref["out"])
    rS = relerr(L.get_state(0, a)[0], ref["S"][0])
    rS2 = relerr(L.get_state(0, b)[0], ref["S"][0])
    print(f"chunked weak decay: out {r1:.2e} split {r2:.2e} S {rS:.2e} split S {rS2:.2e}")
    assert max(r1, r2, rS, rS2) <= PREFILL_TOL
    L.close()


@pytest.mark.parametrize("W", [2, 6])
def test_prefill_chunked_d128_conv_width_and_buffer(W):
    """d = 128 with conv width W = 2 (fewer taps than the 4-tap fast path) and W = 6 (the 8-tap path), from
    non-zero slot conv buffers and N(0, 0.1) states: the chunked pre-pass takes the W-1 positions before each
    sequence from its slot's conv buffer, including sequences shorter than W-1; the buffers then advance."""
    lengths = [1, 2, 70, 129, 5]
    n = len(lengths)
    L = Layer(14, 1, 2, 128, conv_w=W, io="bf16", out="f32", num_slots=8, max_prefill_tokens=sum(lengths))
    slots = [L.pool.alloc() for _ in range(n)]
    S0 = np.stack([synth.initial_state(14, 0, j, 2, 128, 128) for j in range(n)]).astype(np.float64)
    conv0 = np.stack([synth.initial_convbuf(14, 0, j, W, L.C, "bf16") for j in range(n)]).astype(np.float64)
    for j, s in enumerate(slots):
        L.set_state(0, s, S0[j], conv0[j])
    inp, cu = synth.varlen_inputs(14, 0, lengths, 1, 2, 128, 128, "bf16")
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, S0, conv0)
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    print(f"chunked d128 W={W}: out {r_out:.2e}, S {r_S:.2e}")
    assert r_out <= PREFILL_TOL and r_S <= PREFILL_TOL
    for j, s in enumerate(slots):
        assert np.array_equal(L.get_state(0, s)[1], ref["convbuf"][j])
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("hqk,hv", [(2, 2), (1, 4)])
def test_prefill_chunked_d128_gqa_ratios(hqk, hv):
    """d = 128 with GQA ratio 1 and 4: the pre-pass shares a q/k head's conv, norms and [K; Q] x K^T between
    the ratio's v-heads, which it takes one after the other; a random state and conv buffer to start from."""
    lengths = [70, 3, 129]
    n = len(lengths)
    L = Layer(15, hqk, hv, 128, io="bf16", out="f32", num_slots=4, max_prefill_tokens=sum(lengths))
    slots = [L.pool.alloc() for _ in range(n)]
    S0 = np.stack([synth.initial_state(15, 0, j, hv, 128, 128) for j in range(n)]).astype(np.float64)
    conv0 = np.stack([synth.initial_convbuf(15, 0, j, 4, L.C, "bf16") for j in range(n)]).astype(np.float64)
    for j, s in enumerate(slots):
        L.set_state(0, s, S0[j], conv0[j])
    inp, cu = synth.varlen_inputs(15, 0, lengths, hqk, hv, 128, 128, "bf16")
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, S0, conv0)
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    print(f"chunked d128 GQA {hv // hqk}: out {r_out:.2e}, S {r_S:.2e}")
    assert r_out <= PREFILL_TOL and r_S <= PREFILL_TOL
    for j, s in enumerate(slots):
        assert np.array_equal(L.get_state(0, s)[1], ref["convbuf"][j])
    assert L.pool.device_status() == 0
    L.close()


@pytest.mark.parametrize("d,chunk,io", [(16, 8, "f32"), (32, 16, "f32"), (32, 32, "bf16"), (64, 64, "f32"),
                                        (64, 16, "bf16")])
def test_prefill_chunked_small_d(d, chunk, io):
    """d < 128 runs the chunked (WY) form in fp32 on the CUDA cores with the pool's chunk length: lengths
    around the chunk boundary, an empty sequence, GQA 2, from random states and conv buffers, against the
    oracle; then 3 decode steps from the handed-off states."""
    lengths = [1, chunk - 1, chunk, chunk + 1, 0, 3 * chunk + 5, 2]
    n = len(lengths)
    L = Layer(16, 2, 4, d, io=io, out="f32", num_slots=n, chunk=chunk, max_prefill_tokens=sum(lengths))
    slots = [L.pool.alloc() for _ in range(n)]
    S0 = np.stack([synth.initial_state(16, 0, j, 4, d, d) for j in range(n)]).astype(np.float64)
    conv0 = np.stack([synth.initial_convbuf(16, 0, j, 4, L.C, io) for j in range(n)]).astype(np.float64)
    for j, s in enumerate(slots):
        L.set_state(0, s, S0[j], conv0[j])
    inp, cu = synth.varlen_inputs(16, 0, lengths, 2, 4, d, d, io)
    o = host(L.gpu_prefill(0, slots, inp, cu))
    ref = L.oracle_run(0, cu, inp, S0, conv0)
    r_out = relerr(o, ref["out"])
    r_S = max(relerr(L.get_state(0, s)[0], ref["S"][j]) for j, s in enumerate(slots))
    print(f"chunked d={d} chunk={chunk} io={io}: out {r_out:.2e}, S {r_S:.2e}")
    assert r_out <= 2e-5 and r_S <= 2e-5
    for j, s in enumerate(slots):
        assert np.array_equal(L.get_state(0, s)[1], ref["convbuf"][j])
    S, conv = ref["S"], ref["convbuf"]
    for step in range(3):
        dinp = L.decode_inputs(list(range(n)), step)
        og = host(L.gpu_decode(0, slots, dinp))
        r = L.oracle_run(0, np.arange(n + 1), dinp, S, conv)
        S, conv = r["S"], r["convbuf"]
        assert relerr(og, r["out"]) <= 2e-5
    assert L.pool.device_status() == 0
    L.close()
