"""The continuous-batching and long-context workloads at full size on the GPU.

Mixed continuous batch with slot reuse: a 512-slot pool of the 35B-A3B-shaped layer; every
iteration finishes 2 random sequences (their slots are recycled), admits 2 new 8192-token
prompts into the recycled slots and decodes 32 random active sequences one step; 50
iterations.  No contamination: every sequence's outputs equal an isolated run of the same
sequence (same kernels, alone in a fresh pool) bit for bit, and eight of the 32 heads of one
sequence match the fp64 oracle.

Long context: one 80 000-token prefill (1 250 chunks), then decode at m = 256 on each of 30
stacked layer pools (30 x 256 slots, 16.1 GB of fp32 state); eight of the 32 heads and sampled
slots against the oracle.  Inputs are drawn on the device by the seeded generator (too large for the host
generator); the oracle runs per sampled head on the head's slice of the inputs.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_rule_gb300 import synth
from gdn_harness import DECODE_TOL, PREFILL_TOL, Layer, check_out, host, oracle_heads, relerr

pytestmark = pytest.mark.gpu

HQK, HV, D = 16, 32, 128


def _cat(parts):
    return {k: torch.cat([p[k] for p in parts]) for k in parts[0]}


def _host_inputs(inp):
    return {k: host(v) for k, v in inp.items()}


def test_mixed_continuous_batch_with_slot_reuse():
    PL, W = 8192, 4
    L = Layer(4, HQK, HV, D, io="bf16", out="bf16", num_slots=512, max_prefill_tokens=2 * PL)
    rng = synth.rng(4)
    active = {}  # slot -> [sequence id, decode steps done]
    rec_pre, rec_dec = {}, {}
    next_id = 0

    def admit(k):
        nonlocal next_id
        new = [(L.pool.alloc(), next_id + j) for j in range(k)]
        next_id += k
        inp = _cat([synth.device_token_inputs(4, 0, sid, PL, HQK, HV, D, D, "bf16") for _, sid in new])
        out = L.gpu_prefill(0, [s for s, _ in new], inp, np.arange(k + 1) * PL)
        for j, (s, sid) in enumerate(new):
            active[s] = [sid, 0]
            rec_pre[sid] = out[j * PL:(j + 1) * PL].clone()
            rec_dec[sid] = []

    for _ in range(20):  # 40 sequences in flight before the schedule starts
        admit(2)
    for it in range(50):
        for s in rng.choice(sorted(active), size=2, replace=False):
            del active[int(s)]
            L.pool.recycle(int(s))
        admit(2)
        slots = [int(x) for x in rng.choice(sorted(active), size=32, replace=False)]
        inp = _cat([synth.device_token_inputs(4, 0, active[s][0], 1, HQK, HV, D, D, "bf16", tag="decode",
                                              sub=active[s][1]) for s in slots])
        out = L.gpu_decode(0, slots, inp)
        for j, s in enumerate(slots):
            rec_dec[active[s][0]].append(out[j].clone())
            active[s][1] += 1
    assert L.pool.device_status() == 0
    L.close()

    # isolated runs: one sequence at a time in a fresh one-slot pool
    I = Layer(4, HQK, HV, D, io="bf16", out="bf16", num_slots=1, max_prefill_tokens=PL)
    for sid in sorted(rec_pre):
        s = I.pool.alloc()
        inp = synth.device_token_inputs(4, 0, sid, PL, HQK, HV, D, D, "bf16")
        o = I.gpu_prefill(0, [s], inp, [0, PL])
        assert torch.equal(o, rec_pre[sid]), f"sequence {sid}: prefill differs from its isolated run"
        for step, row in enumerate(rec_dec[sid]):
            dinp = synth.device_token_inputs(4, 0, sid, 1, HQK, HV, D, D, "bf16", tag="decode", sub=step)
            od = I.gpu_decode(0, [s], dinp)
            assert torch.equal(od[0], row), f"sequence {sid}: decode step {step} differs from its isolated run"
        I.pool.recycle(s)
    # the oracle on eight heads of the sequence that decoded the most steps
    sid = max(rec_dec, key=lambda k: len(rec_dec[k]))
    inp = synth.device_token_inputs(4, 0, sid, PL, HQK, HV, D, D, "bf16")
    heads = [0, 1, 3, 12, 17, 22, 30, 31]
    C = I.C
    ref = oracle_heads(I, 0, [0, PL], inp, np.zeros((1, HV, D, D)), np.zeros((1, W - 1, C)), heads)
    got = host(rec_pre[sid])
    for h in heads:
        check_out(got[:, h * D:(h + 1) * D], ref[h][0], "bf16", PREFILL_TOL, f"seq {sid} head {h} prefill")
    I.close()


def test_long_prefill_80k_then_30_layer_decode():
    T, NL, M, W = 80000, 30, 256, 4
    L = Layer(5, HQK, HV, D, io="bf16", out="bf16", num_slots=M, num_layers=NL, layer_ids=range(NL),
              max_prefill_tokens=T)
    slots = [L.pool.alloc() for _ in range(M)]
    g = torch.Generator(device="cuda").manual_seed(55)
    for layer in range(1, NL):  # layer 0 starts from zero states (the prefill's), the others random
        blk = L.pool.state_block(layer)
        blk.copy_(torch.randn(blk.shape, generator=g, device="cuda") * (0.1 ** 0.5))
    torch.cuda.synchronize()

    inp = synth.device_token_inputs(5, 0, 0, T, HQK, HV, D, D, "bf16")
    out = L.gpu_prefill(0, [slots[0]], inp, [0, T])
    heads = [0, 1, 9, 14, 17, 22, 30, 31]
    ref = oracle_heads(L, 0, [0, T], inp, np.zeros((1, HV, D, D)), np.zeros((1, W - 1, L.C)), heads)
    got = host(out)
    S0, C0 = L.get_state(0, slots[0])
    for h in heads:
        check_out(got[:, h * D:(h + 1) * D], ref[h][0], "bf16", PREFILL_TOL, f"80k prefill head {h}")
        assert relerr(S0[h], ref[h][1][0]) <= PREFILL_TOL, f"80k prefill final S head {h}"
    x = np.concatenate([host(inp["q"][-(W - 1):]), host(inp["k"][-(W - 1):]), host(inp["v"][-(W - 1):])], axis=1)
    assert np.array_equal(C0, x), "conv buffer after the 80k prefill holds the last W-1 raw inputs"

    # one decode step at m = 256 on every layer; sampled (layer, slot) pairs against the oracle
    samples = {0: [slots[0], slots[200]], 17: [slots[5]], 29: [slots[255]]}
    before = {(ly, s): L.get_state(ly, s) for ly, ss in samples.items() for s in ss}
    dinp = {ly: synth.device_token_inputs(5, ly, 1000, M, HQK, HV, D, D, "bf16", tag="decode") for ly in range(NL)}
    outs = {ly: L.gpu_decode(ly, slots, dinp[ly]) for ly in range(NL)}
    for ly, ss in samples.items():
        hd = _host_inputs(dinp[ly])
        for s in ss:
            j = slots.index(s)
            one = {k: v[j:j + 1] for k, v in hd.items()}
            Sb, Cb = before[(ly, s)]
            r = L.oracle_run(ly, [0, 1], one, Sb[None], Cb[None])
            check_out(host(outs[ly][j:j + 1]), r["out"], "bf16", DECODE_TOL, f"layer {ly} slot {s} decode")
            Sa, _ = L.get_state(ly, s)
            assert relerr(Sa, r["S"][0]) <= DECODE_TOL, f"layer {ly} slot {s} decode state"
    assert L.pool.device_status() == 0
    L.close()
