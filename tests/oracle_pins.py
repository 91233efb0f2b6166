"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
the oracle disagrees with what the definitions, the library routines or the
hand-worked examples fix.  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` plants mistakes in copies of the oracle's C source
and checks that every planted mistake fails at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


def _close(a, b, tol, what):
    r = _rel(a, b)
    assert r <= tol, f"{what}: relative error {r:.3e} > {tol:.1e}"


def _unit_rows(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


# ---------------------------------------------------------------- conv ----

def _torch_conv_silu(x, w, buf):
    """Depthwise conv via torch conv1d over [buffer; x] without padding, then SiLU."""
    L, C = x.shape
    W = w.shape[1]
    full = np.concatenate([buf, x], axis=0)  # [(W-1)+L][C]
    inp = torch.from_numpy(full.T.copy())[None]  # [1][C][len]
    wt = torch.from_numpy(w.copy())[:, None, :]  # [C][1][W]
    y = F.conv1d(inp, wt, groups=C)[0].T  # [L][C]
    return F.silu(y).numpy(), full[-(W - 1):].copy() if W > 1 else np.zeros((0, C))


def pin_conv_zero_buffer(o):
    """Zero buffer: equals torch conv1d(groups=C, padding=W-1) truncated to the causal part, then SiLU."""
    rng = np.random.default_rng(1)
    for L, C, W in ((9, 5, 4), (1, 3, 4), (6, 4, 2), (5, 2, 1)):
        x = rng.standard_normal((L, C))
        w = rng.standard_normal((C, W))
        y, _ = o.conv_silu(x, w, np.zeros((max(W - 1, 0), C)))
        ref = F.conv1d(torch.from_numpy(x.T.copy())[None], torch.from_numpy(w)[:, None, :], padding=W - 1,
                       groups=C)[0, :, :L].T
        _close(y, F.silu(ref).numpy(), 1e-13, f"conv zero-buffer L={L} C={C} W={W}")


def pin_conv_with_buffer(o):
    """Non-zero buffer, including sequences shorter than W-1: conv over [buffer; x], new buffer = last W-1 rows."""
    rng = np.random.default_rng(2)
    for L, C, W in ((7, 6, 4), (1, 6, 4), (2, 6, 4), (3, 6, 4), (4, 3, 3)):
        x = rng.standard_normal((L, C))
        w = rng.standard_normal((C, W))
        buf = rng.standard_normal((W - 1, C))
        y, nb = o.conv_silu(x, w, buf)
        ry, rb = _torch_conv_silu(x, w, buf)
        _close(y, ry, 1e-13, f"conv with buffer L={L}")
        assert np.array_equal(nb, rb), f"conv buffer update L={L}"


def pin_conv_golden(o):
    """Hand-worked conv value (tap W-1 multiplies the current token)."""
    for line in open(os.path.join(GOLDEN, "gates_conv_worked_example.txt")):
        if line.startswith("conv "):
            vals = [float(t) for t in line.split()[1:]]
            w = np.array(vals[0:4])[None, :]
            buf = np.array(vals[4:7])[:, None]
            x = np.array([[vals[7]]])
            pre = vals[8]
            y, nb = o.conv_silu(x, w, buf)
            _close(y[0, 0], pre / (1.0 + math.exp(-pre)), 1e-15, "conv golden")
            assert np.array_equal(nb[:, 0], np.array([vals[5], vals[6], vals[7]])), "conv golden buffer"


# ------------------------------------------------------------ L2 / gates ----

def pin_l2norm(o):
    """eps = 0 equals torch F.normalize; eps = 1e-6 stays within 1e-6 of it; a zero vector stays zero."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 16)) * 3.0
    ref = F.normalize(torch.from_numpy(x), dim=-1).numpy()
    _close(o.l2norm(x, eps=0.0), ref, 1e-15, "l2norm eps=0")
    _close(o.l2norm(x, eps=1e-6), ref, 1e-6, "l2norm eps=1e-6")
    assert np.all(o.l2norm(np.zeros((2, 8)), eps=1e-6) == 0.0), "l2norm of zero"


def pin_gates_torch(o):
    """g = -exp(A_log)*softplus(a+dt_bias) and beta = sigmoid(b) against torch, including large |a|."""
    rng = np.random.default_rng(4)
    a = np.concatenate([rng.standard_normal(50) * 3, [30.0, -30.0, 700.0, -700.0, 0.0]])
    b = np.concatenate([rng.standard_normal(50) * 3, [30.0, -30.0, 700.0, -700.0, 0.0]])
    for A_log, dtb in ((0.3, 0.0), (math.log(16.0), 0.5), (0.0, -1.25)):
        g, beta = o.gates(a, b, A_log, dtb)
        ta = torch.from_numpy(a)
        rg = (-math.exp(A_log) * F.softplus(ta + dtb, threshold=750.0)).numpy()
        rb = torch.sigmoid(torch.from_numpy(b)).numpy()
        assert np.allclose(g, rg, rtol=1e-14, atol=0), f"gates g A_log={A_log}"
        assert np.allclose(beta, rb, rtol=1e-14, atol=1e-300), f"gates beta A_log={A_log}"


def pin_gates_golden(o):
    """Hand-worked gate values."""
    for line in open(os.path.join(GOLDEN, "gates_conv_worked_example.txt")):
        if line.startswith("gate "):
            A_log, a, dtb, b, alpha, beta = (float(t) for t in line.split()[1:])
            g, bt = o.gates([a], [b], A_log, dtb)
            _close(math.exp(g[0]), alpha, 1e-14, "golden alpha")
            _close(bt[0], beta, 1e-15, "golden beta")


# ------------------------------------------------------------ delta rule ----

def _golden_tokens():
    toks, S0, cur = [], None, None
    for line in open(os.path.join(GOLDEN, "delta_worked_example.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, val = (s.strip() for s in line.split("="))
        vals = np.array([float(t) for t in val.split()])
        if key == "S0":
            S0 = vals.reshape(2, 2)
        elif key == "alpha":
            cur = {"alpha": vals[0]}
            toks.append(cur)
        else:
            cur[key] = vals if key != "beta" else vals[0]
    return S0, toks


def pin_delta_golden(o):
    """The hand-worked 2x2 example: o and S after every token."""
    S0, toks = _golden_tokens()
    S = S0
    for i, t in enumerate(toks):
        g = np.array([math.log(t["alpha"])])
        out, S = o.delta_recurrent(t["q"][None], t["k"][None], t["v"][None], g, np.array([t["beta"]]), S)
        _close(out[0], t["o"], 1e-14, f"golden o token {i + 1}")
        _close(S.ravel(), t["S"], 1e-14, f"golden S token {i + 1}")


def pin_pure_decay(o):
    """beta = 0: S_t = alpha_t S_{t-1} exactly, so o_t = (prod_{s<=t} alpha_s) S0 q_t."""
    rng = np.random.default_rng(5)
    L, dk, dv = 6, 5, 3
    q, k, v = rng.standard_normal((L, dk)), _unit_rows(rng, L, dk), rng.standard_normal((L, dv))
    g = -rng.uniform(0.05, 2.0, L)
    S0 = rng.standard_normal((dv, dk))
    out, S = o.delta_recurrent(q, k, v, g, np.zeros(L), S0)
    cum = np.exp(np.cumsum(g))
    for t in range(L):
        _close(out[t], cum[t] * (S0 @ q[t]), 1e-13, f"pure decay o_{t}")
    _close(S, cum[-1] * S0, 1e-13, "pure decay S")


def pin_write_then_read(o):
    """alpha = 1, beta = 1, unit k: the state read back along k_t returns v_t."""
    rng = np.random.default_rng(6)
    L, dk, dv = 8, 6, 4
    k = _unit_rows(rng, L, dk)
    v = rng.standard_normal((L, dv))
    S = rng.standard_normal((dv, dk))
    for t in range(L):
        _, S = o.delta_recurrent(k[t:t + 1], k[t:t + 1], v[t:t + 1], np.zeros(1), np.ones(1), S)
        _close(S @ k[t], v[t], 1e-13, f"write-then-read t={t}")


def pin_associative_recall(o):
    """Orthonormal keys, alpha = beta = 1: after writing all pairs, querying k_j returns v_j for every j."""
    rng = np.random.default_rng(7)
    dk, dv, n = 6, 3, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :n].T.copy()
    v = rng.standard_normal((n, dv))
    S0 = rng.standard_normal((dv, dk))
    _, S = o.delta_recurrent(k, k, v, np.zeros(n), np.ones(n), S0)
    for j in range(n):
        out, _ = o.delta_recurrent(k[j:j + 1], np.zeros((1, dk)), np.zeros((1, dv)), np.zeros(1), np.zeros(1), S)
        _close(out[0], v[j], 1e-13, f"associative recall j={j}")


def pin_reset(o):
    """alpha = 0 (g = -inf): the old state vanishes and S_t = beta_t v_t k_t^T."""
    rng = np.random.default_rng(8)
    dk, dv = 4, 3
    k = _unit_rows(rng, 1, dk)
    v = rng.standard_normal((1, dv))
    q = rng.standard_normal((1, dk))
    beta = np.array([0.37])
    S0 = rng.standard_normal((dv, dk)) * 10
    out, S = o.delta_recurrent(q, k, v, np.array([-np.inf]), beta, S0)
    _close(S, beta[0] * np.outer(v[0], k[0]), 1e-15, "reset S")
    _close(out[0], beta[0] * v[0] * (k[0] @ q[0]), 1e-15, "reset o")


def brute_force_states(S0, q, k, v, g, beta):
    """Unrolled closed form with explicit transition matrices M_t = alpha_t (I - beta_t k_t k_t^T):
    S_t = S0 M_1...M_t + sum_{j<=t} beta_j v_j k_j^T M_{j+1}...M_t, and o_t = S_t q_t."""
    L, dk = k.shape
    M = [math.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) for t in range(L)]
    outs, states = [], []
    for t in range(L):
        P = np.eye(dk)
        for s in range(t + 1):
            P = P @ M[s]
        St = S0 @ P
        for j in range(t + 1):
            Pj = np.eye(dk)
            for s in range(j + 1, t + 1):
                Pj = Pj @ M[s]
            St = St + beta[j] * np.outer(v[j], k[j]) @ Pj
        states.append(St)
        outs.append(St @ q[t])
    return np.array(outs), states


def pin_brute_force(o):
    """Tiny shapes (d <= 4, L <= 6): every o_t and the final S equal the unrolled closed form."""
    rng = np.random.default_rng(9)
    for L, dk, dv in ((6, 4, 3), (5, 3, 3), (4, 2, 4), (1, 4, 2)):
        q, k, v = rng.standard_normal((L, dk)), _unit_rows(rng, L, dk), rng.standard_normal((L, dv))
        g = -rng.uniform(0.0, 1.5, L)
        beta = rng.uniform(0.05, 0.95, L)
        S0 = rng.standard_normal((dv, dk))
        out, S = o.delta_recurrent(q, k, v, g, beta, S0)
        ro, rs = brute_force_states(S0, q, k, v, g, beta)
        _close(out, ro, 1e-12, f"brute force o L={L}")
        _close(S, rs[-1], 1e-12, f"brute force S L={L}")


def pin_chunked_equals_recurrent(o):
    """The chunked WY form reaches the recurrent result to 1e-12 for chunk 1, 3, 8, 64 and ragged L."""
    rng = np.random.default_rng(10)
    for L, dk, dv, strong in ((70, 16, 8, False), (23, 8, 8, True), (9, 4, 6, False), (64, 8, 4, True)):
        q, k, v = rng.standard_normal((L, dk)), _unit_rows(rng, L, dk), rng.standard_normal((L, dv))
        g = -rng.uniform(0.5, 12.0, L) if strong else -rng.uniform(0.0, 0.2, L)
        beta = rng.uniform(0.0, 1.0, L)
        S0 = rng.standard_normal((dv, dk))
        ro, rs = o.delta_recurrent(q, k, v, g, beta, S0)
        for chunk in (1, 3, 8, 64):
            co, cs = o.delta_chunked(q, k, v, g, beta, S0, chunk)
            _close(co, ro, 1e-12, f"chunked o L={L} chunk={chunk}")
            _close(cs, rs, 1e-12, f"chunked S L={L} chunk={chunk}")


# ---------------------------------------------------------------- norm ----

def pin_gated_rmsnorm(o):
    """Equals torch F.rms_norm(o, [dv], w, eps) * F.silu(z)."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 16)) * 0.3
    z = rng.standard_normal((5, 16)) * 2
    w = rng.uniform(0.5, 1.5, 16)
    for eps in (1e-6, 0.0):
        y = o.gated_rmsnorm(x, z, w, eps)
        ref = F.rms_norm(torch.from_numpy(x), (16,), torch.from_numpy(w), eps=eps) * F.silu(torch.from_numpy(z))
        _close(y, ref.numpy(), 1e-14, f"gated rmsnorm eps={eps}")


# ---------------------------------------------------------------- layer ----

def _rand_layer_case(rng, hqk, hv, d, W, lengths, S_scale=0.3):
    C = 2 * hqk * d + hv * d
    T = int(sum(lengths))
    case = {
        "shape": {"hqk": hqk, "hv": hv, "dk": d, "dv": d, "conv_w": W, "l2_eps": 1e-6, "norm_eps": 1e-6},
        "cu": np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
        "q": rng.standard_normal((T, hqk * d)), "k": rng.standard_normal((T, hqk * d)),
        "v": rng.standard_normal((T, hv * d)), "z": rng.standard_normal((T, hv * d)),
        "a": rng.standard_normal((T, hv)), "b": rng.standard_normal((T, hv)),
        "conv_w": rng.standard_normal((C, W)) * 0.5, "A_log": rng.uniform(0, math.log(16), hv) - 1.5,
        "dt_bias": rng.standard_normal(hv) * 0.1, "norm_w": rng.uniform(0.5, 1.5, d),
        "S": rng.standard_normal((len(lengths), hv, d, d)) * S_scale,
        "convbuf": rng.standard_normal((len(lengths), W - 1, C)),
    }
    return case


def _run_layer(o, c, **kw):
    return o.layer(c["shape"], c["cu"], c["q"], c["k"], c["v"], c["a"], c["b"], c["z"], c["conv_w"], c["A_log"],
                   c["dt_bias"], c["norm_w"], c["S"], c["convbuf"], **kw)


def pin_layer_composition(o):
    """Whole layer equals the library routines composed in the order of the definition:
    torch conv1d + SiLU, F.normalize, dk^-1/2, torch softplus/sigmoid gates, the brute-force
    closed form of the recurrence, F.rms_norm * SiLU(z).  GQA ratio 2, two sequences."""
    rng = np.random.default_rng(12)
    hqk, hv, d, W = 1, 2, 4, 4
    r = hv // hqk
    c = _rand_layer_case(rng, hqk, hv, d, W, [5, 3])
    c["shape"]["l2_eps"] = 0.0
    res = _run_layer(o, c, want_o=True)
    Cq = hqk * d
    for s in range(2):
        t0, t1 = c["cu"][s], c["cu"][s + 1]
        x = np.concatenate([c["q"][t0:t1], c["k"][t0:t1], c["v"][t0:t1]], axis=1)
        y, nb = _torch_conv_silu(x, c["conv_w"], c["convbuf"][s])
        assert np.array_equal(res["convbuf"][s], nb), "layer conv buffer"
        qn = F.normalize(torch.from_numpy(y[:, :Cq].reshape(-1, hqk, d)), dim=-1).numpy() / math.sqrt(d)
        kn = F.normalize(torch.from_numpy(y[:, Cq:2 * Cq].reshape(-1, hqk, d)), dim=-1).numpy()
        vv = y[:, 2 * Cq:].reshape(-1, hv, d)
        for h in range(hv):
            ta = torch.from_numpy(c["a"][t0:t1, h] + c["dt_bias"][h])
            g = (-math.exp(c["A_log"][h]) * F.softplus(ta)).numpy()
            beta = torch.sigmoid(torch.from_numpy(c["b"][t0:t1, h])).numpy()
            ro, rs = brute_force_states(c["S"][s, h], qn[:, h // r], kn[:, h // r], vv[:, h], g, beta)
            _close(res["o"][t0:t1, h * d:(h + 1) * d], ro, 1e-12, f"layer o seq {s} head {h}")
            _close(res["S"][s, h], rs[-1], 1e-12, f"layer S seq {s} head {h}")
            yr = F.rms_norm(torch.from_numpy(ro), (d,), torch.from_numpy(c["norm_w"]), eps=1e-6) * \
                F.silu(torch.from_numpy(c["z"][t0:t1, h * d:(h + 1) * d]))
            _close(res["out"][t0:t1, h * d:(h + 1) * d], yr.numpy(), 1e-12, f"layer out seq {s} head {h}")


def pin_gqa_is_head_repeat(o):
    """GQA ratio r: v-head h reads q/k head h // r, i.e. the same as repeating each q/k head r times
    (contiguous groups, with the conv weights of the q/k channels repeated alike) at ratio 1."""
    rng = np.random.default_rng(13)
    hqk, hv, d, W = 2, 4, 4, 4
    r = hv // hqk
    c = _rand_layer_case(rng, hqk, hv, d, W, [6])
    res = _run_layer(o, c)
    Cq = hqk * d
    rep = dict(c)
    rep["shape"] = dict(c["shape"], hqk=hv)
    rep["q"] = np.repeat(c["q"].reshape(-1, hqk, d), r, axis=1).reshape(-1, hv * d)
    rep["k"] = np.repeat(c["k"].reshape(-1, hqk, d), r, axis=1).reshape(-1, hv * d)
    wq = np.repeat(c["conv_w"][:Cq].reshape(hqk, d, W), r, axis=0).reshape(-1, W)
    wk = np.repeat(c["conv_w"][Cq:2 * Cq].reshape(hqk, d, W), r, axis=0).reshape(-1, W)
    rep["conv_w"] = np.concatenate([wq, wk, c["conv_w"][2 * Cq:]], axis=0)
    bq = np.repeat(c["convbuf"][:, :, :Cq].reshape(1, W - 1, hqk, d), r, axis=2).reshape(1, W - 1, -1)
    bk = np.repeat(c["convbuf"][:, :, Cq:2 * Cq].reshape(1, W - 1, hqk, d), r, axis=2).reshape(1, W - 1, -1)
    rep["convbuf"] = np.concatenate([bq, bk, c["convbuf"][:, :, 2 * Cq:]], axis=2)
    rr = _run_layer(o, rep)
    _close(res["out"], rr["out"], 1e-13, "gqa out")
    _close(res["S"], rr["S"], 1e-13, "gqa S")


def pin_split_call(o):
    """A sequence run in two calls (state and conv buffer carried over) equals one call, for every
    split point, which also covers prefill(L) followed by a one-token decode equalling prefill(L+1)."""
    rng = np.random.default_rng(14)
    c = _rand_layer_case(rng, 1, 2, 4, 4, [7])
    whole = _run_layer(o, c)
    for cut in (1, 2, 3, 5, 6):
        a = dict(c, cu=np.array([0, cut], dtype=np.int64))
        for key in ("q", "k", "v", "z", "a", "b"):
            a[key] = c[key][:cut]
        ra = _run_layer(o, a)
        b = dict(c, cu=np.array([0, 7 - cut], dtype=np.int64), S=ra["S"], convbuf=ra["convbuf"])
        for key in ("q", "k", "v", "z", "a", "b"):
            b[key] = c[key][cut:]
        rb = _run_layer(o, b)
        _close(np.concatenate([ra["out"], rb["out"]]), whole["out"], 1e-13, f"split out cut={cut}")
        _close(rb["S"], whole["S"], 1e-13, f"split S cut={cut}")
        assert np.array_equal(rb["convbuf"], whole["convbuf"]), f"split conv buffer cut={cut}"


def pin_layer_chunked(o):
    """The layer run with the chunked form equals the recurrent definition (fp64, 1e-12)."""
    rng = np.random.default_rng(15)
    c = _rand_layer_case(rng, 2, 4, 8, 4, [1, 17, 30])
    rec = _run_layer(o, c)
    for chunk in (3, 8):
        ch = _run_layer(o, c, chunk=chunk)
        _close(ch["out"], rec["out"], 1e-12, f"layer chunked out chunk={chunk}")
        _close(ch["S"], rec["S"], 1e-12, f"layer chunked S chunk={chunk}")


def pin_head_mask(o):
    """head_mask computes only the selected heads, with the same values as the full call."""
    rng = np.random.default_rng(16)
    c = _rand_layer_case(rng, 2, 4, 4, 4, [5, 2])
    full = _run_layer(o, c)
    mask = np.array([0, 1, 0, 1], dtype=np.int32)
    part = _run_layer(o, c, head_mask=mask)
    for h in range(4):
        sl = slice(h * 4, (h + 1) * 4)
        if mask[h]:
            assert np.array_equal(part["out"][:, sl], full["out"][:, sl]), "head mask out"
            assert np.array_equal(part["S"][:, h], full["S"][:, h]), "head mask S"
        else:
            assert np.array_equal(part["S"][:, h], c["S"][:, h]), "masked head S untouched"


# --------------------------------------------------------- projections ----

def pin_in_proj_selectors_and_split(o):
    """Weight rows that are unit vectors copy input columns: row j of segment s selects input
    feature f(s, j), so every output column is a known column of x; the six outputs come out in
    the order q | k | v | z | a | b with their widths (a transposed weight or a shifted split
    fails here)."""
    hqk, hv, dk, dv, hidden, T = 2, 4, 8, 8, 64, 5
    widths = [hqk * dk, hqk * dk, hv * dv, hv * dv, hv, hv]
    N = sum(widths)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, hidden))
    sel = (np.arange(N) * 7 + 3) % hidden  # output column n copies input feature sel[n]
    w = np.zeros((N, hidden))
    w[np.arange(N), sel] = 1.0
    r = o.in_proj(x, w, hqk, hv, dk, dv)
    c = 0
    for name, wd in zip(("q", "k", "v", "z", "a", "b"), widths):
        assert r[name].shape == (T, wd), name
        assert np.array_equal(r[name], x[:, sel[c:c + wd]]), name
        c += wd


def pin_in_proj_is_linear_rows(o):
    """Each output row depends on its input row only, linearly: scaling row t of x by s scales row
    t of every output and leaves the others unchanged."""
    hqk, hv, dk, dv, hidden, T = 1, 2, 8, 8, 64, 4
    N = 2 * hqk * dk + 2 * hv * dv + 2 * hv
    rng = np.random.default_rng(6)
    x = rng.standard_normal((T, hidden))
    w = rng.standard_normal((N, hidden))
    r0 = o.in_proj(x, w, hqk, hv, dk, dv)
    x2 = x.copy()
    x2[2] *= -3.0
    r1 = o.in_proj(x2, w, hqk, hv, dk, dv)
    for name in r0:
        _close(r1[name][2], -3.0 * r0[name][2], 1e-14, name)
        assert np.array_equal(np.delete(r1[name], 2, 0), np.delete(r0[name], 2, 0)), name


def pin_out_proj_one_hot(o):
    """A one-hot input row e_j reads column j of the weight: y = w_out[:, j]."""
    hidden, D = 16, 24
    rng = np.random.default_rng(7)
    w = rng.standard_normal((hidden, D))
    x = np.zeros((3, D))
    for t, j in enumerate((0, 5, 23)):
        x[t, j] = 1.0
    y = o.out_proj(x, w)
    assert y.shape == (3, hidden)
    for t, j in enumerate((0, 5, 23)):
        assert np.array_equal(y[t], w[:, j])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
