"""fp64 CPU oracle of the Gated Delta Rule layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never does, and
this package imports nothing from it: the two share no code.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision); this
module compiles it with the host C compiler and wraps it with ctypes and numpy.
Every function states the step of the layer it follows; the steps are the ones
the "System Design" page lists for a GatedDeltaNet layer ("Runtime Data Flow"
and "GDN Kernel Dispatch Detail"): depthwise causal conv1d, L2 normalisation of
q and k, the gated delta-rule state update and read-out, gated RMSNorm.

Parity status per function (what pins it, see the tests):
  conv_silu          pinned: torch conv1d (groups=C) + SiLU, with and without buffer
  l2norm             pinned: torch F.normalize (eps effect below 1e-9 relative)
  gates              pinned: torch softplus / sigmoid / exp
  delta_recurrent    pinned: closed forms (pure decay, write-then-read, associative
                     recall, reset), brute-force transition-matrix products,
                     hand-worked golden example
  delta_chunked      pinned: equals delta_recurrent to 1e-12
  gated_rmsnorm      pinned: torch F.rms_norm * F.silu
  layer              pinned: composition of the pinned library routines above,
                     GQA head mapping, split-call and prefill/decode invariants
  in_proj, out_proj  pinned: selector weights copy input columns, the output split
                     order, one-hot inputs read weight columns (the projections are
                     the plain product, numpy in float64)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()


def build(src: str = _SRC, out: str = _LIB_PATH, openmp: bool = True) -> str:
    """Compile the oracle C source into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:
        if openmp:  # a toolchain without OpenMP still builds the single-thread oracle
            return build(src, out, openmp=False)
        raise RuntimeError(f"oracle build failed: {e.stderr}") from e
    return out


class _Shape(ctypes.Structure):
    _fields_ = [
        ("hqk", ctypes.c_int),
        ("hv", ctypes.c_int),
        ("dk", ctypes.c_int),
        ("dv", ctypes.c_int),
        ("conv_w", ctypes.c_int),
        ("l2_eps", ctypes.c_double),
        ("norm_eps", ctypes.c_double),
    ]


def _dp(x: np.ndarray):
    assert x.dtype == np.float64 and x.flags["C_CONTIGUOUS"], "oracle arrays are contiguous float64"
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


class Oracle:
    """ctypes wrapper around one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = ctypes.CDLL(lib_path)
        P = ctypes.POINTER(ctypes.c_double)
        I = ctypes.c_int
        self.lib.gdn_oracle_conv_silu.argtypes = [I, I, I, P, P, P, P]
        self.lib.gdn_oracle_l2norm.argtypes = [I, I, ctypes.c_double, P, P]
        self.lib.gdn_oracle_gates.argtypes = [I, ctypes.c_double, ctypes.c_double, P, P, P, P]
        self.lib.gdn_oracle_delta_recurrent.argtypes = [I, I, I, P, P, P, P, P, P, P]
        self.lib.gdn_oracle_delta_chunked.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
        self.lib.gdn_oracle_gated_rmsnorm.argtypes = [I, I, ctypes.c_double, P, P, P, P]
        self.lib.gdn_oracle_layer.argtypes = [
            ctypes.POINTER(_Shape), I, ctypes.POINTER(ctypes.c_int64),
            P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.POINTER(ctypes.c_int), I, I,
        ]
        self.lib.gdn_oracle_layer.restype = I
        self.lib.gdn_oracle_max_threads.restype = I

    # -- single steps ------------------------------------------------------
    def conv_silu(self, x, w, buf):
        """Depthwise causal conv1d + SiLU. x [L][C], w [C][W], buf [W-1][C].
        Returns (y [L][C], new buffer [W-1][C])."""
        x, w, buf = _f64(x), _f64(w), _f64(buf).copy()
        L, C = x.shape
        W = w.shape[1]
        y = np.zeros((L, C))
        self.lib.gdn_oracle_conv_silu(C, W, L, _dp(x), _dp(w), _dp(buf), _dp(y))
        return y, buf

    def l2norm(self, x, eps=1e-6):
        """Row-wise x / sqrt(sum x^2 + eps) over the last axis."""
        x = _f64(x)
        d = x.shape[-1]
        n = x.size // d if d else 0
        y = np.zeros_like(x)
        self.lib.gdn_oracle_l2norm(n, d, eps, _dp(x), _dp(y))
        return y

    def gates(self, a, b, A_log, dt_bias=0.0):
        """Per-token gates of one v-head: returns (g, beta) with alpha = exp(g)."""
        a, b = _f64(a).ravel(), _f64(b).ravel()
        g, beta = np.zeros_like(a), np.zeros_like(a)
        self.lib.gdn_oracle_gates(a.size, float(A_log), float(dt_bias), _dp(a), _dp(b), _dp(g), _dp(beta))
        return g, beta

    def delta_recurrent(self, q, k, v, g, beta, S0):
        """Recurrent gated delta rule for one head. Returns (o [L][dv], S [dv][dk])."""
        q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g).ravel(), _f64(beta).ravel()
        S = _f64(S0).copy()
        L, dk = k.shape
        dv = v.shape[1]
        o = np.zeros((L, dv))
        self.lib.gdn_oracle_delta_recurrent(L, dk, dv, _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta), _dp(S), _dp(o))
        return o, S

    def delta_chunked(self, q, k, v, g, beta, S0, chunk):
        """Chunked WY form of the same recurrence (self-check only)."""
        q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g).ravel(), _f64(beta).ravel()
        S = _f64(S0).copy()
        L, dk = k.shape
        dv = v.shape[1]
        o = np.zeros((L, dv))
        self.lib.gdn_oracle_delta_chunked(L, dk, dv, int(chunk), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                          _dp(S), _dp(o))
        return o, S

    def gated_rmsnorm(self, o, z, w, eps=1e-6):
        """o / sqrt(mean(o^2) + eps) * w * silu(z), rows over the last axis."""
        o, z, w = _f64(o), _f64(z), _f64(w)
        dv = o.shape[-1]
        n = o.size // dv
        y = np.zeros_like(o)
        self.lib.gdn_oracle_gated_rmsnorm(n, dv, eps, _dp(o), _dp(z), _dp(w), _dp(y))
        return y

    # -- whole layer -------------------------------------------------------
    def layer(self, shape, cu_seqlens, q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, S, convbuf,
              head_mask=None, chunk=0, threads=0, want_o=False):
        """One GDN layer over packed sequences.

        shape: dict with hqk, hv, dk, dv, conv_w, l2_eps, norm_eps.
        S [n][Hv][dv][dk] and convbuf [n][W-1][C] are the initial states (not modified).
        Returns dict(out, S, convbuf[, o]) -- new arrays."""
        sh = _Shape(shape["hqk"], shape["hv"], shape["dk"], shape["dv"], shape["conv_w"],
                    float(shape.get("l2_eps", 1e-6)), float(shape.get("norm_eps", 1e-6)))
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        n = cu.size - 1
        q, k, v, a, b, z = (_f64(t) for t in (q, k, v, a, b, z))
        conv_w, A_log, dt_bias, norm_w = (_f64(t) for t in (conv_w, A_log, dt_bias, norm_w))
        S = _f64(S).copy()
        convbuf = _f64(convbuf).copy()
        T = int(cu[-1] - cu[0])
        out = np.zeros((T, shape["hv"] * shape["dv"]))
        o = np.zeros_like(out) if want_o else None
        hm = None
        if head_mask is not None:
            hm = np.ascontiguousarray(np.asarray(head_mask, dtype=np.int32))
        rc = self.lib.gdn_oracle_layer(
            ctypes.byref(sh), n, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            _dp(q), _dp(k), _dp(v), _dp(a), _dp(b), _dp(z), _dp(conv_w), _dp(A_log), _dp(dt_bias),
            _dp(norm_w), _dp(S), _dp(convbuf), _dp(out), _dp(o) if o is not None else None,
            hm.ctypes.data_as(ctypes.POINTER(ctypes.c_int)) if hm is not None else None,
            int(chunk), int(threads))
        if rc != 0:
            raise ValueError("oracle layer rejected its arguments")
        res = {"out": out, "S": S, "convbuf": convbuf}
        if want_o:
            res["o"] = o
        return res

    # The projections around the layer (the layer tree of the pages: "Projections: in_proj_qkv,
    # in_proj_z, in_proj_b, in_proj_a" before the conv, "out_proj" after the gated RMSNorm).
    # Each is a linear map with weight rows = output features: y = x . W^T.
    def in_proj(self, x, w_in, hqk, hv, dk, dv):
        """x [T][hidden], w_in [N][hidden] with rows q (hqk*dk) | k (hqk*dk) | v (hv*dv) | z (hv*dv) |
        a (hv) | b (hv).  Returns dict(q, k, v, z, a, b), each [T][width]."""
        y = _f64(x) @ _f64(w_in).T
        widths = [("q", hqk * dk), ("k", hqk * dk), ("v", hv * dv), ("z", hv * dv), ("a", hv), ("b", hv)]
        out, c = {}, 0
        for name, w in widths:
            out[name] = np.ascontiguousarray(y[:, c:c + w])
            c += w
        assert c == y.shape[1], "w_in has the wrong number of rows"
        return out

    def out_proj(self, o, w_out):
        """o [T][hv*dv], w_out [hidden][hv*dv] -> y [T][hidden]."""
        return _f64(o) @ _f64(w_out).T

    def max_threads(self) -> int:
        return int(self.lib.gdn_oracle_max_threads())


_default: Oracle | None = None


def load(lib_path: str | None = None) -> Oracle:
    """The oracle built from ``gdn_oracle.c`` (compiled on first use), or a given build."""
    global _default
    if lib_path is not None:
        return Oracle(lib_path)
    with _lock:
        if _default is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _default = Oracle(_LIB_PATH)
    return _default
