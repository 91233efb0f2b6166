"""ctypes binding of libgdn (include/gdn.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module turns
torch tensors into device pointers and streams into handles, and raises
``GdnError`` on a non-zero status.  It has no fallback: if ``libgdn.so`` has not
been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

GDN_OK = 0
STATUS = {
    0: "ok", -1: "invalid argument", -2: "pool full", -3: "bad slot", -4: "CUDA error",
    -5: "device wait timed out", -6: "unsupported shape", -7: "layer parameters not registered",
    -8: "device reported skipped work",
}
DEV_BAD_SLOT_PTR, DEV_BAD_SLOT_ID, DEV_BAD_SEQLENS, DEV_TIMEOUT, DEV_SLOT_OVERLAP, DEV_BOUNDS = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20

# every extern "C" symbol include/gdn.h declares
EXPORTS = [
    "gdn_pool_create", "gdn_pool_destroy", "gdn_pool_reset", "gdn_slot_alloc", "gdn_slot_recycle",
    "gdn_slot_addr", "gdn_slot_ptrs", "gdn_layer_params", "gdn_decode_step", "gdn_prefill_varlen",
    "gdn_last_device_status", "gdn_pool_get_info", "gdn_status_string", "gdn_version",
    "gdn_prefill_varlen_noalloc", "gdn_slot_snapshot", "gdn_slot_restore", "gdn_mixed_step",
    "gdn_in_proj", "gdn_out_proj",
]


class GdnError(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {STATUS.get(code, 'unknown')} ({code})")
        self.code = code


class GdnShape(ctypes.Structure):
    _fields_ = [
        ("hqk", ctypes.c_int), ("hv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("conv_w", ctypes.c_int), ("chunk", ctypes.c_int), ("io_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
        ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float), ("max_prefill_tokens", ctypes.c_int),
    ]


class GdnPoolInfo(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
        ("state_bytes", ctypes.c_uint64), ("conv_bytes", ctypes.c_uint64), ("num_slots", ctypes.c_int),
        ("num_layers", ctypes.c_int), ("free_slots", ctypes.c_int), ("workspace_bytes", ctypes.c_uint64),
    ]


def lib_path() -> str:
    """libgdn.so, or the checked debug build (libgdn_checked.so) when the environment variable
    GDN_LIBRARY_VARIANT is "checked"."""
    return _build.LIB_CHECKED if os.environ.get("GDN_LIBRARY_VARIANT") == "checked" else _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so; raises if it was never built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libgdn.so is not built ({path}); run gated_deltanet_linear_rule_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i, u64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)
        L.gdn_pool_create.argtypes = [ctypes.POINTER(GdnShape), i, i, ctypes.POINTER(vp)]
        L.gdn_pool_destroy.argtypes = [vp]
        L.gdn_pool_reset.argtypes = [vp, vp]
        L.gdn_slot_alloc.argtypes = [vp, ctypes.POINTER(i)]
        L.gdn_slot_recycle.argtypes = [vp, i, vp]
        L.gdn_slot_addr.argtypes = [vp, i, i, u64p]
        L.gdn_slot_ptrs.argtypes = [vp, i, vp, i, vp, vp]
        L.gdn_layer_params.argtypes = [vp, i, vp, vp, vp, vp]
        L.gdn_decode_step.argtypes = [vp, i, vp, i, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gdn_prefill_varlen.argtypes = [vp, i, vp, vp, i, i, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gdn_in_proj.argtypes = [ctypes.POINTER(GdnShape), i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gdn_out_proj.argtypes = [ctypes.POINTER(GdnShape), i, i, vp, vp, vp, vp, vp]
        L.gdn_mixed_step.argtypes = [vp, i, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp, vp, vp, vp,
                                     vp, vp]
        L.gdn_last_device_status.argtypes = [vp, vp]
        L.gdn_pool_get_info.argtypes = [vp, ctypes.POINTER(GdnPoolInfo)]
        L.gdn_prefill_varlen_noalloc.argtypes = [ctypes.POINTER(GdnShape), vp, vp, vp, vp, vp, i, vp, vp, i, i,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gdn_slot_snapshot.argtypes = [vp, i, vp, vp]
        L.gdn_slot_restore.argtypes = [vp, i, vp, vp]
        L.gdn_status_string.argtypes = [i]
        L.gdn_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "gdn_status_string":
                getattr(L, name).restype = i
        _lib = L
    return _lib


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise GdnError(what, rc)
    return rc


def _p(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensors passed to libgdn must be contiguous")
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


_DTYPES = {"f32": (0, torch.float32), "bf16": (1, torch.bfloat16)}


class _DevView:
    """A device range exposed through __cuda_array_interface__ so torch can alias it."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


class Pool:
    """One slot pool (gdn_pool_create) and the calls that act on it."""

    def __init__(self, hqk: int, hv: int, dk: int, dv: int, num_slots: int, num_layers: int = 1, conv_w: int = 4,
                 io_dtype: str = "bf16", out_dtype: str | None = None, chunk: int = 0, max_prefill_tokens: int = 0,
                 l2_eps: float = 1e-6, norm_eps: float = 1e-6):
        self.io_dtype, self.out_dtype = io_dtype, out_dtype or io_dtype
        self.torch_io = _DTYPES[self.io_dtype][1]
        self.torch_out = _DTYPES[self.out_dtype][1]
        self.shape = GdnShape(hqk, hv, dk, dv, conv_w, chunk, _DTYPES[self.io_dtype][0], _DTYPES[self.out_dtype][0],
                              l2_eps, norm_eps, max_prefill_tokens)
        self.hqk, self.hv, self.dk, self.dv, self.conv_w = hqk, hv, dk, dv, conv_w
        self.C = 2 * hqk * dk + hv * dv
        self.num_slots, self.num_layers = num_slots, num_layers
        self._h = ctypes.c_void_p()
        self._params = {}
        _check(lib().gdn_pool_create(ctypes.byref(self.shape), num_slots, num_layers, ctypes.byref(self._h)),
               "gdn_pool_create")

    # -- lifecycle ---------------------------------------------------------
    def close(self):
        if self._h:
            _check(lib().gdn_pool_destroy(self._h), "gdn_pool_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self):
        return self._h

    def info(self) -> GdnPoolInfo:
        inf = GdnPoolInfo()
        _check(lib().gdn_pool_get_info(self._h, ctypes.byref(inf)), "gdn_pool_get_info")
        return inf

    def reset(self, stream=None):
        _check(lib().gdn_pool_reset(self._h, _stream(stream)), "gdn_pool_reset")

    # -- slots -------------------------------------------------------------
    def alloc(self) -> int:
        sid = ctypes.c_int(-1)
        _check(lib().gdn_slot_alloc(self._h, ctypes.byref(sid)), "gdn_slot_alloc")
        return sid.value

    def recycle(self, slot: int, stream=None):
        _check(lib().gdn_slot_recycle(self._h, int(slot), _stream(stream)), "gdn_slot_recycle")

    def slot_addr(self, layer: int, slot: int) -> int:
        a = ctypes.c_uint64()
        _check(lib().gdn_slot_addr(self._h, int(layer), int(slot), ctypes.byref(a)), "gdn_slot_addr")
        return a.value

    def snapshot_bytes(self) -> int:
        inf = self.info()
        return int(inf.slot_bytes) * self.num_layers

    def snapshot(self, slot: int, dst: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Copy every layer of a slot into dst (a uint8 tensor on the device or in pinned host memory)."""
        if dst is None:
            dst = torch.empty(self.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        assert dst.numel() * dst.element_size() >= self.snapshot_bytes()
        _check(lib().gdn_slot_snapshot(self._h, int(slot), _p(dst), _stream(stream)), "gdn_slot_snapshot")
        return dst

    def restore(self, slot: int, src: torch.Tensor, stream=None):
        """Overwrite every layer of an allocated slot with a snapshot."""
        assert src.numel() * src.element_size() >= self.snapshot_bytes()
        _check(lib().gdn_slot_restore(self._h, int(slot), _p(src), _stream(stream)), "gdn_slot_restore")

    def slot_ptrs(self, layer: int, slot_ids: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        """Device u64 slot-pointer array (returned as an int64 tensor) for the given int32 device ids."""
        assert slot_ids.dtype == torch.int32 and slot_ids.is_cuda
        if out is None:
            out = torch.empty(slot_ids.numel(), dtype=torch.int64, device=slot_ids.device)
        _check(lib().gdn_slot_ptrs(self._h, int(layer), _p(slot_ids), slot_ids.numel(), _p(out), _stream(stream)),
               "gdn_slot_ptrs")
        return out

    def state_views(self, layer: int, slot: int):
        """Torch tensors aliasing (slot, layer): S [Hv][dv][dk] fp32 and the conv buffer [W-1][C] (io dtype)."""
        base = self.slot_addr(layer, slot)
        inf = self.info()
        S = torch.as_tensor(_DevView(base, (self.hv, self.dv, self.dk), "<f4"), device="cuda")
        W1 = self.conv_w - 1
        if self.io_dtype == "bf16":
            conv = torch.as_tensor(_DevView(base + inf.state_bytes, (W1, self.C), "<i2"), device="cuda")
            conv = conv.view(torch.bfloat16)
        else:
            conv = torch.as_tensor(_DevView(base + inf.state_bytes, (W1, self.C), "<f4"), device="cuda")
        return S, conv

    def state_block(self, layer: int):
        """Strided fp32 view [num_slots][Hv][dv][dk] over the S of every slot of one layer."""
        inf = self.info()
        base = self.slot_addr(layer, 0)
        slot_stride = inf.slot_bytes * self.num_layers
        view = _DevView(base, (self.num_slots, self.hv, self.dv, self.dk), "<f4")
        view.__cuda_array_interface__["strides"] = (slot_stride, self.dv * self.dk * 4, self.dk * 4, 4)
        return torch.as_tensor(view, device="cuda")

    # -- layer -------------------------------------------------------------
    def layer_params(self, layer: int, conv_w, A_log, dt_bias, norm_w):
        ts = [t.contiguous().to(device="cuda", dtype=torch.float32) for t in (conv_w, A_log, dt_bias, norm_w)]
        _check(lib().gdn_layer_params(self._h, int(layer), *(_p(t) for t in ts)), "gdn_layer_params")
        self._params[layer] = ts  # the pool borrows these arrays

    def decode_step(self, layer: int, slot_ptrs, m: int, q, k, v, a, b, z, out, stream=None):
        _check(lib().gdn_decode_step(self._h, int(layer), _p(slot_ptrs), int(m), _p(q), _p(k), _p(v), _p(a), _p(b),
                                     _p(z), _p(out), _stream(stream)), "gdn_decode_step")

    def prefill_varlen(self, layer: int, cu_seqlens, slot_ids, n_seqs: int, total_tokens: int, q, k, v, a, b, z,
                       out, stream=None):
        _check(lib().gdn_prefill_varlen(self._h, int(layer), _p(cu_seqlens), _p(slot_ids), int(n_seqs),
                                        int(total_tokens), _p(q), _p(k), _p(v), _p(a), _p(b), _p(z), _p(out),
                                        _stream(stream)), "gdn_prefill_varlen")

    def mixed_step(self, layer: int, slot_ptrs, m: int, dq, dk, dv, da, db, dz, dout, cu_seqlens, slot_ids,
                   n_seqs: int, total_tokens: int, pq, pk, pv, pa, pb, pz, pout, stream=None):
        """gdn_mixed_step: m decode rows and n_seqs prefill sequences of `layer` in one call."""
        _check(lib().gdn_mixed_step(self._h, int(layer), _p(slot_ptrs), int(m), _p(dq), _p(dk), _p(dv), _p(da),
                                    _p(db), _p(dz), _p(dout), _p(cu_seqlens), _p(slot_ids), int(n_seqs),
                                    int(total_tokens), _p(pq), _p(pk), _p(pv), _p(pa), _p(pb), _p(pz), _p(pout),
                                    _stream(stream)), "gdn_mixed_step")

    def device_status(self, stream=None) -> int:
        return _check(lib().gdn_last_device_status(self._h, _stream(stream)), "gdn_last_device_status")


def slot_bytes(hqk: int, hv: int, dk: int, dv: int, conv_w: int = 4, io_dtype: str = "bf16") -> int:
    """Bytes of one slot (fp32 S then the conv buffer, rounded up to 256), as a pool lays it out."""
    io = 2 if io_dtype == "bf16" else 4
    raw = hv * dv * dk * 4 + (conv_w - 1) * (2 * hqk * dk + hv * dv) * io
    return (raw + 255) // 256 * 256


def prefill_varlen_noalloc(shape: GdnShape, conv_w, A_log, dt_bias, norm_w, states, num_slots: int, cu_seqlens,
                           slot_ids, n_seqs: int, total_tokens: int, q, k, v, a, b, z, out, status=None,
                           stream=None):
    """gdn_prefill_varlen_noalloc: the prefill kernels on caller-owned slots, with the library's static
    scratch instead of a pool workspace (no device allocation inside the call)."""
    _check(lib().gdn_prefill_varlen_noalloc(ctypes.byref(shape), _p(conv_w), _p(A_log), _p(dt_bias), _p(norm_w),
                                            _p(states), int(num_slots), _p(cu_seqlens), _p(slot_ids), int(n_seqs),
                                            int(total_tokens), _p(q), _p(k), _p(v), _p(a), _p(b), _p(z), _p(out),
                                            _p(status), _stream(stream)), "gdn_prefill_varlen_noalloc")


def in_proj(shape: GdnShape, hidden: int, T: int, x, w_in, q, k, v, z, a, b, status=None, stream=None):
    """gdn_in_proj: x [T][hidden] times the concatenated weight rows -> q, k, v, z, a, b (bf16)."""
    _check(lib().gdn_in_proj(ctypes.byref(shape), int(hidden), int(T), _p(x), _p(w_in), _p(q), _p(k), _p(v), _p(z),
                             _p(a), _p(b), _p(status), _stream(stream)), "gdn_in_proj")


def out_proj(shape: GdnShape, hidden: int, T: int, o, w_out, y, status=None, stream=None):
    """gdn_out_proj: y [T][hidden] = o [T][Hv*dv] times w_out^T (bf16)."""
    _check(lib().gdn_out_proj(ctypes.byref(shape), int(hidden), int(T), _p(o), _p(w_out), _p(y), _p(status),
                              _stream(stream)), "gdn_out_proj")


def version() -> int:
    return lib().gdn_version()


def status_string(code: int) -> str:
    return lib().gdn_status_string(int(code)).decode()
