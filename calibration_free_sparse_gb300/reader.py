"""Thin ctypes binding of ``libmoe_reader.so`` (the C ABI in include/moe_reader.h).

Argument marshalling only: every step of prepare and decode runs in the CUDA
library.  The binding raises ``ReaderError`` when the library is missing --
there is no fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_reader.so")

OK, EINVAL, ENOMEM, ECUDA, ETIMEOUT, EDEVICE, ESTATE, ETOOBIG = 0, -1, -2, -3, -4, -5, -6, -7
FLAG_RHO_RANK = 0x1   # full screen ranked by the expected skip error (screen_coords = 128)
FLAG_TRIT5 = 0x2      # sketch codes stored five trits per byte
ERR_EXPERT_RANGE, ERR_EXPERT_DUP, ERR_WEIGHT, ERR_X_NONFINITE, ERR_TIMEOUT = 1, 2, 4, 8, 16
# one-shot fault injections for tests of failure detection (moe_reader_inject_fault)
INJECT_DECODE_STALL, INJECT_PREPARE_STALL, INJECT_ALLOC_FAIL = 0x1, 0x2, 0x4
ARRAYS = ("codes", "scales", "dnorm", "G", "V", "Dt", "b", "U")

EXPORT = {
    "codes": 0, "scales": 1, "rho": 2, "dnorm": 3, "Dt": 4, "U": 5, "b": 6, "sigma": 7,
    "eigvals": 8, "mask": 9, "ghat": 10, "vhat": 11, "score": 12,
}
EXPORTED_SYMBOLS = (
    "moe_reader_prepare", "moe_reader_decode", "moe_reader_decode_host", "moe_reader_status",
    "moe_reader_get_stats", "moe_reader_get_kept", "moe_reader_export_size", "moe_reader_export",
    "moe_reader_get_info", "moe_reader_destroy", "moe_reader_strerror", "moe_reader_abi_version",
    "moe_reader_set_profiling", "moe_reader_read_profile", "moe_reader_topk_noalloc",
    "moe_reader_decode_stack", "moe_reader_decode_shared", "moe_reader_get_kept_shared",
    "moe_reader_set_wait_limit", "moe_reader_inject_fault",
)
PHASES = ("decode", "screen", "score_topk", "exact", "out")


class ReaderError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = _lib().moe_reader_strerror(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("experts_per_token", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("screen_coords", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("flags", ctypes.c_int32)]


class Stats(ctypes.Structure):
    _fields_ = [("sectors", ctypes.c_uint64 * 8), ("dense_sectors", ctypes.c_uint64),
                ("activation_bytes", ctypes.c_uint64), ("batch", ctypes.c_int32),
                ("k", ctypes.c_int32)]


class Info(ctypes.Structure):
    _fields_ = [("hidden_padded", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("routed_channels", ctypes.c_int32), ("run_stride", ctypes.c_int32),
                ("resident_bytes", ctypes.c_uint64 * 9)]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m calibration_free_sparse_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.moe_reader_prepare.argtypes = [ctypes.POINTER(Config), vp, vp, vp, vp, vp,
                                           ctypes.POINTER(vp)]
        lib.moe_reader_prepare.restype = ctypes.c_int
        lib.moe_reader_decode.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp]
        lib.moe_reader_decode.restype = ctypes.c_int
        lib.moe_reader_decode_host.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp]
        lib.moe_reader_decode_host.restype = ctypes.c_int
        lib.moe_reader_decode_stack.argtypes = [vp, i32, vp, i32, vp, vp, i32, vp, vp, vp]
        lib.moe_reader_decode_stack.restype = ctypes.c_int
        lib.moe_reader_decode_shared.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp]
        lib.moe_reader_decode_shared.restype = ctypes.c_int
        lib.moe_reader_get_kept_shared.argtypes = [vp, vp, i64, ctypes.POINTER(ctypes.c_int32)]
        lib.moe_reader_get_kept_shared.restype = ctypes.c_int
        lib.moe_reader_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.moe_reader_status.restype = ctypes.c_int
        lib.moe_reader_get_stats.argtypes = [vp, ctypes.POINTER(Stats)]
        lib.moe_reader_get_stats.restype = ctypes.c_int
        lib.moe_reader_get_kept.argtypes = [vp, vp, i64]
        lib.moe_reader_get_kept.restype = ctypes.c_int
        lib.moe_reader_export_size.argtypes = [vp, i32]
        lib.moe_reader_export_size.restype = ctypes.c_int64
        lib.moe_reader_export.argtypes = [vp, i32, vp, i64]
        lib.moe_reader_export.restype = ctypes.c_int
        lib.moe_reader_get_info.argtypes = [vp, ctypes.POINTER(Info)]
        lib.moe_reader_get_info.restype = ctypes.c_int
        lib.moe_reader_destroy.argtypes = [vp]
        lib.moe_reader_destroy.restype = None
        lib.moe_reader_strerror.argtypes = [ctypes.c_int]
        lib.moe_reader_strerror.restype = ctypes.c_char_p
        lib.moe_reader_set_profiling.argtypes = [vp, i32]
        lib.moe_reader_set_profiling.restype = ctypes.c_int
        lib.moe_reader_read_profile.argtypes = [vp, ctypes.POINTER(ctypes.c_double), i64,
                                                ctypes.POINTER(ctypes.c_int64)]
        lib.moe_reader_read_profile.restype = ctypes.c_int
        lib.moe_reader_topk_noalloc.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        lib.moe_reader_topk_noalloc.restype = ctypes.c_int
        lib.moe_reader_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
        lib.moe_reader_set_wait_limit.restype = ctypes.c_int
        lib.moe_reader_inject_fault.argtypes = [vp, ctypes.c_uint32]
        lib.moe_reader_inject_fault.restype = ctypes.c_int
        lib.moe_reader_abi_version.argtypes = []
        lib.moe_reader_abi_version.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def library():
    """The loaded CDLL (raises if the library was not built)."""
    return _lib()


def _ptr(a):
    """Device or host address of a torch tensor, a numpy array or an int."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return a.data_ptr()
    raise TypeError(f"cannot take the address of {type(a)}")


def _stream(stream):
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, what):
    if code != OK:
        raise ReaderError(code, what)


def _require(t, dtype, shape, what):
    """A contiguous CUDA tensor of the given dtype and shape on the current device."""
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{what} is on cuda:{t.device.index}, not the current device")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")


def topk_noalloc(scores, k, kept, ids=None, stream=None):
    """Exact top-k per row of device scores [rows][cols] into device kept
    [rows][k] (ascending column indices) without any device allocation.
    scores: float32 [rows][cols]; kept: int32 [rows][k]; ids: int32
    [rows][cols] tie-break ids or None (the column index)."""
    import torch

    if scores.dim() != 2:
        raise ValueError("scores must be 2-D [rows][cols]")
    rows, cols = int(scores.shape[0]), int(scores.shape[1])
    _require(scores, torch.float32, (rows, cols), "scores")
    _require(kept, torch.int32, (rows, int(k)), "kept")
    if ids is not None:
        _require(ids, torch.int32, (rows, cols), "ids")
    code = _lib().moe_reader_topk_noalloc(_ptr(scores), _ptr(ids), rows, cols, int(k),
                                          _ptr(kept), _stream(stream))
    _check(code, "moe_reader_topk_noalloc")


def inject_fault(what, reader=None):
    """Arm a one-shot failure (INJECT_* bits): a decode stall on `reader`, or,
    with reader None, a stall in the next prepare or a failed next device
    allocation.  Nothing faults the GPU; the failure surfaces as a status."""
    _check(_lib().moe_reader_inject_fault(None if reader is None else reader.handle, int(what)),
           "moe_reader_inject_fault")


def decode_stack(readers, h_in, ids, w, k, h_out, y_layers=None, stream=None):
    """Enqueue one decode of B = h_in.shape[0] tokens through the stacked
    layers `readers` (distinct MoeReader objects of one shape) in a single
    launch: layer l decodes h_l / RMS(h_l) and h_{l+1} = h_l + y_l; h_out
    receives h_L.  ids, w: device [L][B][topk]; y_layers: device [L][B][H]
    or None."""
    L = len(readers)
    arr = (ctypes.c_void_p * L)(*[r.handle for r in readers])
    code = _lib().moe_reader_decode_stack(arr, L, _ptr(h_in), int(h_in.shape[0]), _ptr(ids),
                                          _ptr(w), int(k), _ptr(h_out), _ptr(y_layers),
                                          _stream(stream))
    _check(code, "moe_reader_decode_stack")


class MoeReader:
    """One prepared MoE layer.  `gate`, `up`, `down` are device BF16 tensors
    ([E][I][H], [E][I][H], [E][H][I]); gate and up must outlive the reader."""

    def __init__(self, hidden, num_experts, experts_per_token, inter, gate, up, down, sigma,
                 screen_coords=80, rank=32, max_batch=16, stream=None, flags=0):
        lib = _lib()
        self.cfg = Config(hidden, num_experts, experts_per_token, inter, screen_coords, rank,
                          max_batch, flags)
        sig = np.ascontiguousarray(sigma, dtype=np.int8)
        self._keep = (gate, up)
        h = ctypes.c_void_p()
        code = lib.moe_reader_prepare(ctypes.byref(self.cfg), _ptr(gate), _ptr(up), _ptr(down),
                                      sig.ctypes.data, _stream(stream), ctypes.byref(h))
        _check(code, "moe_reader_prepare")
        self._h = h
        self.H, self.E, self.topk, self.I = hidden, num_experts, experts_per_token, inter
        self.r, self.c, self.max_batch = rank, screen_coords, max_batch
        info = self.info()
        self.Hp, self.nb, self.N, self.S = (info["hidden_padded"], info["num_blocks"],
                                            info["routed_channels"], info["run_stride"])

    # -- lifetime ---------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            _lib().moe_reader_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h.value

    # -- decode -----------------------------------------------------------
    def decode(self, x, ids, w, k, y, stream=None):
        """Enqueue one decode of B = x.shape[0] tokens (device tensors)."""
        B = int(x.shape[0])
        code = _lib().moe_reader_decode(self._h, _ptr(x), B, _ptr(ids), _ptr(w), int(k), _ptr(y),
                                        _stream(stream))
        _check(code, "moe_reader_decode")

    def decode_shared(self, x, ids, w, k, y, stream=None):
        """Enqueue one decode of B = x.shape[0] tokens with one kept set for
        the whole batch (device tensors)."""
        B = int(x.shape[0])
        code = _lib().moe_reader_decode_shared(self._h, _ptr(x), B, _ptr(ids), _ptr(w), int(k),
                                               _ptr(y), _stream(stream))
        _check(code, "moe_reader_decode_shared")

    def kept_shared(self):
        """The last shared decode's kept set: ascending global ids (host int32)."""
        K = ctypes.c_int32(0)
        code = _lib().moe_reader_get_kept_shared(self._h, None, 0, ctypes.byref(K))
        if code not in (OK, EINVAL):
            _check(code, "moe_reader_get_kept_shared")
        out = np.zeros(max(1, K.value), np.int32)
        _check(_lib().moe_reader_get_kept_shared(self._h, _ptr(out), out.size, ctypes.byref(K)),
               "moe_reader_get_kept_shared")
        return out[:K.value]

    def decode_host(self, x, ids, w, k, y=None, stream=None):
        """Decode with host numpy buffers; returns y (host, fp32 [B][H])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        B = x.shape[0]
        if y is None:
            y = np.empty((B, self.H), np.float32)
        code = _lib().moe_reader_decode_host(self._h, _ptr(x), B, _ptr(ids), _ptr(w), int(k),
                                             _ptr(y), _stream(stream))
        _check(code, "moe_reader_decode_host")
        return y

    def set_wait_limit(self, ns):
        """Bound (ns of the GPU timer) of every device wait of later decodes; 0 = 1 s."""
        _check(_lib().moe_reader_set_wait_limit(self._h, int(ns)), "moe_reader_set_wait_limit")

    def status(self):
        bits = ctypes.c_uint32(0)
        code = _lib().moe_reader_status(self._h, ctypes.byref(bits))
        return code, bits.value

    def stats(self):
        st = Stats()
        _check(_lib().moe_reader_get_stats(self._h, ctypes.byref(st)), "moe_reader_get_stats")
        out = {name: int(st.sectors[i]) for i, name in enumerate(ARRAYS)}
        out["dense"] = int(st.dense_sectors)
        out["activation_bytes"] = int(st.activation_bytes)
        out["batch"], out["k"] = int(st.batch), int(st.k)
        return out

    def kept(self, B, k):
        out = np.zeros((B, k), np.int32)
        _check(_lib().moe_reader_get_kept(self._h, _ptr(out), out.size), "moe_reader_get_kept")
        return out

    def export(self, name, B=None):
        which = EXPORT[name]
        n = _lib().moe_reader_export_size(self._h, which)
        if n < 0:
            raise ReaderError(int(n), f"export {name}")
        buf = np.empty(int(n), np.uint8)
        _check(_lib().moe_reader_export(self._h, which, _ptr(buf), int(n)), f"export {name}")
        E, I, H, r, nb, S, Hp, N = self.E, self.I, self.H, self.r, self.nb, self.S, self.Hp, self.N
        shapes = {
            "codes": (np.uint8, (E, nb, 128, 2, S)), "scales": (np.float16, (E, nb, 2, I)),
            "rho": (np.float16, (E, nb, 2, I)), "dnorm": (np.float32, (E, I)),
            "Dt": (np.uint16, (E, I, H)), "U": (np.float16, (H, r)), "b": (np.float16, (E, I, r)),
            "sigma": (np.int8, (Hp,)), "eigvals": (np.float64, (r,)),
            "mask": (np.uint32, (-1, nb, 4)), "ghat": (np.float32, (-1, N)),
            "vhat": (np.float32, (-1, N)), "score": (np.float32, (-1, N)),
        }
        dt, shape = shapes[name]
        return buf.view(dt).reshape(shape)

    def set_profiling(self, enable):
        _check(_lib().moe_reader_set_profiling(self._h, 1 if enable else 0), "set_profiling")

    def read_profile(self):
        """Per recorded decode slot, the milliseconds of each phase: list of dicts."""
        cap = 64
        ms = (ctypes.c_double * (cap * len(PHASES)))()
        calls = ctypes.c_int64(0)
        _check(_lib().moe_reader_read_profile(self._h, ms, cap, ctypes.byref(calls)),
               "read_profile")
        n = int(calls.value)
        return [dict(zip(PHASES, ms[i * len(PHASES):(i + 1) * len(PHASES)])) for i in range(n)]

    def info(self):
        inf = Info()
        _check(_lib().moe_reader_get_info(self._h, ctypes.byref(inf)), "moe_reader_get_info")
        return {"hidden_padded": inf.hidden_padded, "num_blocks": inf.num_blocks,
                "routed_channels": inf.routed_channels, "run_stride": inf.run_stride,
                "resident_bytes": [int(v) for v in inf.resident_bytes]}
