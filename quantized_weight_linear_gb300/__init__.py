"""quantized_weight_linear_gb300 -- Python binding of libqlin (quantized linear forward on GB300).

The library (``libqlin.so``, built from ``csrc/`` for sm_103a) implements
Y = X . W_hat^T for three compressed weight formats -- W4 g128 (GPTQ page),
SpQR 3-bit g16 with fp16 outliers (SpQR page) and SmoothQuant W8A8
(SmoothQuant page) -- behind a C ABI declared in ``include/qlin.h``.  This module
only marshals arguments: it loads the library with ctypes, mirrors its entry
points under the same names, and offers ``QLinear``, which uses PyTorch for device
memory and streams.  Every step of the forward runs in the library's kernels;
there is no other code path, and importing the package fails loudly if the
library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqlin.so")

QLIN_OK = 0
QLIN_ERR_INVALID_ARG = 1
QLIN_ERR_UNSUPPORTED = 2
QLIN_ERR_CUDA = 3
QLIN_ERR_WORKSPACE = 4
QLIN_ERR_TIMEOUT = 5
QLIN_ERR_NOT_BOUND = 6

FMT_W4G128 = 1
FMT_SPQR = 2
FMT_W8A8 = 3

#: every entry point include/qlin.h declares
EXPORTED_SYMBOLS = (
    "qlin_pack_w4g128", "qlin_pack_w4g128_gptq", "qlin_pack_spqr", "qlin_pack_w8", "qlin_device_bytes",
    "qlin_workspace_bytes",
    "qlin_bind", "qlin_attach", "qlin_set_workspace", "qlin_forward", "qlin_forward_host", "qlin_act_quant",
    "qlin_forward_acc", "qlin_dequant_device", "qlin_poll_status", "qlin_export", "qlin_info",
    "qlin_destroy", "qlin_status_string", "qlin_sm_count", "qlin_debug_wait_timeout", "qlin_forward_spqr_static",
    "qlin_poll_static_status", "qlin_import",
)


class QlinError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class LayerInfo(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32), ("nnz", ctypes.c_int64),
                ("packed_bytes", ctypes.c_int64), ("bits_per_param", ctypes.c_double),
                ("device_bytes", ctypes.c_int64), ("alpha", ctypes.c_float), ("outlier_frac", ctypes.c_float)]


class Canonical(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("codes", "scale", "zero", "codes3", "qs3", "qz3", "stats", "rowptr",
                                               "col", "val", "qw", "sw", "s", "s_inv", "perm")]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Loads libqlin.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqlin.so not found at {LIB_PATH}; build it with "
                              "`python -m quantized_weight_linear_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        H = ctypes.c_void_p
        sig = {
            "qlin_pack_w4g128": ([vp, i32, i32, ctypes.POINTER(H)], i32),
            "qlin_pack_w4g128_gptq": ([vp, i32, i32, vp, i32, ctypes.c_double, i32, ctypes.POINTER(H)], i32),
            "qlin_pack_spqr": ([vp, i32, i32, f32, ctypes.POINTER(H)], i32),
            "qlin_pack_w8": ([vp, i32, i32, vp, f32, ctypes.POINTER(H)], i32),
            "qlin_device_bytes": ([H, ctypes.POINTER(sz)], i32),
            "qlin_workspace_bytes": ([H, i32, ctypes.POINTER(sz)], i32),
            "qlin_bind": ([H, vp, sz, vp], i32),
            "qlin_attach": ([H, vp, sz], i32),
            "qlin_set_workspace": ([H, vp, sz, i32, vp], i32),
            "qlin_forward": ([H, vp, vp, i32, vp], i32),
            "qlin_forward_host": ([H, vp, vp, vp, vp, i32, vp], i32),
            "qlin_act_quant": ([H, vp, vp, vp, i32, vp], i32),
            "qlin_forward_acc": ([H, vp, vp, i32, vp], i32),
            "qlin_dequant_device": ([H, vp, vp], i32),
            "qlin_poll_status": ([H, vp], i32),
            "qlin_export": ([H, ctypes.POINTER(Canonical)], i32),
            "qlin_info": ([H, ctypes.POINTER(LayerInfo)], i32),
            "qlin_destroy": ([H], None),
            "qlin_status_string": ([i32], ctypes.c_char_p),
            "qlin_sm_count": ([], i32),
            "qlin_debug_wait_timeout": ([vp, i32, vp], i32),
            "qlin_forward_spqr_static": ([H, vp, vp, i32, vp], i32),
            "qlin_poll_static_status": ([vp], i32),
            "qlin_import": ([i32, i32, i32, ctypes.POINTER(Canonical), ctypes.POINTER(H)], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().qlin_status_string(status).decode()


def _check(status: int, what: str):
    if status != QLIN_OK:
        raise QlinError(status, what)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _vp(x) -> ctypes.c_void_p:
    """Pointer of a numpy array, a torch tensor, an int address or None."""
    if x is None:
        return ctypes.c_void_p(None)
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    if isinstance(x, np.ndarray):
        return ctypes.c_void_p(x.ctypes.data)
    return ctypes.c_void_p(x.data_ptr())


def _stream(s) -> ctypes.c_void_p:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        except Exception:  # pragma: no cover
            pass
        return ctypes.c_void_p(None)
    if isinstance(s, int):
        return ctypes.c_void_p(s)
    return ctypes.c_void_p(s.cuda_stream)


class Handle:
    """Owns a qlin_handle (host object); destroyed with the Python object."""

    def __init__(self, ptr: ctypes.c_void_p):
        self.ptr = ptr
        self._info = None

    def __del__(self):
        if getattr(self, "ptr", None) and self.ptr.value:
            try:
                lib().qlin_destroy(self.ptr)
            except Exception:  # pragma: no cover
                pass
            self.ptr = ctypes.c_void_p(None)

    @property
    def info(self) -> LayerInfo:
        if self._info is None:
            inf = LayerInfo()
            _check(lib().qlin_info(self.ptr, ctypes.byref(inf)), "qlin_info")
            self._info = inf
        return self._info


# -------------------------------------------------------------------------------- C ABI mirror

def qlin_pack_w4g128(W) -> Handle:
    W = _f32(W)
    h = ctypes.c_void_p()
    _check(lib().qlin_pack_w4g128(_vp(W), W.shape[0], W.shape[1], ctypes.byref(h)), "qlin_pack_w4g128")
    return Handle(h)


def qlin_pack_w4g128_gptq(W, Xcal, damp: float = 0.01, act_order: bool = False) -> Handle:
    W = _f32(W)
    X = _f32(Xcal)
    if X.ndim != 2 or X.shape[1] != W.shape[1]:
        raise ValueError("Xcal must be [S, K] with the layer's K")
    h = ctypes.c_void_p()
    _check(lib().qlin_pack_w4g128_gptq(_vp(W), W.shape[0], W.shape[1], _vp(X), X.shape[0], float(damp),
                                       int(bool(act_order)), ctypes.byref(h)), "qlin_pack_w4g128_gptq")
    return Handle(h)


def qlin_pack_spqr(W, outlier_frac: float) -> Handle:
    W = _f32(W)
    h = ctypes.c_void_p()
    _check(lib().qlin_pack_spqr(_vp(W), W.shape[0], W.shape[1], float(outlier_frac), ctypes.byref(h)),
           "qlin_pack_spqr")
    return Handle(h)


def qlin_pack_w8(W, act_absmax, alpha: float) -> Handle:
    W = _f32(W)
    a = _f32(act_absmax)
    h = ctypes.c_void_p()
    _check(lib().qlin_pack_w8(_vp(W), W.shape[0], W.shape[1], _vp(a), float(alpha), ctypes.byref(h)), "qlin_pack_w8")
    return Handle(h)


def qlin_device_bytes(h: Handle) -> int:
    n = ctypes.c_size_t()
    _check(lib().qlin_device_bytes(h.ptr, ctypes.byref(n)), "qlin_device_bytes")
    return n.value


def qlin_workspace_bytes(h: Handle, max_M: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().qlin_workspace_bytes(h.ptr, max_M, ctypes.byref(n)), "qlin_workspace_bytes")
    return n.value


def qlin_bind(h: Handle, dev_weights, nbytes: int, stream=None):
    _check(lib().qlin_bind(h.ptr, _vp(dev_weights), nbytes, _stream(stream)), "qlin_bind")


def qlin_attach(h: Handle, dev_weights, nbytes: int):
    _check(lib().qlin_attach(h.ptr, _vp(dev_weights), nbytes), "qlin_attach")


def qlin_set_workspace(h: Handle, dev_ws, nbytes: int, max_M: int, stream=None):
    _check(lib().qlin_set_workspace(h.ptr, _vp(dev_ws), nbytes, max_M, _stream(stream)), "qlin_set_workspace")


def qlin_forward(h: Handle, X, Y, M: int, stream=None):
    _check(lib().qlin_forward(h.ptr, _vp(X), _vp(Y), M, _stream(stream)), "qlin_forward")


def qlin_forward_spqr_static(h: Handle, X, Y, M: int, stream=None):
    """SpQR decode forward (1 <= M <= 16) that uses the library's fixed scratch array instead
    of a workspace: for callers that may not allocate device memory (see include/qlin.h)."""
    _check(lib().qlin_forward_spqr_static(h.ptr, _vp(X), _vp(Y), M, _stream(stream)), "qlin_forward_spqr_static")


def qlin_poll_static_status(stream=None) -> int:
    """Status of the qlin_forward_spqr_static calls on the current device since the last poll
    (waits for the stream; QLIN_OK or QLIN_ERR_TIMEOUT)."""
    return lib().qlin_poll_static_status(_stream(stream))


def qlin_forward_host(h: Handle, X_host, Y_host, X_dev, Y_dev, M: int, stream=None):
    _check(lib().qlin_forward_host(h.ptr, _vp(X_host), _vp(Y_host), _vp(X_dev), _vp(Y_dev), M, _stream(stream)),
           "qlin_forward_host")


def qlin_act_quant(h: Handle, X, qx, sx, M: int, stream=None):
    _check(lib().qlin_act_quant(h.ptr, _vp(X), _vp(qx), _vp(sx), M, _stream(stream)), "qlin_act_quant")


def qlin_forward_acc(h: Handle, X, acc, M: int, stream=None):
    _check(lib().qlin_forward_acc(h.ptr, _vp(X), _vp(acc), M, _stream(stream)), "qlin_forward_acc")


def qlin_dequant_device(h: Handle, out, stream=None):
    _check(lib().qlin_dequant_device(h.ptr, _vp(out), _stream(stream)), "qlin_dequant_device")


def qlin_poll_status(h: Handle, stream=None) -> int:
    return lib().qlin_poll_status(h.ptr, _stream(stream))


def qlin_sm_count() -> int:
    return lib().qlin_sm_count()


def qlin_debug_wait_timeout(status_dev, limit_us: int, stream=None):
    _check(lib().qlin_debug_wait_timeout(_vp(status_dev), limit_us, _stream(stream)), "qlin_debug_wait_timeout")


def qlin_export(h: Handle) -> dict:
    """Copies of the canonical packed arrays (layouts in include/qlin.h)."""
    c = Canonical()
    _check(lib().qlin_export(h.ptr, ctypes.byref(c)), "qlin_export")
    inf = h.info
    N, K, nnz = inf.N, inf.K, inf.nnz

    def arr(ptr, dtype, shape):
        count = int(np.prod(shape))
        if ptr is None or count == 0:
            return np.zeros(shape, dtype=dtype)
        buf = (ctypes.c_char * (count * np.dtype(dtype).itemsize)).from_address(ptr)
        return np.frombuffer(buf, dtype=dtype).reshape(shape).copy()

    if inf.format == FMT_W4G128:
        out = {"codes": arr(c.codes, np.uint32, (N, K // 8)),
               "scale": arr(c.scale, np.uint16, (N, K // 128)).view(np.float16),
               "zero": arr(c.zero, np.uint16, (N, K // 128)).view(np.float16)}
        if c.perm:  # act-order
            out["perm"] = arr(c.perm, np.int32, (K,))
        return out
    if inf.format == FMT_SPQR:
        return {"codes": arr(c.codes3, np.uint8, (N, 3 * K // 8)),
                "qs_bits": arr(c.qs3, np.uint8, (N, 3 * (K // 16) // 8)),
                "qz_bits": arr(c.qz3, np.uint8, (N, 3 * (K // 16) // 8)),
                "stats": arr(c.stats, np.uint16, (N, K // 256, 4)).view(np.float16),
                "rowptr": arr(c.rowptr, np.int32, (N + 1,)),
                "col": arr(c.col, np.int16, (nnz,)),
                "val": arr(c.val, np.uint16, (nnz,)).view(np.float16)}
    return {"qw": arr(c.qw, np.int8, (N, K)), "sw": arr(c.sw, np.float32, (N,)),
            "s": arr(c.s, np.float32, (K,)), "s_inv": arr(c.s_inv, np.float32, (K,))}


# canonical array names per format, with their dtypes (the dict qlin_export returns)
_CANONICAL = {
    FMT_W4G128: {"codes": np.uint32, "scale": np.float16, "zero": np.float16},
    FMT_SPQR: {"codes": np.uint8, "qs_bits": np.uint8, "qz_bits": np.uint8, "stats": np.float16,
               "rowptr": np.int32, "col": np.int16, "val": np.float16},
    FMT_W8A8: {"qw": np.int8, "sw": np.float32, "s": np.float32, "s_inv": np.float32},
}
_FIELD = {"codes3": "codes", "qs3": "qs_bits", "qz3": "qz_bits"}  # struct field -> dict key (SpQR)


def qlin_import(fmt: int, N: int, K: int, arrays: dict) -> Handle:
    """A handle from canonical arrays (a qlin_export dict or a loaded checkpoint); no quantization."""
    if fmt not in _CANONICAL:
        raise ValueError(f"unknown format {fmt}")
    keep = {k: np.ascontiguousarray(arrays[k], dtype=dt) for k, dt in _CANONICAL[fmt].items()}
    c = Canonical()
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p).value if a.size else None
    if fmt == FMT_W4G128:
        c.codes, c.scale, c.zero = ptr(keep["codes"]), ptr(keep["scale"]), ptr(keep["zero"])
        if arrays.get("perm") is not None:  # act-order
            keep["perm"] = np.ascontiguousarray(arrays["perm"], dtype=np.int32)
            c.perm = ptr(keep["perm"])
    elif fmt == FMT_SPQR:
        c.codes3, c.qs3, c.qz3 = ptr(keep["codes"]), ptr(keep["qs_bits"]), ptr(keep["qz_bits"])
        c.stats, c.rowptr, c.col, c.val = ptr(keep["stats"]), ptr(keep["rowptr"]), ptr(keep["col"]), ptr(keep["val"])
    else:
        c.qw, c.sw, c.s, c.s_inv = ptr(keep["qw"]), ptr(keep["sw"]), ptr(keep["s"]), ptr(keep["s_inv"])
    h = ctypes.c_void_p()
    _check(lib().qlin_import(int(fmt), int(N), int(K), ctypes.byref(c), ctypes.byref(h)), "qlin_import")
    return Handle(h)


# -------------------------------------------------------------------------------- torch front end

class QLinear:
    """A packed layer resident on one GPU; tensors come from PyTorch, compute from libqlin."""

    def __init__(self, handle: Handle):
        self.handle = handle
        inf = handle.info
        self.format, self.N, self.K = inf.format, inf.N, inf.K
        self.weights = None
        self.workspace = None
        self.max_M = 0

    @classmethod
    def from_w4g128(cls, W):
        return cls(qlin_pack_w4g128(W))

    @classmethod
    def from_w4g128_gptq(cls, W, Xcal, damp: float = 0.01, act_order: bool = False):
        return cls(qlin_pack_w4g128_gptq(W, Xcal, damp, act_order))

    @classmethod
    def from_spqr(cls, W, outlier_frac: float = 0.01):
        return cls(qlin_pack_spqr(W, outlier_frac))

    @classmethod
    def from_w8(cls, W, act_absmax, alpha: float = 0.85):
        return cls(qlin_pack_w8(W, act_absmax, alpha))

    def to(self, device="cuda", max_M: int = 16, stream=None):
        import torch
        nb = qlin_device_bytes(self.handle)
        self.weights = torch.empty(nb + 256, dtype=torch.uint8, device=device)
        w = self.weights[(-self.weights.data_ptr()) % 256:][:nb]
        qlin_bind(self.handle, w.data_ptr(), nb, stream)
        self.set_max_M(max_M, device, stream)
        return self

    def set_max_M(self, max_M: int, device="cuda", stream=None):
        import torch
        wb = qlin_workspace_bytes(self.handle, max_M)
        self.workspace = torch.empty(wb + 256, dtype=torch.uint8, device=device)
        ws = self.workspace[(-self.workspace.data_ptr()) % 256:][:wb]
        qlin_set_workspace(self.handle, ws.data_ptr(), wb, max_M, stream)
        self.max_M = max_M

    def __call__(self, X, out=None, stream=None):
        import torch
        assert X.dtype == torch.bfloat16 and X.is_contiguous() and X.shape[-1] == self.K
        M = X.shape[0]
        Y = out if out is not None else torch.empty((M, self.N), dtype=torch.bfloat16, device=X.device)
        qlin_forward(self.handle, X, Y, M, stream)
        return Y

    def forward_host(self, X_host, Y_host, X_dev, Y_dev, stream=None):
        qlin_forward_host(self.handle, X_host, Y_host, X_dev, Y_dev, X_host.shape[0], stream)
        return Y_host

    def act_quant(self, X, stream=None):
        import torch
        M = X.shape[0]
        qx = torch.empty((M, self.K), dtype=torch.int8, device=X.device)
        sx = torch.empty((M,), dtype=torch.float32, device=X.device)
        qlin_act_quant(self.handle, X, qx, sx, M, stream)
        return qx, sx

    def forward_acc(self, X, stream=None):
        import torch
        M = X.shape[0]
        acc = torch.empty((M, self.N), dtype=torch.int32, device=X.device)
        qlin_forward_acc(self.handle, X, acc, M, stream)
        return acc

    def dequant_device(self, stream=None):
        import torch
        dt = torch.int8 if self.format == FMT_W8A8 else torch.float32
        out = torch.empty((self.N, self.K), dtype=dt, device=self.weights.device)
        qlin_dequant_device(self.handle, out, stream)
        return out

    def poll_status(self, stream=None) -> int:
        return qlin_poll_status(self.handle, stream)

    def export(self) -> dict:
        return qlin_export(self.handle)

    def save(self, path) -> None:
        """Writes the canonical packed arrays (the qlin_export layouts) to an .npz checkpoint."""
        np.savez(path, format=np.int32(self.format), N=np.int32(self.N), K=np.int32(self.K), **self.export())

    @classmethod
    def load(cls, path):
        """A layer from a checkpoint written by save(); the weights are not requantized."""
        with np.load(path) as z:
            fmt, N, K = int(z["format"]), int(z["N"]), int(z["K"])
            arrays = {k: z[k] for k in _CANONICAL.get(fmt, {})}
            if "perm" in z.files:
                arrays["perm"] = z["perm"]
            return cls(qlin_import(fmt, N, K, arrays))


def build(force: bool = False) -> str:
    from .build import build as _b
    return _b(force=force)
