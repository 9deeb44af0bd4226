"""Python binding of libdn: the C ABI of include/dn.h under the same names.

Argument marshalling only.  Every step of the layer runs in the library's
CUDA kernels; nothing here computes.  Host arrays are numpy arrays (or CPU
torch tensors) and are passed as DN_PTR_HOST; CUDA torch tensors are passed
as DN_PTR_DEVICE together with torch's current stream.  There is no
fallback: if libdn.so is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

DN_OK = 0
DN_EINVAL = -1
DN_ENOMEM = -2
DN_ECUDA = -3
DN_EFAILED = -4
DN_EINJECTED = -5
DN_PTR_HOST = 0
DN_PTR_DEVICE = 1
DN_FLAG_KEY_GATE = 1
DN_FLAG_DEVICE_GATES = 2
DN_FLAG_INT4_WEIGHTS = 4


def pack_int4(w: np.ndarray) -> np.ndarray:
    """int4 weights (integers in [-8, 7], [rows][K], K even) in the ABI's
    packed form: byte i of a row holds k = 2i in its low and k = 2i + 1 in
    its high four bits, two's complement."""
    w = np.asarray(w)
    if w.ndim != 2 or w.shape[1] % 2 or w.min(initial=0) < -8 or w.max(initial=0) > 7:
        raise ValueError("int4 weights: a [rows][K] array, K even, values in [-8, 7]")
    u = (w.astype(np.int16) & 0xF).astype(np.uint8)
    return np.ascontiguousarray((u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8).view(np.int8))

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdn.so")

#: every call the header declares, in declaration order
ABI_SYMBOLS = ("dn_create", "dn_set_state", "dn_get_state", "dn_step", "dn_stack_step", "dn_prefill", "dn_destroy",
               "dn_debug_fail_next", "dn_debug_expire_wait", "dn_profile_next_step", "dn_proj_i8_noalloc",
               "dn_device_bytes", "dn_step_kernels", "dn_strerror")


class DNError(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call} failed: {code} ({_strerror(code)})")


class dn_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_qk_heads", ctypes.c_int32),
                ("n_v_heads", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("conv_k", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("q_scale", ctypes.c_float), ("flags", ctypes.c_int32)]


class dn_weights(ctypes.Structure):
    _fields_ = [("w_in", ctypes.c_void_p), ("s_in", ctypes.c_void_p),
                ("w_conv", ctypes.c_void_p), ("w_norm", ctypes.c_void_p),
                ("w_out", ctypes.c_void_p), ("s_out", ctypes.c_void_p),
                ("w_ab", ctypes.c_void_p), ("s_ab", ctypes.c_void_p), ("gate_A", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gated_deltanet_hybrid_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, f32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    lib.dn_create.argtypes = [ctypes.POINTER(dn_config), ctypes.POINTER(dn_weights), vp,
                              ctypes.POINTER(ctypes.c_void_p)]
    lib.dn_create.restype = i32
    lib.dn_set_state.argtypes = [vp, i32, i32, f32p, f32p, vp, i32]
    lib.dn_set_state.restype = i32
    lib.dn_get_state.argtypes = [vp, i32, i32, f32p, f32p, vp, i32]
    lib.dn_get_state.restype = i32
    lib.dn_step.argtypes = [vp, i32, f32p, f32p, f32p, f32p, i32, vp]
    lib.dn_step.restype = i32
    lib.dn_stack_step.argtypes = [ctypes.POINTER(vp), i32, i32, f32p, f32p, f32p, ctypes.c_float, vp]
    lib.dn_stack_step.restype = i32
    lib.dn_prefill.argtypes = [vp, i32, i32, f32p, f32p, f32p, f32p, vp]
    lib.dn_prefill.restype = i32
    lib.dn_destroy.argtypes = [vp]
    lib.dn_destroy.restype = None
    lib.dn_debug_fail_next.argtypes = [vp, i32]
    lib.dn_debug_fail_next.restype = i32
    lib.dn_debug_expire_wait.argtypes = [vp, i32]
    lib.dn_debug_expire_wait.restype = i32
    lib.dn_profile_next_step.argtypes = [vp, ctypes.POINTER(ctypes.c_void_p)]
    lib.dn_profile_next_step.restype = i32
    lib.dn_proj_i8_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
    lib.dn_proj_i8_noalloc.restype = i32
    lib.dn_step_kernels.argtypes = [vp, i32]
    lib.dn_step_kernels.restype = i32
    lib.dn_device_bytes.argtypes = []
    lib.dn_device_bytes.restype = ctypes.c_int64
    lib.dn_strerror.argtypes = [i32]
    lib.dn_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _strerror(code: int) -> str:
    try:
        return load_library().dn_strerror(code).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(call: str, rc: int, check: bool) -> int:
    if check and rc != DN_OK:
        raise DNError(call, rc)
    return rc


def _is_cuda_tensor(a) -> bool:
    return hasattr(a, "is_cuda") and bool(a.is_cuda)


def _ptr(a, dtype: str):
    """(pointer, kind) of a contiguous array of the given dtype name."""
    if a is None:
        return None, None
    if hasattr(a, "data_ptr"):  # torch tensor
        import torch
        want = {"float32": torch.float32, "int32": torch.int32, "int8": torch.int8}[dtype]
        if a.dtype != want or not a.is_contiguous():
            raise TypeError(f"expected a contiguous {dtype} tensor")
        return a.data_ptr(), (DN_PTR_DEVICE if a.is_cuda else DN_PTR_HOST)
    arr = a
    if not isinstance(arr, np.ndarray) or arr.dtype != np.dtype(dtype) or not arr.flags.c_contiguous:
        raise TypeError(f"expected a C-contiguous numpy {dtype} array")
    return arr.ctypes.data, DN_PTR_HOST


def _same_kind(*kinds):
    ks = {k for k in kinds if k is not None}
    if len(ks) != 1:
        raise TypeError("all array arguments of one call must be on the host or all on the device")
    return ks.pop()


def _stream_of(stream, kind):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    if kind == DN_PTR_DEVICE:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(None)


def dn_create(cfg, weights, max_batch: int, stream=None, check: bool = True):
    """Create a layer from a DNConfig-like object and host weight arrays.
    Returns the layer handle (ctypes.c_void_p)."""
    lib = load_library()
    dev_gates = bool(getattr(cfg, "device_gates", False))
    int4 = bool(getattr(cfg, "int4", False))
    flags = ((DN_FLAG_KEY_GATE if getattr(cfg, "key_gate", False) else 0) | (DN_FLAG_DEVICE_GATES if dev_gates else 0)
             | (DN_FLAG_INT4_WEIGHTS if int4 else 0))
    mat = pack_int4 if int4 else (lambda a: np.ascontiguousarray(a, np.int8))
    c = dn_config(cfg.hidden, cfg.n_qk_heads, cfg.n_v_heads, cfg.dk, cfg.dv, cfg.conv_k,
                  int(max_batch), cfg.l2_eps, cfg.norm_eps, cfg.qscale, flags)
    arrs = [mat(weights.w_in), np.ascontiguousarray(weights.s_in, np.float32),
            np.ascontiguousarray(weights.w_conv, np.float32), np.ascontiguousarray(weights.w_norm, np.float32),
            mat(weights.w_out), np.ascontiguousarray(weights.s_out, np.float32)]
    if dev_gates:
        arrs += [mat(weights.w_ab), np.ascontiguousarray(weights.s_ab, np.float32),
                 np.ascontiguousarray(weights.gate_A, np.float32)]
    w = dn_weights(*[a.ctypes.data for a in arrs])
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
        except ImportError:  # pragma: no cover
            stream = None
    handle = ctypes.c_void_p()
    rc = lib.dn_create(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(stream), ctypes.byref(handle))
    _check("dn_create", rc, check)
    return handle if rc == DN_OK else rc


def dn_set_state(layer, seq0: int, S, ring, ring_pos, check: bool = True) -> int:
    lib = load_library()
    ps, ks = _ptr(S, "float32")
    pr, kr = _ptr(ring, "float32")
    pp, kp = _ptr(ring_pos, "int32")
    kind = _same_kind(ks, kr, kp)
    n = int(S.shape[0])
    rc = lib.dn_set_state(layer, int(seq0), n, ps, pr, pp, kind)
    return _check("dn_set_state", rc, check)


def dn_get_state(layer, seq0: int, n: int, S=None, ring=None, ring_pos=None, check: bool = True) -> int:
    """Fill whichever of S, ring, ring_pos are given (host or device arrays)."""
    lib = load_library()
    ps, ks = _ptr(S, "float32")
    pr, kr = _ptr(ring, "float32")
    pp, kp = _ptr(ring_pos, "int32")
    kind = _same_kind(ks, kr, kp)
    rc = lib.dn_get_state(layer, int(seq0), int(n), ps, pr, pp, kind)
    return _check("dn_get_state", rc, check)


def dn_step(layer, batch: int, x, g, beta, out, stream=None, check: bool = True) -> int:
    lib = load_library()
    px, kx = _ptr(x, "float32")
    pg, kg = _ptr(g, "float32")
    pb, kb = _ptr(beta, "float32")
    po, ko = _ptr(out, "float32")
    kind = _same_kind(kx, kg, kb, ko)
    rc = lib.dn_step(layer, int(batch), px, pg, pb, po, kind, _stream_of(stream, kind))
    return _check("dn_step", rc, check)


def dn_stack_step(layers, batch: int, h, g, beta, eps: float = 1e-6, stream=None, check: bool = True) -> int:
    """One token through a stack of layers (device tensors only): h [B][hidden]
    is read and overwritten, g/beta [n_layers][B][n_v_heads]."""
    lib = load_library()
    ph, kh = _ptr(h, "float32")
    pg, kg = _ptr(g, "float32")
    pb, kb = _ptr(beta, "float32")
    if _same_kind(kh, kg, kb) != DN_PTR_DEVICE:
        raise TypeError("dn_stack_step takes device tensors")
    arr = (ctypes.c_void_p * len(layers))(*[ctypes.c_void_p(getattr(l, "value", l)) for l in layers])
    rc = lib.dn_stack_step(arr, len(layers), int(batch), ph, pg, pb, float(eps), _stream_of(stream, DN_PTR_DEVICE))
    return _check("dn_stack_step", rc, check)


def dn_prefill(layer, batch: int, n_tokens: int, x, g, beta, out, stream=None, check: bool = True) -> int:
    """A prompt of n_tokens tokens for sequences [0, batch): x, out
    [batch][n_tokens][hidden], g [batch][n_tokens][heads](dk), beta
    [batch][n_tokens][heads] CUDA tensors (g, beta None with device gates)."""
    lib = load_library()
    px, kx = _ptr(x, "float32")
    pg, kg = _ptr(g, "float32")
    pb, kb = _ptr(beta, "float32")
    po, ko = _ptr(out, "float32")
    if _same_kind(kx, kg, kb, ko) != DN_PTR_DEVICE:
        raise TypeError("dn_prefill takes device tensors")
    rc = lib.dn_prefill(layer, int(batch), int(n_tokens), px, pg, pb, po, _stream_of(stream, DN_PTR_DEVICE))
    return _check("dn_prefill", rc, check)


def dn_destroy(layer) -> None:
    load_library().dn_destroy(layer)


def dn_debug_fail_next(layer, code: int, check: bool = True) -> int:
    return _check("dn_debug_fail_next", load_library().dn_debug_fail_next(layer, int(code)), check)


def dn_debug_expire_wait(layer, limit_us: int, check: bool = True) -> int:
    """The next dn_step first runs a bounded device wait that runs out after
    limit_us; the give-up surfaces at the next dn_get_state (DN_ECUDA)."""
    return _check("dn_debug_expire_wait", load_library().dn_debug_expire_wait(layer, int(limit_us)), check)


def dn_profile_next_step(layer, events, check: bool = True) -> int:
    """events: five torch.cuda.Event(enable_timing=True) (or None to cancel)."""
    lib = load_library()
    if events is None:
        return _check("dn_profile_next_step", lib.dn_profile_next_step(layer, None), check)
    if len(events) != 5:
        raise ValueError("dn_profile_next_step takes five events")
    arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return _check("dn_profile_next_step", lib.dn_profile_next_step(layer, arr), check)


def dn_proj_i8_noalloc(W, s, x, y, stream=None, check: bool = True) -> int:
    """y = s * (W x) for W int8 [M][K], s [M], x [B][K], y [B][M], all CUDA
    tensors; the library allocates nothing for the call (its scratch is a
    static device array)."""
    lib = load_library()
    pw, kw = _ptr(W, "int8")
    ps, ks = _ptr(s, "float32")
    px, kx = _ptr(x, "float32")
    py, ky = _ptr(y, "float32")
    if _same_kind(kw, ks, kx, ky) != DN_PTR_DEVICE:
        raise TypeError("dn_proj_i8_noalloc takes device tensors")
    M, K = int(W.shape[0]), int(W.shape[1])
    rc = lib.dn_proj_i8_noalloc(pw, ps, px, py, M, K, int(x.shape[0]), _stream_of(stream, DN_PTR_DEVICE))
    return _check("dn_proj_i8_noalloc", rc, check)


def dn_step_kernels(layer, batch: int) -> int:
    """Kernels one dn_step of `batch` sequences launches (0 if out of range)."""
    return int(load_library().dn_step_kernels(layer, int(batch)))


def dn_device_bytes() -> int:
    return int(load_library().dn_device_bytes())
