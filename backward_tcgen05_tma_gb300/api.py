"""Thin Python binding of libswiglu_mlp.so (include/swiglu_mlp.h).

Argument marshalling only: torch supplies device memory (``data_ptr()``) and
the current CUDA stream; every step of the MLP runs in the library's CUDA
kernels.  If the library is missing this module raises -- there is no
fallback path.

The three calls keep the C ABI's names:

* ``swiglu_mlp_fwd(X, Wgu, Wd)``        -> (Y, saved)      saved = [G | U | A]
* ``swiglu_mlp_fwd_nograd(X, Wgu, Wd)`` -> (Y, A)
* ``swiglu_mlp_bwd(dY, X, Wgu, Wd, saved)`` -> (dX, dWgu, dWd); consumes saved

Outputs may be passed in (``out=`` dicts) to avoid allocation.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswiglu_mlp.so")
# the same library compiled with -DSWIGLU_DEBUG (device index checks)
DEBUG_LIB_PATH = os.path.join(_HERE, "libswiglu_mlp_debug.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "swiglu_mlp.h")

SWIGLU_BF16, SWIGLU_F16, SWIGLU_F32_IEEE = 0, 1, 2
SWIGLU_OP_FWD, SWIGLU_OP_FWD_NOGRAD, SWIGLU_OP_BWD = 0, 1, 2
STATUS = {0: "SWIGLU_OK", 1: "SWIGLU_ERR_INVALID_ARG", 2: "SWIGLU_ERR_ALIGNMENT",
          3: "SWIGLU_ERR_UNSUPPORTED", 4: "SWIGLU_ERR_WORKSPACE", 5: "SWIGLU_ERR_CUDA",
          6: "SWIGLU_ERR_DEVICE_TIMEOUT", 7: "SWIGLU_ERR_DEVICE_BOUNDS"}

_DT = {torch.bfloat16: SWIGLU_BF16, torch.float16: SWIGLU_F16, torch.float32: SWIGLU_F32_IEEE}

_lock = threading.Lock()
_lib = None
_loaded = {}  # path -> CDLL
_use_debug = False


class SwigluError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, STATUS.get(code, code), status_string(code)))


class Options(ctypes.Structure):
    """swiglu_mlp_options: gate/down multipliers and weight-gradient accumulation."""
    _fields_ = [("gate_multiplier", ctypes.c_float), ("down_multiplier", ctypes.c_float),
                ("accumulate", ctypes.c_int)]


def _opts(gate_mul: float, down_mul: float, accumulate: bool):
    """NULL for the standard MLP, else a pointer to an Options."""
    if gate_mul == 1.0 and down_mul == 1.0 and not accumulate:
        return ctypes.c_void_p(0)
    return ctypes.byref(Options(float(gate_mul), float(down_mul), 1 if accumulate else 0))


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built): the release
    build, or the debug build while use_debug_library(True) is in effect."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(DEBUG_LIB_PATH if _use_debug else LIB_PATH)
        return _lib


def use_debug_library(on: bool) -> bool:
    """Routes every later call of this module to the debug build
    (libswiglu_mlp_debug.so: device index checks, SWIGLU_ERR_DEVICE_BOUNDS)
    or back to the release build; returns the previous setting.  Both stay
    loaded; each keeps its own process-wide settings (wait limit, SM-pair
    and few-token modes)."""
    global _lib, _use_debug
    with _lock:
        prev = _use_debug
        _use_debug = bool(on)
        _lib = None
    lib()
    return prev


def _load(path: str) -> ctypes.CDLL:
    if path in _loaded:
        return _loaded[path]
    if not os.path.exists(path):
        raise ImportError("%s is not built (run __graft_entry__.build() or python -m "
                          "backward_tcgen05_tma_gb300.build); no fallback exists"
                          % os.path.basename(path))
    L = ctypes.CDLL(path)
    vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.swiglu_mlp_element_bytes.restype = sz
    L.swiglu_mlp_element_bytes.argtypes = [ci]
    L.swiglu_mlp_saved_bytes.restype = sz
    L.swiglu_mlp_saved_bytes.argtypes = [i64, i64, ci]
    L.swiglu_mlp_workspace_bytes.restype = sz
    L.swiglu_mlp_workspace_bytes.argtypes = [i64, i64, i64, ci, ci]
    L.swiglu_mlp_workspace_min_bytes.restype = sz
    L.swiglu_mlp_workspace_min_bytes.argtypes = [i64, i64, i64, ci, ci]
    L.swiglu_mlp_fwd.restype = ci
    L.swiglu_mlp_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp, sz, vp]
    L.swiglu_mlp_fwd_nograd.restype = ci
    L.swiglu_mlp_fwd_nograd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp, sz, vp]
    L.swiglu_mlp_fwd_nograd_noalloc.restype = ci
    L.swiglu_mlp_fwd_nograd_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    L.swiglu_mlp_graph_create_fwd_nograd.restype = ci
    L.swiglu_mlp_graph_create_fwd_nograd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp,
                                                     sz, ctypes.POINTER(vp)]
    L.swiglu_mlp_graph_launch.restype = ci
    L.swiglu_mlp_graph_launch.argtypes = [vp, vp]
    L.swiglu_mlp_graph_destroy.restype = ci
    L.swiglu_mlp_graph_destroy.argtypes = [vp]
    op = ctypes.c_void_p
    L.swiglu_mlp_fwd_ex.restype = ci
    L.swiglu_mlp_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, op, vp, sz, vp]
    L.swiglu_mlp_fwd_nograd_ex.restype = ci
    L.swiglu_mlp_fwd_nograd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, op, vp, sz,
                                           vp]
    L.swiglu_mlp_bwd_ex.restype = ci
    L.swiglu_mlp_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, op, vp,
                                    sz, vp]
    L.swiglu_mlp_packed_weights_bytes.restype = sz
    L.swiglu_mlp_packed_weights_bytes.argtypes = [i64, i64, ci]
    L.swiglu_mlp_pack_weights.restype = ci
    L.swiglu_mlp_pack_weights.argtypes = [vp, vp, vp, i64, i64, ci, vp]
    L.swiglu_mlp_fwd_nograd_packed.restype = ci
    L.swiglu_mlp_fwd_nograd_packed.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, op, vp, sz, vp]
    L.swiglu_mlp_bwd.restype = ci
    L.swiglu_mlp_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, vp, sz, vp]
    L.swiglu_mlp_query_error.restype = ci
    L.swiglu_mlp_query_error.argtypes = [vp, vp]
    L.swiglu_status_string.restype = ctypes.c_char_p
    L.swiglu_status_string.argtypes = [ci]
    L.swiglu_mlp_set_wait_limit_ns.restype = ctypes.c_uint64
    L.swiglu_mlp_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.swiglu_mlp_inject_stall_once.restype = None
    L.swiglu_mlp_inject_stall_once.argtypes = [ci]
    L.swiglu_mlp_last_launch_count.restype = ci
    L.swiglu_mlp_last_launch_count.argtypes = []
    fp = ctypes.c_void_p
    L.swiglu_mlp_test_elementwise.restype = ci
    L.swiglu_mlp_test_elementwise.argtypes = [ci, i64, fp, fp, vp, vp, vp, fp, vp, vp, vp, vp,
                                              ctypes.c_float, ctypes.c_float, vp]
    L.swiglu_mlp_set_cta_pairs.restype = ci
    L.swiglu_mlp_set_cta_pairs.argtypes = [ci]
    L.swiglu_mlp_set_nograd_fused.restype = ci
    L.swiglu_mlp_set_nograd_fused.argtypes = [ci]
    L.swiglu_mlp_set_wide_tiles.restype = ci
    L.swiglu_mlp_set_wide_tiles.argtypes = [ci]
    L.swiglu_mlp_profile_enable.restype = None
    L.swiglu_mlp_profile_enable.argtypes = [ci]
    L.swiglu_mlp_profile_read.restype = ci
    L.swiglu_mlp_profile_read.argtypes = [ci, vp, vp]
    L.swiglu_mlp_kernel_name.restype = ctypes.c_char_p
    L.swiglu_mlp_kernel_name.argtypes = [ci]
    L.swiglu_mlp_debug_build.restype = ci
    L.swiglu_mlp_debug_build.argtypes = []
    L.swiglu_mlp_debug_narrow_once.restype = None
    L.swiglu_mlp_debug_narrow_once.argtypes = [ci]
    _loaded[path] = L
    return L


def declared_symbols() -> list[str]:
    """Function names declared in include/swiglu_mlp.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swiglu_(?:mlp|status)_\w+)\s*\(", text)))


def status_string(code: int) -> str:
    return lib().swiglu_status_string(code).decode()


def dtype_code(dtype: torch.dtype) -> int:
    if dtype not in _DT:
        raise TypeError("unsupported dtype %s (bf16, fp16 or fp32)" % dtype)
    return _DT[dtype]


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(code: int, where: str):
    if code != 0:
        raise SwigluError(code, where)


def _device_check(ws, where: str):
    """While the debug build is in use: wait for the call and raise on the
    device status in its workspace (a failed index check, a timeout).  The
    release build returns at once, as every call is asynchronous."""
    if _use_debug:
        code = int(lib().swiglu_mlp_query_error(_ptr(ws), _stream(ws.device)))
        if code != 0:
            raise SwigluError(code, where + " (device)")


def workspace(M: int, D: int, H: int, dtype: torch.dtype, op: int, device,
              minimal: bool = False) -> torch.Tensor:
    """A zero-filled workspace: the recommended size, or with ``minimal`` the
    smallest accepted one (stream-K off where its partials would not fit)."""
    f = lib().swiglu_mlp_workspace_min_bytes if minimal else lib().swiglu_mlp_workspace_bytes
    n = f(M, D, H, dtype_code(dtype), op)
    return torch.zeros(int(n), dtype=torch.uint8, device=device)


def _dims(X, Wgu, Wd):
    M, D = X.shape
    H = Wgu.shape[0] // 2
    if Wgu.shape != (2 * H, D) or Wd.shape != (D, H):
        raise ValueError("shape mismatch: X %s, Wgu %s, Wd %s" % (tuple(X.shape), tuple(Wgu.shape),
                                                                   tuple(Wd.shape)))
    for t in (X, Wgu, Wd):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != X.dtype:
            raise ValueError("inputs must be contiguous CUDA tensors of one dtype")
    return M, D, H


def swiglu_mlp_fwd(X, Wgu, Wd, out: dict | None = None, ws=None, gate_mul: float = 1.0,
                   down_mul: float = 1.0):
    """Training forward: returns (Y [M,D], saved [M,3H]).  ``gate_mul`` /
    ``down_mul``: the multiplier variant (swiglu_mlp_fwd_ex)."""
    M, D, H = _dims(X, Wgu, Wd)
    out = out or {}
    Y = out.get("Y")
    Y = torch.empty(M, D, dtype=X.dtype, device=X.device) if Y is None else Y
    saved = out.get("saved")
    saved = torch.empty(M, 3 * H, dtype=X.dtype, device=X.device) if saved is None else saved
    ws = workspace(M, D, H, X.dtype, SWIGLU_OP_FWD, X.device) if ws is None else ws
    _check(lib().swiglu_mlp_fwd_ex(_ptr(X), _ptr(Wgu), _ptr(Wd), _ptr(Y), _ptr(saved), M, D, H,
                                   dtype_code(X.dtype), _opts(gate_mul, down_mul, False),
                                   _ptr(ws), ws.numel(), _stream(X.device)),
           "swiglu_mlp_fwd")
    _device_check(ws, "swiglu_mlp_fwd")
    return Y, saved


def swiglu_mlp_fwd_nograd(X, Wgu, Wd, out: dict | None = None, ws=None, gate_mul: float = 1.0,
                          down_mul: float = 1.0):
    """Inference forward: returns (Y [M,D], A [M,H]); G and U are never stored."""
    M, D, H = _dims(X, Wgu, Wd)
    out = out or {}
    Y = out.get("Y")
    Y = torch.empty(M, D, dtype=X.dtype, device=X.device) if Y is None else Y
    A = out.get("A")
    A = torch.empty(M, H, dtype=X.dtype, device=X.device) if A is None else A
    ws = workspace(M, D, H, X.dtype, SWIGLU_OP_FWD_NOGRAD, X.device) if ws is None else ws
    _check(lib().swiglu_mlp_fwd_nograd_ex(_ptr(X), _ptr(Wgu), _ptr(Wd), _ptr(Y), _ptr(A), M, D,
                                          H, dtype_code(X.dtype),
                                          _opts(gate_mul, down_mul, False), _ptr(ws), ws.numel(),
                                          _stream(X.device)),
           "swiglu_mlp_fwd_nograd")
    _device_check(ws, "swiglu_mlp_fwd_nograd")
    return Y, A


def swiglu_mlp_fwd_nograd_noalloc(X, Wgu, Wd, out: dict | None = None):
    """Few-token no-grad forward that allocates nothing in the library (its
    scratch is a static device array): returns (Y [M,D], A [M,H])."""
    M, D, H = _dims(X, Wgu, Wd)
    out = out or {}
    Y = out.get("Y")
    Y = torch.empty(M, D, dtype=X.dtype, device=X.device) if Y is None else Y
    A = out.get("A")
    A = torch.empty(M, H, dtype=X.dtype, device=X.device) if A is None else A
    _check(lib().swiglu_mlp_fwd_nograd_noalloc(_ptr(X), _ptr(Wgu), _ptr(Wd), _ptr(Y), _ptr(A), M,
                                               D, H, dtype_code(X.dtype), _stream(X.device)),
           "swiglu_mlp_fwd_nograd_noalloc")
    return Y, A


def swiglu_mlp_pack_weights(Wgu, Wd, packed=None) -> torch.Tensor:
    """The packed copy of (Wgu [2H,D], Wd [D,H]) that
    swiglu_mlp_fwd_nograd_packed streams (a uint8 device tensor)."""
    H2, D = Wgu.shape
    H = H2 // 2
    if Wgu.shape != (2 * H, D) or Wd.shape != (D, H):
        raise ValueError("expected Wgu [2H, D] and Wd [D, H]")
    n = int(lib().swiglu_mlp_packed_weights_bytes(D, H, dtype_code(Wgu.dtype)))
    if n == 0:
        raise SwigluError(3, "swiglu_mlp_pack_weights")
    packed = torch.empty(n, dtype=torch.uint8, device=Wgu.device) if packed is None else packed
    if packed.numel() < n:
        raise ValueError("packed buffer too small")
    _check(lib().swiglu_mlp_pack_weights(_ptr(Wgu), _ptr(Wd), _ptr(packed), D, H,
                                         dtype_code(Wgu.dtype), _stream(Wgu.device)),
           "swiglu_mlp_pack_weights")
    return packed


def swiglu_mlp_fwd_nograd_packed(X, packed, H: int, out: dict | None = None, ws=None,
                                 gate_mul: float = 1.0, down_mul: float = 1.0):
    """Few-token (M <= 64) no-grad forward on weights packed by
    swiglu_mlp_pack_weights: returns (Y [M,D], A [M,H])."""
    M, D = X.shape
    out = out or {}
    Y = out.get("Y")
    Y = torch.empty(M, D, dtype=X.dtype, device=X.device) if Y is None else Y
    A = out.get("A")
    A = torch.empty(M, H, dtype=X.dtype, device=X.device) if A is None else A
    ws = workspace(M, D, H, X.dtype, SWIGLU_OP_FWD_NOGRAD, X.device) if ws is None else ws
    _check(lib().swiglu_mlp_fwd_nograd_packed(_ptr(X), _ptr(packed), _ptr(Y), _ptr(A), M, D, H,
                                              dtype_code(X.dtype),
                                              _opts(gate_mul, down_mul, False), _ptr(ws),
                                              ws.numel(), _stream(X.device)),
           "swiglu_mlp_fwd_nograd_packed")
    _device_check(ws, "swiglu_mlp_fwd_nograd_packed")
    return Y, A


class FwdNogradGraph:
    """A no-grad forward recorded once as a CUDA graph (swiglu_mlp_graph_*)
    on static buffers ``X`` [M,D], ``Y`` [M,D], ``A`` [M,H] and a workspace;
    each call copies new tokens into ``X`` (unless they are ``X`` itself),
    replays the graph on the current stream and returns ``Y``.  Holds
    references to every buffer the graph reads or writes."""

    def __init__(self, Wgu, Wd, M: int, X=None, out: dict | None = None, ws=None):
        D = Wd.shape[0]
        dev, dt = Wgu.device, Wgu.dtype
        self.X = torch.empty(M, D, dtype=dt, device=dev) if X is None else X
        M, D, H = _dims(self.X, Wgu, Wd)
        out = out or {}
        self.Y = out.get("Y")
        self.Y = torch.empty(M, D, dtype=dt, device=dev) if self.Y is None else self.Y
        self.A = out.get("A")
        self.A = torch.empty(M, H, dtype=dt, device=dev) if self.A is None else self.A
        self.ws = workspace(M, D, H, dt, SWIGLU_OP_FWD_NOGRAD, dev) if ws is None else ws
        self.Wgu, self.Wd = Wgu, Wd
        torch.cuda.synchronize(dev)  # the workspace's zero-fill is complete before any replay
        h = ctypes.c_void_p(0)
        L = lib()
        with torch.cuda.device(dev):
            _check(L.swiglu_mlp_graph_create_fwd_nograd(
                _ptr(self.X), _ptr(Wgu), _ptr(Wd), _ptr(self.Y), _ptr(self.A), M, D, H,
                dtype_code(dt), _ptr(self.ws), self.ws.numel(), ctypes.byref(h)),
                "swiglu_mlp_graph_create_fwd_nograd")
        self._h = h
        self._L = L

    def launch(self, stream=None):
        s = torch.cuda.current_stream(self.X.device) if stream is None else stream
        _check(self._L.swiglu_mlp_graph_launch(self._h, ctypes.c_void_p(s.cuda_stream)),
               "swiglu_mlp_graph_launch")
        if _use_debug:  # as _device_check, with the graph's own library
            code = int(self._L.swiglu_mlp_query_error(_ptr(self.ws),
                                                      ctypes.c_void_p(s.cuda_stream)))
            if code != 0:
                raise SwigluError(code, "swiglu_mlp_graph_launch (device)")

    def __call__(self, x=None):
        if x is not None and x.data_ptr() != self.X.data_ptr():
            self.X.copy_(x)
        self.launch()
        return self.Y

    def close(self):
        """Destroys the graph after pending launches on this device finish
        (so the buffers it holds may be freed afterwards)."""
        if getattr(self, "_h", None) is not None and self._h.value:
            torch.cuda.synchronize(self.X.device)
            _check(self._L.swiglu_mlp_graph_destroy(self._h), "swiglu_mlp_graph_destroy")
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def swiglu_mlp_bwd(dY, X, Wgu, Wd, saved, out: dict | None = None, ws=None,
                   gate_mul: float = 1.0, down_mul: float = 1.0, accumulate: bool = False):
    """Backward: returns (dX [M,D], dWgu [2H,D], dWd [D,H]).  Overwrites the
    G/U columns of ``saved`` with dG/dU (a second call on it is undefined).
    ``accumulate``: add into the dWgu / dWd given in ``out`` (beta = 1)."""
    M, D, H = _dims(X, Wgu, Wd)
    if dY.shape != (M, D) or saved.shape != (M, 3 * H):
        raise ValueError("dY/saved shape mismatch")
    out = out or {}
    dX = out.get("dX")
    dX = torch.empty(M, D, dtype=X.dtype, device=X.device) if dX is None else dX
    dWgu = out.get("dWgu")
    dWgu = torch.empty(2 * H, D, dtype=X.dtype, device=X.device) if dWgu is None else dWgu
    dWd = out.get("dWd")
    dWd = torch.empty(D, H, dtype=X.dtype, device=X.device) if dWd is None else dWd
    ws = workspace(M, D, H, X.dtype, SWIGLU_OP_BWD, X.device) if ws is None else ws
    if accumulate and (out.get("dWgu") is None or out.get("dWd") is None):
        raise ValueError("accumulate needs the held dWgu and dWd in out")
    _check(lib().swiglu_mlp_bwd_ex(_ptr(dY), _ptr(X), _ptr(Wgu), _ptr(Wd), _ptr(saved),
                                   _ptr(dX), _ptr(dWgu), _ptr(dWd), M, D, H,
                                   dtype_code(X.dtype), _opts(gate_mul, down_mul, accumulate),
                                   _ptr(ws), ws.numel(), _stream(X.device)),
           "swiglu_mlp_bwd")
    _device_check(ws, "swiglu_mlp_bwd")
    return dX, dWgu, dWd


def swiglu_mlp_query_error(ws) -> int:
    """Synchronises the current stream and returns the device error status."""
    return int(lib().swiglu_mlp_query_error(_ptr(ws), _stream(ws.device)))


def swiglu_mlp_set_wait_limit_ns(ns: int) -> int:
    return int(lib().swiglu_mlp_set_wait_limit_ns(int(ns)))


def swiglu_mlp_inject_stall_once(on: bool | int = True) -> None:
    """True / 1: stall the next tensor-core launch; n: the n-th from now;
    False / 0: clear."""
    lib().swiglu_mlp_inject_stall_once(int(on))


def swiglu_mlp_last_launch_count() -> int:
    return int(lib().swiglu_mlp_last_launch_count())


def swiglu_mlp_set_cta_pairs(mode: int = 1) -> int:
    """Tensor-core GEMMs on SM pairs: 1 = by size (default), 2 = always,
    0 = never; returns the previous mode."""
    return int(lib().swiglu_mlp_set_cta_pairs(int(mode)))


def swiglu_mlp_set_wide_tiles(mode: int = 1) -> int:
    """Weight-gradient and dX GEMMs on SM pairs: 1 = 512-column tiles by
    size (the default), 0 = 256-column tiles, 2 = 512-column tiles always;
    returns the previous mode."""
    return int(lib().swiglu_mlp_set_wide_tiles(int(mode)))


def swiglu_mlp_set_nograd_fused(mode: int = 0) -> int:
    """Few-token no-grad calls: 0 two kernels (the default), 1 the fused kernel
    for 33..64 tokens, 2 always the fused kernel; returns the previous mode."""
    return int(lib().swiglu_mlp_set_nograd_fused(int(mode)))


def swiglu_mlp_profile_enable(on: bool = True) -> None:
    lib().swiglu_mlp_profile_enable(1 if on else 0)


def swiglu_mlp_profile_read() -> dict:
    """{kernel name: (launches, total device ms)} since the previous read."""
    n = 64
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    k = lib().swiglu_mlp_profile_read(n, ctypes.cast(launches, ctypes.c_void_p),
                                      ctypes.cast(ms, ctypes.c_void_p))
    if k < 0:
        raise SwigluError(5, "swiglu_mlp_profile_read")
    out = {}
    for i in range(k):
        if launches[i]:
            out[lib().swiglu_mlp_kernel_name(i).decode()] = (int(launches[i]), float(ms[i]))
    return out


def swiglu_mlp_test_elementwise(dtype: torch.dtype, acc_g=None, acc_u=None, dA=None, gs=None,
                                us=None, gate_mul: float = 1.0, down_mul: float = 1.0) -> dict:
    """Test hook: the tensor-core epilogues' elementwise stage applied to the
    given values (1-D CUDA tensors, length a multiple of 32).  Forward from
    fp32 accumulators acc_g, acc_u -> {"A", "G", "U"}; backward from the fp32
    dA and the stored gs, us (``dtype``) -> {"dG", "dU"}."""
    fwd, bwd = acc_g is not None, dA is not None
    ref = acc_g if fwd else dA
    n = ref.numel()
    out = {}
    new = lambda: torch.empty(n, dtype=dtype, device=ref.device)
    if fwd:
        out = {"A": new(), "G": new(), "U": new()}
    if bwd:
        out.update({"dG": new(), "dU": new()})
    _check(lib().swiglu_mlp_test_elementwise(
        dtype_code(dtype), n, _ptr(acc_g), _ptr(acc_u), _ptr(out.get("A")), _ptr(out.get("G")),
        _ptr(out.get("U")), _ptr(dA), _ptr(gs), _ptr(us), _ptr(out.get("dG")),
        _ptr(out.get("dU")), float(gate_mul), float(down_mul), _stream(ref.device)),
        "swiglu_mlp_test_elementwise")
    return out
