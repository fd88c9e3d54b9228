"""CPU fp64 oracle for the fused SwiGLU MLP (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does: it
shares no code with the CUDA library and neither imports the other.

The arithmetic lives in ``swiglu_oracle.c`` (plain C, fp64 loops, OpenMP
across rows), built here with gcc ``-O2 -ffp-contract=off`` and no fast-math
so that the same source gives the same fp64 results on x86 and on Arm.
This module is argument marshalling around it, plus ``rel_frob``.

Sources: "[RFC] Full-pipeline SwiGLU MLP with forward/backward
co-optimization" (Liger-Kernel #1347), sections "Summary" and "Correctness",
and its maintainer thread (the gate/down multiplier variant deferred to a
follow-up; the reading taken is stated in swiglu_oracle.c);
"Scope one-round FP32 SwiGLU to the exact Qwen3.5 contract" (xorl #51),
review section (one-round vs two-round programs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiglu_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

# storage types understood by the oracle
BF16, F16, F32, F64 = 0, 1, 2, 3
# rounding programs
EXACT, ONE_ROUND, TWO_ROUND = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (gcc, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_SO)
        vp, i64, ci, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_round.restype = ctypes.c_double
        lib.oracle_round.argtypes = [ctypes.c_double, ci]
        for name in ("oracle_sigmoid", "oracle_silu", "oracle_dsilu"):
            getattr(lib, name).restype = ctypes.c_double
            getattr(lib, name).argtypes = [ctypes.c_double]
        lib.oracle_decode.argtypes = [vp, ci, i64, dp]
        lib.oracle_round_array.argtypes = [dp, ci, i64, dp]
        cd = ctypes.c_double
        lib.oracle_fwd.argtypes = [vp, vp, vp, vp, ci, i64, i64, i64, ci, ci, dp, dp, dp, dp]
        lib.oracle_fwd_ex.argtypes = [vp, vp, vp, vp, ci, i64, i64, i64, ci, ci, cd, cd,
                                      dp, dp, dp, dp]
        lib.oracle_bwd.argtypes = [vp, vp, vp, vp, vp, ci, dp, dp, dp, i64, i64, i64, ci, ci,
                                   dp, dp, dp, dp, dp, dp]
        lib.oracle_bwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, dp, dp, dp, i64, i64, i64, ci, ci,
                                      cd, cd, dp, dp, dp, dp, dp, dp, dp, dp, dp]
        lib.oracle_rows.argtypes = [vp, vp, vp, vp, vp, ci, i64, i64, i64, vp, i64, ci, ci,
                                    dp, dp, dp, dp, dp, dp, dp]
        lib.oracle_cols.argtypes = [vp, vp, vp, vp, vp, ci, i64, i64, i64, vp, i64, ci, ci,
                                    dp, dp, dp]
        lib.oracle_elementwise.argtypes = [i64, dp, dp, dp, dp, dp, ci, ci, cd, dp, dp, dp]
        lib.oracle_num_threads.restype = ci
        _lib = lib
        return lib


# --------------------------------------------------------------------------
# array marshalling
# --------------------------------------------------------------------------

_NP_CODES = {np.dtype(np.float32): F32, np.dtype(np.float64): F64}


def storage_view(a) -> tuple[np.ndarray, int]:
    """Return (contiguous numpy array, storage code) for a numpy array or a CPU
    torch tensor.  bf16/fp16 torch tensors are passed as their raw 16-bit words."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(a, torch.Tensor):
        t = a.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy().view(np.uint16), F16
        a = t.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16), F16
    if a.dtype not in _NP_CODES:
        raise TypeError("oracle: unsupported input dtype %s" % a.dtype)
    return a, _NP_CODES[a.dtype]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _inputs(*arrays):
    views = [storage_view(a) for a in arrays]
    codes = {c for _, c in views}
    if len(codes) != 1:
        raise TypeError("oracle: all inputs must share one storage type")
    return [v for v, _ in views], codes.pop()


def round_to(x, dt: int) -> np.ndarray:
    """Round fp64 values to storage type dt (nearest, ties to even), as fp64."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib.oracle_round_array(_ptr(x), dt, x.size, _ptr(out))
    return out


def decode(a) -> np.ndarray:
    """Storage-type array -> exact fp64 values (shape kept)."""
    lib = _load()
    v, code = storage_view(a)
    out = np.empty(v.shape, dtype=np.float64)
    lib.oracle_decode(_ptr(v), code, v.size, _ptr(out))
    return out


def silu(g: float) -> float:
    return _load().oracle_silu(float(g))


def dsilu(g: float) -> float:
    return _load().oracle_dsilu(float(g))


def sigmoid(g: float) -> float:
    return _load().oracle_sigmoid(float(g))


def forward(X, Wg, Wu, Wd, mode: int = ONE_ROUND, dt: int | None = None,
            gate_mul: float = 1.0, down_mul: float = 1.0):
    """Full forward.  Returns dict of fp64 arrays G, U, A [M,H] and Y [M,D].
    ``gate_mul`` / ``down_mul``: A = SiLU(gate_mul X Wg^T) U, Y = down_mul A Wd^T
    (G is then the stored pre-activation gate_mul X Wg^T)."""
    lib = _load()
    (X, Wg, Wu, Wd), in_dt = _inputs(X, Wg, Wu, Wd)
    dt = in_dt if dt is None else dt
    M, D = X.shape
    H = Wg.shape[0]
    assert Wg.shape == (H, D) and Wu.shape == (H, D) and Wd.shape == (D, H)
    G = np.empty((M, H)); U = np.empty((M, H)); A = np.empty((M, H)); Y = np.empty((M, D))
    lib.oracle_fwd_ex(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd), in_dt, M, D, H, mode, dt,
                      float(gate_mul), float(down_mul), _ptr(G), _ptr(U), _ptr(A), _ptr(Y))
    return {"G": G, "U": U, "A": A, "Y": Y}


def backward(dY, X, Wg, Wu, Wd, fwd: dict, mode: int = ONE_ROUND, dt: int | None = None,
             gate_mul: float = 1.0, down_mul: float = 1.0, accumulate: dict | None = None):
    """Full backward from the oracle's own stored forward values ``fwd``.
    Returns dict of fp64 arrays dG, dU, dX, dWg, dWu, dWd.  ``accumulate``:
    the weight gradients already held ({"dWg", "dWu", "dWd"}, fp64 values),
    to which the new ones are added with one rounding; None overwrites."""
    lib = _load()
    (dY, X, Wg, Wu, Wd), in_dt = _inputs(dY, X, Wg, Wu, Wd)
    dt = in_dt if dt is None else dt
    M, D = X.shape
    H = Wg.shape[0]
    G = np.ascontiguousarray(fwd["G"], dtype=np.float64)
    U = np.ascontiguousarray(fwd["U"], dtype=np.float64)
    A = np.ascontiguousarray(fwd["A"], dtype=np.float64)
    out = {k: np.empty(s) for k, s in (("dG", (M, H)), ("dU", (M, H)), ("dX", (M, D)),
                                         ("dWg", (H, D)), ("dWu", (H, D)), ("dWd", (D, H)))}
    acc = {}
    null = ctypes.c_void_p(0)
    for k, shape in (("dWg", (H, D)), ("dWu", (H, D)), ("dWd", (D, H))):
        if accumulate is not None:
            acc[k] = np.ascontiguousarray(accumulate[k], dtype=np.float64)
            assert acc[k].shape == shape
    ap = {k: (_ptr(acc[k]) if k in acc else null) for k in ("dWg", "dWu", "dWd")}
    lib.oracle_bwd_ex(_ptr(dY), _ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd), in_dt,
                      _ptr(G), _ptr(U), _ptr(A), M, D, H, mode, dt, float(gate_mul),
                      float(down_mul), ap["dWg"], ap["dWu"], ap["dWd"],
                      _ptr(out["dG"]), _ptr(out["dU"]), _ptr(out["dX"]),
                      _ptr(out["dWg"]), _ptr(out["dWu"]), _ptr(out["dWd"]))
    return out


def sampled_rows(X, Wg, Wu, Wd, dY, rows, mode: int = ONE_ROUND, dt: int | None = None):
    """Exact rows of G, U, A, Y, dG, dU, dX for the token indices ``rows``."""
    lib = _load()
    (X, Wg, Wu, Wd, dY), in_dt = _inputs(X, Wg, Wu, Wd, dY)
    dt = in_dt if dt is None else dt
    M, D = X.shape
    H = Wg.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.size
    assert rows.min() >= 0 and rows.max() < M
    o = {k: np.empty((R, H)) for k in ("G", "U", "A", "dG", "dU")}
    o["Y"] = np.empty((R, D)); o["dX"] = np.empty((R, D))
    lib.oracle_rows(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(dY), in_dt, M, D, H,
                    _ptr(rows), R, mode, dt, _ptr(o["G"]), _ptr(o["U"]), _ptr(o["A"]),
                    _ptr(o["Y"]), _ptr(o["dG"]), _ptr(o["dU"]), _ptr(o["dX"]))
    return o


def sampled_cols(X, Wg, Wu, Wd, dY, cols, mode: int = ONE_ROUND, dt: int | None = None):
    """Rows cols of dWg and dWu, and columns cols of dWd (returned transposed,
    as [C, D]), each reduced over all M token rows."""
    lib = _load()
    (X, Wg, Wu, Wd, dY), in_dt = _inputs(X, Wg, Wu, Wd, dY)
    dt = in_dt if dt is None else dt
    M, D = X.shape
    H = Wg.shape[0]
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = cols.size
    assert cols.min() >= 0 and cols.max() < H
    o = {k: np.empty((C, D)) for k in ("dWg", "dWu", "dWdT")}
    lib.oracle_cols(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(dY), in_dt, M, D, H,
                    _ptr(cols), C, mode, dt, _ptr(o["dWg"]), _ptr(o["dWu"]), _ptr(o["dWdT"]))
    return o


def elementwise(dt: int, g=None, u=None, gs=None, us=None, da=None, mode: int = ONE_ROUND,
                gate_mul: float = 1.0):
    """The elementwise SwiGLU stage alone, on 1-D fp64 arrays of exact values.
    Forward (g, u given): A from the sums g, u (gate multiplier applied; gs, us
    their stored values, needed by the two-round program and defaulting to
    rnd(g), rnd(u)).  Backward (da, gs, us given): dG, dU from dA and the
    stored gs, us.  Returns a dict with "A" and/or "dG", "dU"."""
    lib = _load()
    arr = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64).ravel()
    g, u, gs, us, da = arr(g), arr(u), arr(gs), arr(us), arr(da)
    fwd = g is not None
    bwd = da is not None
    if fwd:
        assert u is not None and u.size == g.size
        gs = round_to(g, dt) if gs is None else gs
        us = round_to(u, dt) if us is None else us
    if bwd:
        assert gs is not None and us is not None and gs.size == da.size == us.size
    n = (g if fwd else da).size
    z = np.zeros(n)
    out = {}
    null = ctypes.c_void_p(0)
    if fwd:
        out["A"] = np.empty(n)
    if bwd:
        out["dG"] = np.empty(n)
        out["dU"] = np.empty(n)
    p = lambda a: _ptr(a if a is not None else z)
    lib.oracle_elementwise(n, p(g), p(u), p(gs), p(us), p(da), mode, dt, float(gate_mul),
                           _ptr(out["A"]) if fwd else null, _ptr(out["dG"]) if bwd else null,
                           _ptr(out["dU"]) if bwd else null)
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def rel_frob(got, ref) -> float:
    """||got - ref||_F / ||ref||_F in fp64."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return float(num / den) if den > 0 else float(num)
