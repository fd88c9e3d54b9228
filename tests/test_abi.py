"""Host-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every declared entry point, and rejects bad arguments before any CUDA call.
No GPU needed (no compute call is made)."""
import ctypes

import pytest

from backward_tcgen05_tma_gb300 import api, build

pytestmark = pytest.mark.filterwarnings("ignore")

OK, INVALID, ALIGN, UNSUP, WSERR = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def test_library_exports_every_declared_symbol(L):
    names = api.declared_symbols()
    for must in ("swiglu_mlp_fwd", "swiglu_mlp_fwd_nograd", "swiglu_mlp_bwd",
                 "swiglu_mlp_query_error", "swiglu_status_string", "swiglu_mlp_workspace_bytes",
                 "swiglu_mlp_saved_bytes"):
        assert must in names
    for n in names:
        assert hasattr(L, n), n


def test_debug_library_exports_the_same_symbols_and_says_what_it_is(L):
    # libswiglu_mlp_debug.so: the same sources with the device index checks
    D = api._load(api.DEBUG_LIB_PATH)
    for n in api.declared_symbols():
        assert hasattr(D, n), n
    assert D.swiglu_mlp_debug_build() == 1 and L.swiglu_mlp_debug_build() == 0
    assert D.swiglu_status_string(7) == b"device index check failed (debug build)"
    assert api.STATUS[7] == "SWIGLU_ERR_DEVICE_BOUNDS"
    # argument checks are the release build's
    for args in [(None, None, None, None, None, 4, 64, 64, 0, None, 0, None),
                 (None, None, None, None, None, -1, 64, 64, 0, None, 0, None),
                 (None, None, None, None, None, 4, 60, 64, 0, None, 0, None)]:
        assert D.swiglu_mlp_fwd(*args) == L.swiglu_mlp_fwd(*args) != OK


def test_sizes(L):
    assert L.swiglu_mlp_element_bytes(0) == 2
    assert L.swiglu_mlp_element_bytes(1) == 2
    assert L.swiglu_mlp_element_bytes(2) == 4
    assert L.swiglu_mlp_element_bytes(7) == 0
    # saved = [G | U | A] = M * 3H elements
    assert L.swiglu_mlp_saved_bytes(65536, 11008, 0) == 65536 * 3 * 11008 * 2
    assert L.swiglu_mlp_saved_bytes(32, 176, 2) == 32 * 528 * 4
    for op in (0, 1, 2):
        assert L.swiglu_mlp_workspace_bytes(65536, 4096, 11008, 0, op) >= 4
    # packed weights: 16 KB blocks, ceil(H/64) x ceil(D/64) for gate/up and
    # ceil(D/128) x ceil(H/64) for down; bf16/fp16 only
    assert L.swiglu_mlp_packed_weights_bytes(4096, 11008, 0) == (172 * 64 + 32 * 172) * 16384
    assert L.swiglu_mlp_packed_weights_bytes(72, 80, 1) == (2 * 2 + 1 * 2) * 16384
    assert L.swiglu_mlp_packed_weights_bytes(64, 64, 2) == 0
    assert L.swiglu_mlp_packed_weights_bytes(0, 64, 0) == 0


def test_packed_entry_points_check_arguments_first(L):
    P = ctypes.c_void_p(256)
    N = ctypes.c_void_p(0)
    assert L.swiglu_mlp_pack_weights(P, P, P, 64, 128, 2, N) == UNSUP
    assert L.swiglu_mlp_pack_weights(P, P, N, 64, 128, 0, N) == INVALID
    assert L.swiglu_mlp_pack_weights(P, P, P, 60, 128, 0, N) == ALIGN
    assert L.swiglu_mlp_pack_weights(P, P, ctypes.c_void_p(264), 64, 128, 0, N) == ALIGN
    ws = ctypes.c_void_p(4096)
    big = 1 << 30
    assert L.swiglu_mlp_fwd_nograd_packed(P, P, P, P, 65, 64, 128, 0, N, ws, big, N) == UNSUP
    assert L.swiglu_mlp_fwd_nograd_packed(P, P, P, P, 4, 64, 128, 2, N, ws, big, N) == UNSUP
    assert L.swiglu_mlp_fwd_nograd_packed(P, N, P, P, 4, 64, 128, 0, N, ws, big, N) == INVALID
    assert L.swiglu_mlp_fwd_nograd_packed(P, P, P, P, 4, 64, 128, 0, N, ws, 8, N) == WSERR
    assert L.swiglu_mlp_fwd_nograd_packed(P, P, P, P, 0, 64, 128, 0, N, ws, big, N) == OK
    assert L.swiglu_mlp_last_launch_count() == 0


def test_status_strings(L):
    for code in range(7):
        assert api.status_string(code)
    assert "timed out" in api.status_string(6)


P = ctypes.c_void_p(0x10000)          # an aligned fake device address (never dereferenced)
P_MIS = ctypes.c_void_p(0x10002)
N = ctypes.c_void_p(0)


BIG = 1 << 30  # more workspace than any call here needs (never dereferenced)


def _fwd(L, X=P, W=P, Wd=P, Y=P, S=P, M=128, D=64, H=128, dt=0, ws=P, wsb=BIG):
    return L.swiglu_mlp_fwd(X, W, Wd, Y, S, M, D, H, dt, ws, wsb, N)


def test_argument_errors_are_reported_before_any_launch(L):
    assert _fwd(L, X=N) == INVALID
    assert _fwd(L, Y=N) == INVALID
    assert _fwd(L, D=0) == INVALID
    assert _fwd(L, H=-8) == INVALID
    assert _fwd(L, M=-1) == INVALID
    assert _fwd(L, dt=9) == INVALID
    assert _fwd(L, X=P_MIS) == ALIGN
    assert _fwd(L, D=60) == ALIGN          # bf16 needs D % 8 == 0
    assert _fwd(L, H=124) == ALIGN
    assert _fwd(L, ws=N) == WSERR
    assert _fwd(L, wsb=8) == WSERR
    assert _fwd(L, M=2 ** 31) == UNSUP
    assert L.swiglu_mlp_fwd_nograd(N, P, P, P, P, 4, 64, 128, 0, P, 1 << 30, N) == INVALID
    assert L.swiglu_mlp_fwd_nograd(P, P, P, P, P, 4, 64, 128, 0, P, 256, N) == WSERR
    assert L.swiglu_mlp_bwd(P, P, P, P, P, P, P, N, 4, 64, 128, 0, P, BIG, N) == INVALID
    assert L.swiglu_mlp_bwd(P, P, P, P, P, P, P, P_MIS, 4, 64, 128, 0, P, BIG, N) == ALIGN
    # the workspace must hold at least the error word and the shared-tile
    # counters; the recommended size adds the stream-K partial tiles
    need = L.swiglu_mlp_workspace_bytes(128, 64, 128, 0, 0)
    least = L.swiglu_mlp_workspace_min_bytes(128, 64, 128, 0, 0)
    assert need >= least > 256
    assert _fwd(L, wsb=least - 1) == WSERR
    assert L.swiglu_mlp_fwd_nograd(P, P, P, P, P, 4, 64, 128, 0, P,
                                   L.swiglu_mlp_workspace_min_bytes(4, 64, 128, 0, 1) - 1,
                                   N) == WSERR


def test_empty_batch_is_ok_without_launch(L):
    assert _fwd(L, M=0) == OK
    assert L.swiglu_mlp_fwd_nograd(P, P, P, P, P, 0, 64, 128, 0, P, BIG, N) == OK
    assert L.swiglu_mlp_bwd(P, P, P, P, P, P, P, P, 0, 64, 128, 1, P, BIG, N) == OK
    assert L.swiglu_mlp_last_launch_count() == 0


def test_wait_limit_setter(L):
    old = api.swiglu_mlp_set_wait_limit_ns(5)
    assert api.swiglu_mlp_set_wait_limit_ns(old) == 1000  # clamped to 1 us


def test_graph_entry_points_check_arguments_first(L):
    h = ctypes.c_void_p(0)
    cg = L.swiglu_mlp_graph_create_fwd_nograd
    assert cg(P, P, P, P, P, 4, 64, 128, 0, P, BIG, None) == INVALID
    assert cg(N, P, P, P, P, 4, 64, 128, 0, P, BIG, ctypes.byref(h)) == INVALID
    assert cg(P, P, P, P, P, 4, 60, 128, 0, P, BIG, ctypes.byref(h)) == ALIGN
    assert cg(P, P, P, P, P_MIS, 4, 64, 128, 0, P, BIG, ctypes.byref(h)) == ALIGN
    assert cg(P, P, P, P, P, 4, 64, 128, 0, P, 8, ctypes.byref(h)) == WSERR
    assert cg(P, P, P, P, P, 4, 64, 128, 7, P, BIG, ctypes.byref(h)) == INVALID
    assert h.value is None  # nothing was created
    assert L.swiglu_mlp_graph_launch(N, N) == INVALID
    assert L.swiglu_mlp_graph_destroy(N) == INVALID


def test_options_are_checked_before_any_launch(L):
    good = api.Options(1.5, 0.5, 0)
    nan = api.Options(float("nan"), 1.0, 0)
    inf = api.Options(1.0, float("inf"), 0)
    acc = api.Options(1.0, 1.0, 1)
    two = api.Options(1.0, 1.0, 2)
    fx = L.swiglu_mlp_fwd_ex
    ngx = L.swiglu_mlp_fwd_nograd_ex
    bx = L.swiglu_mlp_bwd_ex
    for o in (nan, inf):
        assert fx(P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(o), P, BIG, N) == INVALID
        assert ngx(P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(o), P, BIG, N) == INVALID
        assert bx(P, P, P, P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(o), P, BIG, N) == INVALID
    # accumulation is a backward option
    assert fx(P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(acc), P, BIG, N) == INVALID
    assert ngx(P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(acc), P, BIG, N) == INVALID
    assert bx(P, P, P, P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(two), P, BIG, N) == INVALID
    # valid options still meet the ordinary argument checks, and M = 0 launches nothing
    assert fx(P, P, P, P, P, 4, 60, 128, 0, ctypes.byref(good), P, BIG, N) == ALIGN
    assert bx(N, P, P, P, P, P, P, P, 4, 64, 128, 0, ctypes.byref(acc), P, BIG, N) == INVALID
    assert bx(P, P, P, P, P, P, P, P, 0, 64, 128, 0, ctypes.byref(acc), P, BIG, N) == OK
    assert fx(P, P, P, P, P, 0, 64, 128, 0, N, P, BIG, N) == OK
