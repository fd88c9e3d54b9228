"""The debug build (libswiglu_mlp_debug.so: the same sources compiled with
-DSWIGLU_DEBUG) on the GPU, through the C ABI.

In the debug build every plain (non-TMA) global load and store of every
kernel is checked against the buffers that launch was given (the caller's
tensors and the workspace, with their sizes), and table indices (partial
slots, tile counters, the few-token queue and ready mask) against their
bounds; a failed check skips the access and records SWIGLU_ERR_DEVICE_BOUNDS
in the workspace error word.  It stands in for a memory checker: these tests
drive every path of the library through it -- training forward + backward on
SM pairs and on single SMs, stream-K splits, both forms of the dG/dU
epilogue, the multiplier and accumulation options, a minimal workspace, the
few-token no-grad kernels (fused and two-kernel), the no-allocation entry
point, the fp32 path -- and require that no check fails and that every output
is bitwise the release build's (the arithmetic is the same code).  A test
hook then halves one launch's output window to show that the checks fire:
the call reports SWIGLU_ERR_DEVICE_BOUNDS, while no access leaves the
caller's buffers."""
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu

OK, BOUNDS = 0, 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    prev = api.use_debug_library(True)
    assert api.lib().swiglu_mlp_debug_build() == 1
    api.use_debug_library(prev)


def with_library(debug, fn, pairs=1, fused=1):
    """fn() under the release or the debug build, with the SM-pair and
    few-token modes set in that library for the call."""
    prev = api.use_debug_library(debug)
    old_p = api.swiglu_mlp_set_cta_pairs(pairs)
    old_f = api.swiglu_mlp_set_nograd_fused(fused)
    try:
        return fn()
    finally:
        api.swiglu_mlp_set_cta_pairs(old_p)
        api.swiglu_mlp_set_nograd_fused(old_f)
        api.use_debug_library(prev)


def same_in_both(fn, **modes):
    """Runs fn in both builds; every status OK, every output bitwise equal."""
    st_r, out_r = with_library(False, fn, **modes)
    st_d, out_d = with_library(True, fn, **modes)
    assert st_r == [OK] * len(st_r)
    assert st_d == [OK] * len(st_d), [api.STATUS.get(s, s) for s in st_d]
    for k in out_r:
        assert torch.equal(out_r[k], out_d[k]), k
    return out_d


def training(t, gm=1.0, md=1.0, accumulate=False, minimal=False):
    def fn():
        X, Wgu, Wd = t["X"], t["Wgu"], t["Wd"]
        M, D = X.shape
        H = Wd.shape[1]
        wsf = api.workspace(M, D, H, X.dtype, api.SWIGLU_OP_FWD, X.device, minimal=minimal)
        wsb = api.workspace(M, D, H, X.dtype, api.SWIGLU_OP_BWD, X.device, minimal=minimal)
        Y, saved = api.swiglu_mlp_fwd(X, Wgu, Wd, ws=wsf, gate_mul=gm, down_mul=md)
        st = [api.swiglu_mlp_query_error(wsf)]
        fwd = saved.clone()
        out = {}
        if accumulate:
            g = torch.Generator(device="cpu").manual_seed(5)
            out = {"dWgu": (0.01 * torch.randn(2 * H, D, generator=g)).to(X.device, X.dtype),
                   "dWd": (0.01 * torch.randn(D, H, generator=g)).to(X.device, X.dtype)}
        dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], X, Wgu, Wd, saved, out=out, ws=wsb,
                                           gate_mul=gm, down_mul=md, accumulate=accumulate)
        st.append(api.swiglu_mlp_query_error(wsb))
        return st, {"Y": Y.cpu(), "fwd": fwd.cpu(), "dGU": saved[:, :2 * H].cpu(),
                    "dX": dX.cpu(), "dWgu": dWgu.cpu(), "dWd": dWd.cpu()}
    return fn


def nograd(t, noalloc=False):
    def fn():
        X, Wgu, Wd = t["X"], t["Wgu"], t["Wd"]
        M, D = X.shape
        H = Wd.shape[1]
        if noalloc:
            Y, A = api.swiglu_mlp_fwd_nograd_noalloc(X, Wgu, Wd)
            torch.cuda.synchronize()
            return [OK], {"Y": Y.cpu(), "A": A.cpu()}
        ws = api.workspace(M, D, H, X.dtype, api.SWIGLU_OP_FWD_NOGRAD, X.device)
        Y, A = api.swiglu_mlp_fwd_nograd(X, Wgu, Wd, ws=ws)
        return [api.swiglu_mlp_query_error(ws)], {"Y": Y.cpu(), "A": A.cpu()}
    return fn


@pytest.mark.parametrize("pairs", [2, 0], ids=["sm_pairs", "single_sm"])
@pytest.mark.parametrize("M,D,H", [(333, 320, 392),     # ragged in every dimension
                                   (2125, 1024, 2816),  # stream-K in every GEMM, direct dG/dU loads
                                   (384, 2304, 512)])   # staged dG/dU loads (D > 2048)
def test_training_paths_pass_every_check_bitwise(M, D, H, pairs):
    t = synthetic.make_inputs(M, D, H, "bf16", seed=M, device="cuda", kind="device")
    same_in_both(training(t), pairs=pairs)


def test_options_fp16_and_minimal_workspace_pass_every_check():
    t = synthetic.make_inputs(333, 320, 392, "f16", seed=3, device="cuda", kind="device")
    same_in_both(training(t, gm=1.7, md=0.6, accumulate=True), pairs=2)
    t = synthetic.make_inputs(2125, 1024, 2816, "bf16", seed=4, device="cuda", kind="device")
    same_in_both(training(t, minimal=True), pairs=1)


@pytest.mark.parametrize("fused", [2, 0], ids=["fused", "two_kernels"])
@pytest.mark.parametrize("M", [1, 17, 40, 64, 100])
def test_nograd_paths_pass_every_check_bitwise(M, fused):
    if M > 64 and fused == 0:
        pytest.skip("more than 64 tokens run the tensor-core path in either mode")
    t = synthetic.make_inputs(M, 1024, 2816, "bf16", seed=M, device="cuda", kind="device")
    same_in_both(nograd(t), fused=fused)


def test_noalloc_and_fp32_paths_pass_every_check_bitwise():
    t = synthetic.make_inputs(16, 1024, 2816, "bf16", seed=6, device="cuda", kind="device")
    same_in_both(nograd(t, noalloc=True))
    t = synthetic.make_inputs(32, 64, 176, "f32", seed=0, device="cuda")
    same_in_both(training(t))
    same_in_both(nograd(t))


def test_debug_build_matches_the_oracle():
    # bitwise equal to the release build above; pinned to the oracle here too
    M, D, H = 333, 320, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=11, device="cuda", kind="device")
    _, out = with_library(True, training(t))
    c = {k: v.cpu() for k, v in t.items()}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"])
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f)
    for got, ref in [(out["Y"], f["Y"]), (out["fwd"][:, 2 * H:], f["A"]), (out["dX"], b["dX"]),
                     (out["dWgu"][:H], b["dWg"]), (out["dWgu"][H:], b["dWu"]),
                     (out["dWd"], b["dWd"])]:
        assert oracle.rel_frob(got.double().numpy(), ref) <= 1e-2


def narrowed_status(debug, call):
    """Status of call() (which returns its workspace) with the next launch's
    output window halved by the test hook."""
    prev = api.use_debug_library(debug)
    try:
        api.lib().swiglu_mlp_debug_narrow_once(1)
        try:
            st = api.swiglu_mlp_query_error(call())
        except api.SwigluError as e:  # with the debug build the binding checks each call
            st = e.code
        api.lib().swiglu_mlp_debug_narrow_once(0)
        return st
    finally:
        api.use_debug_library(prev)


@pytest.mark.parametrize("path", ["training", "fused_nograd", "two_kernel_nograd", "fp32"])
def test_a_narrowed_window_is_reported_not_accessed(path):
    dtn = "f32" if path == "fp32" else "bf16"
    M, D, H = {"training": (333, 320, 392), "fp32": (32, 64, 176)}.get(path, (40, 1024, 2816))
    t = synthetic.make_inputs(M, D, H, dtn, seed=2, device="cuda")

    def call():
        if path in ("training", "fp32"):
            ws = api.workspace(M, D, H, t["X"].dtype, api.SWIGLU_OP_FWD, t["X"].device)
            api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], ws=ws)
        else:
            old = api.swiglu_mlp_set_nograd_fused(2 if path == "fused_nograd" else 0)
            try:
                ws = api.workspace(M, D, H, t["X"].dtype, api.SWIGLU_OP_FWD_NOGRAD, t["X"].device)
                api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"], ws=ws)
            finally:
                api.swiglu_mlp_set_nograd_fused(old)
        return ws

    assert narrowed_status(True, call) == BOUNDS
    assert narrowed_status(False, call) == OK  # the hook has no effect on the release build
    # the next call of the debug build is clean again
    same_in_both(training(t) if path in ("training", "fp32") else nograd(t))
