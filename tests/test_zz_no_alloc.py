"""The no-allocation no-grad forward (swiglu_mlp_fwd_nograd_noalloc).

Some callers cannot allocate device memory -- code running under CUDA-graph
capture, plug-ins whose host framework owns all device memory, decode loops
that must not call cudaMalloc -- so this entry point takes no workspace and
keeps its scratch in a static device array inside the library.  This file
checks, through the C ABI, that two calls in a row give bit for bit the
outputs of the workspace entry point (they run the same kernels), with the
array left dirty by a call on other inputs before them, and that shapes
beyond the array's limit are refused without a launch.  It is collected last
so that a failure here never hides the other tests' results."""
import ctypes

import pytest
import torch

from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-2  # relative Frobenius tolerance of the bf16/fp16 parity tests


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def _rel(got, ref):
    g, r = got.double(), ref.double()
    return float((g - r).norm() / r.norm().clamp_min(1e-30))


def _noalloc(L, t, M, D, H, dt):
    # outputs start as NaN: every element must be written by the call
    Y = torch.full((M, D), float("nan"), dtype=t["X"].dtype, device="cuda")
    A = torch.full((M, H), float("nan"), dtype=t["X"].dtype, device="cuda")
    rc = L.swiglu_mlp_fwd_nograd_noalloc(
        ctypes.c_void_p(t["X"].data_ptr()), ctypes.c_void_p(t["Wgu"].data_ptr()),
        ctypes.c_void_p(t["Wd"].data_ptr()), ctypes.c_void_p(Y.data_ptr()),
        ctypes.c_void_p(A.data_ptr()), M, D, H, dt,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, Y, A


@pytest.mark.parametrize("dtn,M,D,H", [("bf16", 1, 4096, 11008), ("bf16", 16, 4096, 11008),
                                       ("bf16", 32, 4096, 11008), ("f16", 5, 320, 392),
                                       ("bf16", 32, 512, 1024), ("bf16", 40, 4096, 11008),
                                       ("bf16", 64, 4096, 11008)])
def test_noalloc_matches_workspace_entry_point(L, dtn, M, D, H):
    # the default few-token form (two kernels) at 1 to 64 tokens
    dt = {"bf16": 0, "f16": 1}[dtn]
    t = synthetic.make_inputs(M, D, H, dtn, seed=M, device="cuda", kind="device")
    Y_ref, A_ref = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    # a call on other inputs first leaves its partial sums, counters and ready
    # bits in the array; the calls checked below must not see any of them
    other = synthetic.make_inputs(M, D, H, dtn, seed=M + 1000, device="cuda", kind="device")
    rc, Y_o, _ = _noalloc(L, other, M, D, H, dt)
    assert rc == 0, api.status_string(rc)
    for _ in range(2):  # the array keeps the previous call's contents
        rc, Y, A = _noalloc(L, t, M, D, H, dt)
        assert rc == 0, api.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_ref) and torch.equal(A, A_ref)
    assert not torch.equal(Y_o, Y_ref)
    assert _rel(Y, Y_ref) <= TOL


def test_noalloc_rejects_sizes_beyond_its_range(L):
    t = synthetic.make_inputs(65, 64, 128, "bf16", seed=1, device="cuda")
    rc, _, _ = _noalloc(L, t, 65, 64, 128, 0)      # more tokens than the path serves
    assert rc == 3 and L.swiglu_mlp_last_launch_count() == 0
