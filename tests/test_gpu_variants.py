"""The gate/down multiplier variant and weight-gradient accumulation
(swiglu_mlp_*_ex) on every path, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic
from backward_tcgen05_tma_gb300.module import SwiGLUMLP

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5}
ODT = {"bf16": oracle.BF16, "f16": oracle.F16, "f32": oracle.F32}
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
MG, MD = 1.7, 0.6


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


@pytest.fixture(params=[2, 0], ids=["sm_pairs", "single_sm"])
def cta_pairs(request):
    old = api.swiglu_mlp_set_cta_pairs(request.param)
    yield request.param
    api.swiglu_mlp_set_cta_pairs(old)


def f64(t):
    return t.detach().cpu().double().numpy()


def run(t, gm, md, acc=None):
    """fwd_ex + bwd_ex; ``acc``: held dWgu, dWd to accumulate into."""
    H = t["Wg"].shape[0]
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], gate_mul=gm, down_mul=md)
    fwd = saved.clone()
    out = {} if acc is None else {"dWgu": acc["dWgu"].clone(), "dWd": acc["dWd"].clone()}
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved, out=out,
                                       gate_mul=gm, down_mul=md, accumulate=acc is not None)
    torch.cuda.synchronize()
    return {"Y": f64(Y), "G": f64(fwd[:, :H]), "U": f64(fwd[:, H:2 * H]),
            "A": f64(fwd[:, 2 * H:]), "dG": f64(saved[:, :H]), "dU": f64(saved[:, H:2 * H]),
            "dX": f64(dX), "dWg": f64(dWgu[:H]), "dWu": f64(dWgu[H:]), "dWd": f64(dWd)}


def reference(t, dtn, gm, md, acc=None):
    c = {k: v.cpu() for k, v in t.items()}
    H = c["Wg"].shape[0]
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn], gate_mul=gm, down_mul=md)
    held = None
    if acc is not None:
        held = {"dWg": f64(acc["dWgu"][:H]), "dWu": f64(acc["dWgu"][H:]),
                "dWd": f64(acc["dWd"])}
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f, dt=ODT[dtn],
                        gate_mul=gm, down_mul=md, accumulate=held)
    return {**f, **b}


def check(g, r, dtn):
    for k in ("Y", "A", "G", "U", "dG", "dU", "dX", "dWg", "dWu", "dWd"):
        e = oracle.rel_frob(g[k], r[k])
        assert e <= TOL[dtn], (k, e)


@pytest.mark.parametrize("dtn", ["bf16", "f16"])
def test_multipliers_parity(dtn, cta_pairs):
    t = synthetic.make_inputs(333, 320, 392, dtn, seed=61, device="cuda")
    check(run(t, MG, MD), reference(t, dtn, MG, MD), dtn)


def test_multipliers_parity_fp32_ieee():
    t = synthetic.make_inputs(32, 64, 176, "f32", seed=62, device="cuda")
    check(run(t, MG, MD), reference(t, "f32", MG, MD), "f32")


@pytest.mark.parametrize("mode", [0, 2], ids=["two_kernels", "fused"])
@pytest.mark.parametrize("M", [1, 16, 48, 300])
def test_multipliers_nograd_parity(M, mode):
    D, H = 320, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=63 + M, device="cuda")
    old = api.swiglu_mlp_set_nograd_fused(mode)
    try:
        Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"], gate_mul=MG, down_mul=MD)
        torch.cuda.synchronize()
    finally:
        api.swiglu_mlp_set_nograd_fused(old)
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], gate_mul=MG, down_mul=MD)
    assert oracle.rel_frob(f64(Y), r["Y"]) <= TOL["bf16"]
    assert oracle.rel_frob(f64(A), r["A"]) <= TOL["bf16"]


def test_power_of_two_multipliers_equal_scaled_weights_bitwise():
    """mg = 2, md = 1/2 scale the fp32 accumulators exactly, so the variant
    agrees bit for bit with the standard MLP on Wg doubled and Wd halved
    (with dWg doubled and dWd halved), as the oracle's exact identity says."""
    t = synthetic.make_inputs(300, 256, 392, "bf16", seed=64, device="cuda")
    g = run(t, 2.0, 0.5)
    H = 392
    s = dict(t)
    s["Wg"] = t["Wg"] * 2
    s["Wd"] = t["Wd"] * 0.5
    s["Wgu"] = torch.cat([s["Wg"], t["Wu"]]).contiguous()
    r = run(s, 1.0, 1.0)
    for k in ("Y", "G", "U", "A", "dU", "dX", "dWu"):
        np.testing.assert_array_equal(g[k], r[k])
    np.testing.assert_array_equal(g["dG"], 2 * r["dG"])
    np.testing.assert_array_equal(g["dWg"], 2 * r["dWg"])
    np.testing.assert_array_equal(g["dWd"], 0.5 * r["dWd"])
    assert H == t["Wg"].shape[0]


def test_default_options_equal_base_call_bitwise():
    t = synthetic.make_inputs(200, 256, 392, "bf16", seed=65, device="cuda")
    a = run(t, 1.0, 1.0)
    H = 392
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])  # NULL options
    opts = api.Options(1.0, 1.0, 0)
    L = api.lib()
    Y2 = torch.empty_like(Y)
    saved2 = torch.empty_like(saved)
    ws = api.workspace(200, 256, H, torch.bfloat16, api.SWIGLU_OP_FWD, "cuda")
    import ctypes
    rc = L.swiglu_mlp_fwd_ex(ctypes.c_void_p(t["X"].data_ptr()), ctypes.c_void_p(t["Wgu"].data_ptr()),
                             ctypes.c_void_p(t["Wd"].data_ptr()), ctypes.c_void_p(Y2.data_ptr()),
                             ctypes.c_void_p(saved2.data_ptr()), 200, 256, H, 0,
                             ctypes.byref(opts), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(saved, saved2)
    np.testing.assert_array_equal(a["Y"], f64(Y))


@pytest.mark.parametrize("dtn", ["bf16", "f16", "f32"])
def test_accumulate_parity(dtn, cta_pairs):
    M, D, H = (333, 320, 392) if dtn != "f32" else (32, 64, 176)
    t = synthetic.make_inputs(M, D, H, dtn, seed=66, device="cuda")
    acc = {"dWgu": (torch.randn(2 * H, D, device="cuda") * 0.05).to(TDT[dtn]),
           "dWd": (torch.randn(D, H, device="cuda") * 0.05).to(TDT[dtn])}
    check(run(t, MG, MD, acc), reference(t, dtn, MG, MD, acc), dtn)


def test_accumulated_micro_batches_match_one_batch():
    """Two micro-batches, the second accumulated onto the first's weight
    gradients, against the oracle's gradients of the concatenated batch."""
    M, D, H = 512, 256, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=67, device="cuda")
    acc = None
    for rows in (slice(0, 200), slice(200, M)):
        part = dict(t)
        part["X"] = t["X"][rows].contiguous()
        part["dY"] = t["dY"][rows].contiguous()
        Y, saved = api.swiglu_mlp_fwd(part["X"], t["Wgu"], t["Wd"])
        out = {} if acc is None else {"dWgu": acc[0], "dWd": acc[1]}
        _, dWgu, dWd = api.swiglu_mlp_bwd(part["dY"], part["X"], t["Wgu"], t["Wd"], saved,
                                          out=out, accumulate=acc is not None)
        acc = (dWgu, dWd)
    torch.cuda.synchronize()
    r = reference(t, "bf16", 1.0, 1.0)
    assert oracle.rel_frob(f64(acc[0][:H]), r["dWg"]) <= TOL["bf16"]
    assert oracle.rel_frob(f64(acc[0][H:]), r["dWu"]) <= TOL["bf16"]
    assert oracle.rel_frob(f64(acc[1]), r["dWd"]) <= TOL["bf16"]


def test_module_with_multipliers_matches_oracle():
    B, S, D, H = 2, 64, 256, 392
    t = synthetic.make_inputs(B * S, D, H, "bf16", seed=68, device="cuda")
    m = SwiGLUMLP.from_weights(t["Wg"], t["Wu"], t["Wd"], gate_multiplier=MG,
                               down_multiplier=MD)
    x = t["X"].reshape(B, S, D).clone().requires_grad_(True)
    y = m(x)
    y.backward(t["dY"].reshape(B, S, D))
    torch.cuda.synchronize()
    r = reference(t, "bf16", MG, MD)
    got = {"Y": f64(y.reshape(B * S, D)), "dX": f64(x.grad.reshape(B * S, D)),
           "dWg": f64(m.gate_up_weight.grad[:H]), "dWu": f64(m.gate_up_weight.grad[H:]),
           "dWd": f64(m.down_weight.grad)}
    for k, v in got.items():
        assert oracle.rel_frob(v, r[k]) <= TOL["bf16"], k
    with torch.no_grad():
        yn = m(t["X"])
    assert oracle.rel_frob(f64(yn), r["Y"]) <= TOL["bf16"]
