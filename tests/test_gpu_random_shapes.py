"""Seeded random shapes through every path against the fp64 oracle: ragged
token counts, D and H any multiple of 8 (down to 8), bf16 and fp16, random
gate/down multipliers, SM pairs or single SMs, and for few tokens both forms
of the no-grad forward."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu

ODT = {"bf16": oracle.BF16, "f16": oracle.F16}
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.choice([1, 2, 7, 16, 33, 64, 65, 127, 129, 200, 257, 383, 600]))
        D = int(rng.integers(1, 97)) * 8
        H = int(rng.integers(1, 97)) * 8
        dtn = "bf16" if i % 2 == 0 else "f16"
        gm, dm = (1.0, 1.0) if i % 3 == 0 else (float(rng.uniform(0.5, 2.0)),
                                                float(rng.uniform(0.5, 2.0)))
        out.append((M, D, H, dtn, gm, dm, int(rng.integers(0, 3))))
    return out


def f64(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("case", _shapes(24, 1234), ids=lambda c: "M%d_D%d_H%d_%s" % c[:4])
def test_random_shape_training_parity(case):
    M, D, H, dtn, gm, dm, pairs_mode = case
    old = api.swiglu_mlp_set_cta_pairs(pairs_mode)
    try:
        t = synthetic.make_inputs(M, D, H, dtn, seed=M + D + H, device="cuda")
        Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], gate_mul=gm, down_mul=dm)
        fs = saved.clone()
        dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved,
                                           gate_mul=gm, down_mul=dm)
        torch.cuda.synchronize()
    finally:
        api.swiglu_mlp_set_cta_pairs(old)
    c = {k: v.cpu() for k, v in t.items()}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn], gate_mul=gm,
                       down_mul=dm)
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f, dt=ODT[dtn],
                        gate_mul=gm, down_mul=dm)
    got = {"Y": f64(Y), "G": f64(fs[:, :H]), "U": f64(fs[:, H:2 * H]), "A": f64(fs[:, 2 * H:]),
           "dG": f64(saved[:, :H]), "dU": f64(saved[:, H:2 * H]), "dX": f64(dX),
           "dWg": f64(dWgu[:H]), "dWu": f64(dWgu[H:]), "dWd": f64(dWd)}
    ref = {**f, **b}
    for k, v in got.items():
        assert np.all(np.isfinite(v)), k
        e = oracle.rel_frob(v, ref[k])
        assert e <= TOL, (k, e)


@pytest.mark.parametrize("case", [c for c in _shapes(40, 99) if c[0] <= 64][:12],
                         ids=lambda c: "M%d_D%d_H%d_%s" % c[:4])
def test_random_shape_nograd_parity(case):
    M, D, H, dtn, gm, dm, mode = case
    t = synthetic.make_inputs(M, D, H, dtn, seed=M * D + H, device="cuda")
    outs = []
    for fused in (0, 2):
        old = api.swiglu_mlp_set_nograd_fused(fused)
        try:
            outs.append(api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"], gate_mul=gm,
                                                  down_mul=dm))
        finally:
            api.swiglu_mlp_set_nograd_fused(old)
    torch.cuda.synchronize()
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn], gate_mul=gm,
                       down_mul=dm)
    for Y, A in outs:
        assert oracle.rel_frob(f64(Y), r["Y"]) <= TOL
        assert oracle.rel_frob(f64(A), r["A"]) <= TOL
