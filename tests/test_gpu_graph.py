"""The CUDA-graph no-grad forward: replays equal direct calls bitwise, pick
up new tokens written into the captured input, and match the oracle."""
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
ODT = {"bf16": oracle.BF16, "f16": oracle.F16, "f32": oracle.F32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


@pytest.mark.parametrize("dtn,M,D,H,fused", [("bf16", 1, 4096, 11008, 0),
                                             ("bf16", 16, 4096, 11008, 0),
                                             ("f16", 33, 1024, 2816, 0), ("f16", 33, 1024, 2816, 2),
                                             ("bf16", 64, 2048, 5632, 0),
                                             ("bf16", 64, 2048, 5632, 2),
                                             ("bf16", 300, 512, 392, 0), ("f32", 32, 64, 176, 0)])
def test_graph_replay_equals_direct_call(dtn, M, D, H, fused):
    """Replays equal direct calls bit for bit, for both few-token forms."""
    t = synthetic.make_inputs(M, D, H, dtn, seed=31, device="cuda", kind="device")
    old = api.swiglu_mlp_set_nograd_fused(fused)
    try:
        g = api.FwdNogradGraph(t["Wgu"], t["Wd"], M)
        for step in range(3):
            x = torch.randn(M, D, device="cuda").to(TDT[dtn])
            y = g(x).clone()
            n_graph = api.swiglu_mlp_last_launch_count()
            Yd, Ad = api.swiglu_mlp_fwd_nograd(x, t["Wgu"], t["Wd"])
            n_direct = api.swiglu_mlp_last_launch_count()
            torch.cuda.synchronize()
            assert torch.equal(y, Yd), step
            assert torch.equal(g.A, Ad), step
            assert n_graph == n_direct >= 1
        g.close()
    finally:
        api.swiglu_mlp_set_nograd_fused(old)


def test_graph_matches_oracle():
    M, D, H = 16, 1024, 2816
    t = synthetic.make_inputs(M, D, H, "bf16", seed=32, device="cuda")
    g = api.FwdNogradGraph(t["Wgu"], t["Wd"], M)
    y = g(t["X"])
    torch.cuda.synchronize()
    c = {k: v.cpu() for k, v in t.items()}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT["bf16"])
    assert oracle.rel_frob(y.double().cpu().numpy(), f["Y"]) <= 1e-2
    assert oracle.rel_frob(g.A.double().cpu().numpy(), f["A"]) <= 1e-2


def test_graph_in_place_input_and_many_replays():
    """A decode loop writes tokens straight into the captured X buffer."""
    M, D, H = 4, 2048, 5632
    t = synthetic.make_inputs(M, D, H, "bf16", seed=33, device="cuda", kind="device")
    g = api.FwdNogradGraph(t["Wgu"], t["Wd"], M)
    outs, xs = [], []
    for _ in range(20):
        g.X.copy_(torch.randn(M, D, device="cuda").bfloat16())
        xs.append(g.X.clone())
        outs.append(g().clone())
    torch.cuda.synchronize()
    for x, y in zip(xs, outs):
        Yd, _ = api.swiglu_mlp_fwd_nograd(x, t["Wgu"], t["Wd"])
        assert torch.equal(y, Yd)
    assert api.swiglu_mlp_query_error(g.ws) == 0


def test_empty_graph_and_profiling_refusal():
    t = synthetic.make_inputs(8, 64, 176, "bf16", seed=34, device="cuda", kind="device")
    g = api.FwdNogradGraph(t["Wgu"], t["Wd"], 0)
    g()
    assert api.swiglu_mlp_last_launch_count() == 0
    g.close()
    api.swiglu_mlp_profile_enable(True)
    try:
        with pytest.raises(api.SwigluError) as e:
            api.FwdNogradGraph(t["Wgu"], t["Wd"], 8)
        assert e.value.code == 3
    finally:
        api.swiglu_mlp_profile_enable(False)
        api.swiglu_mlp_profile_read()
