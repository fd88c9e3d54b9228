"""bench.py's GPU-side legs on small shapes: the training timer, the
end-to-end leg (host-fed steps through the C ABI, copies on a second stream)
and the parity that the CPU-baseline leg reports."""
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def test_e2e_leg_counts_its_copies_and_matches_the_device_step():
    import bench
    w = {"B": 2, "S": 128, "D": 256, "H": 512}
    M, D, H = 256, 256, 512
    sec, launches, _, (t, o), med = bench._time_training(api, w, "bf16", 2, 3, 0, "cuda:0")
    assert sec > 0 and med > 0 and launches == 2 * 6  # two steps of six GEMMs
    Y_dev, dX_dev = o["Y"].clone(), o["dX"].clone()
    e2e_sec, h2d, d2h, idle = bench._e2e(api, t, o, 3)
    assert e2e_sec > 0 and idle["h2d"] > 0 and idle["d2h"] > 0
    assert h2d == 2 * M * D * 2                       # X and dY in
    assert d2h == (2 * H * D + D * H) * 2             # dWgu, dWd out
    # the e2e steps recompute the same step from the same inputs (slot 0 is the
    # device step's own buffers): same results, bit for bit
    torch.cuda.synchronize()
    assert torch.equal(o["Y"], Y_dev) and torch.equal(o["dX"], dX_dev)


def test_cpu_baseline_parity_is_small():
    import bench
    t = synthetic.make_inputs(16, 256, 512, "bf16", seed=3, device="cuda", kind="device")
    c = {k: t[k].cpu() for k in ("X", "dY", "Wg", "Wu", "Wd")}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"])
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f)
    p = bench._sample_parity(t, f, b)
    for k in ("Y", "dX", "dWg", "dWu", "dWd"):
        assert 0 <= p[k] <= 1e-2, (k, p[k])
