"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances (relative Frobenius error against the oracle's one-round program):
1e-2 for bf16/fp16, 1e-5 for the fp32 IEEE mode; the elementwise SwiGLU stage
(G, U, A, dG, dU) within 1 unit in the last place of the storage type."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic
from tests.conftest import device_status

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5}
ODT = {"bf16": oracle.BF16, "f16": oracle.F16, "f32": oracle.F32}
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
MANT = {"bf16": 8, "f16": 11, "f32": 24}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def f64(t):
    return t.detach().float().cpu().double().numpy() if t.dtype != torch.float32 else \
        t.detach().cpu().double().numpy()


def ulp(ref, dtn):
    """Spacing of the storage type at |ref| (normal range; subnormal floor)."""
    p = MANT[dtn]
    emin = -14 if dtn == "f16" else -126
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (p - 1)).astype(int))


def run_gpu(t, dtn):
    """fwd + bwd through the C ABI; returns host fp64 copies of everything."""
    H = t["Wg"].shape[0]
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    fwd_saved = saved.clone()
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved)
    torch.cuda.synchronize()
    return {"Y": f64(Y), "G": f64(fwd_saved[:, :H]), "U": f64(fwd_saved[:, H:2 * H]),
            "A": f64(fwd_saved[:, 2 * H:]), "dG": f64(saved[:, :H]), "dU": f64(saved[:, H:2 * H]),
            "dX": f64(dX), "dWg": f64(dWgu[:H]), "dWu": f64(dWgu[H:]), "dWd": f64(dWd)}


def run_oracle(t, dtn):
    c = {k: v.cpu() for k, v in t.items()}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn])
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f, dt=ODT[dtn])
    return {**f, **b}


def within_ulp_frac(got, ref, dtn):
    """Fraction of elements within one unit in the last place of the oracle."""
    return float(np.mean(np.abs(got - ref) <= ulp(ref, dtn)))


def check_all(g, r, dtn, ulp_keys=("G", "U", "A", "dG", "dU")):
    """Relative Frobenius error of every output, and for the elementwise
    stage on random data: at least 99% of elements within one ulp.  (Where a
    sum cancels to near zero, fp32 accumulation order alone moves the result
    by more than an ulp of the small value; the strict one-ulp pin uses
    exact-accumulation inputs instead.)"""
    for k in ("Y", "A", "G", "U", "dG", "dU", "dX", "dWg", "dWu", "dWd"):
        e = oracle.rel_frob(g[k], r[k])
        assert e <= TOL[dtn], (k, e)
    for k in ulp_keys:
        f = within_ulp_frac(g[k], r[k], dtn)
        assert f >= 0.99, (k, f)


def test_tiny_fp32_ieee_parity():
    # B=2, S=16, D=64, H=176; X, dY ~ N(0,1); Wg, Wu ~ N(0,1/64); Wd ~ N(0,1/176); seed 0
    t = synthetic.make_inputs(32, 64, 176, "f32", seed=0, device="cuda")
    g = run_gpu(t, "f32")
    r = run_oracle(t, "f32")
    check_all(g, r, "f32", ulp_keys=())
    for k in ("G", "U", "A", "dG", "dU"):
        assert oracle.rel_frob(g[k], r[k]) <= 1e-6, k


@pytest.fixture(params=[2, 0], ids=["sm_pairs", "single_sm"])
def cta_pairs(request):
    """Runs a test with every tensor-core GEMM on SM pairs, then on single SMs."""
    old = api.swiglu_mlp_set_cta_pairs(request.param)
    yield request.param
    api.swiglu_mlp_set_cta_pairs(old)


@pytest.mark.parametrize("dtn", ["bf16", "f16"])
def test_ragged_multi_tile_parity(dtn, cta_pairs):
    # 3 row tiles (ragged), 4 gate/up column tiles (ragged), K=2H=784 (ragged k-blocks)
    t = synthetic.make_inputs(333, 320, 392, dtn, seed=3, device="cuda")
    check_all(run_gpu(t, dtn), run_oracle(t, dtn), dtn)


@pytest.mark.parametrize("M,D,H", [(1, 64, 176), (3, 64, 176), (127, 64, 176), (129, 64, 176),
                                   (64, 8, 8), (200, 1024, 64)])
def test_edge_shapes(M, D, H):
    t = synthetic.make_inputs(M, D, H, "bf16", seed=M, device="cuda")
    check_all(run_gpu(t, "bf16"), run_oracle(t, "bf16"), "bf16")


@pytest.mark.parametrize("dtn", ["bf16", "f16"])
def test_exact_accumulation_inputs_bitwise_gate_up(dtn, cta_pairs):
    """Dyadic-grid inputs make every fp32 partial sum exact, so the GPU's
    accumulators equal the oracle's exact sums: stored G, U must be bitwise
    equal, A and dG/dU within one unit in the last place."""
    t = synthetic.make_inputs(273, 512, 384, dtn, seed=11, device="cuda", kind="grid")
    g = run_gpu(t, dtn)
    r = run_oracle(t, dtn)
    np.testing.assert_array_equal(g["G"], r["G"])
    np.testing.assert_array_equal(g["U"], r["U"])
    for k in ("A", "dG", "dU"):
        d = np.abs(g[k] - r[k])
        assert np.all(d <= ulp(r[k], dtn)), (k, float(np.max(d / ulp(r[k], dtn))))
    frac_a = float(np.mean(g["A"] == r["A"]))
    assert frac_a > 0.97, frac_a


def test_one_round_program_not_two_round():
    t = synthetic.make_inputs(256, 1024, 256, "bf16", seed=0, device="cuda")
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    A = f64(saved[:, 512:])
    c = {k: v.cpu() for k, v in t.items()}
    one = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], mode=oracle.ONE_ROUND)
    two = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], mode=oracle.TWO_ROUND)
    d_one = float(np.mean(A != one["A"]))
    d_two = float(np.mean(A != two["A"]))
    assert d_one < 0.01, d_one
    assert d_two > 0.05, d_two


def test_nograd_equals_training_forward_bitwise():
    t = synthetic.make_inputs(300, 256, 392, "bf16", seed=5, device="cuda")
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    Yn, An = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    torch.cuda.synchronize()
    assert torch.equal(Yn, Y)
    assert torch.equal(An, saved[:, 2 * 392:])


def test_deterministic_bitwise():
    t = synthetic.make_inputs(384, 512, 640, "bf16", seed=6, device="cuda")
    a = run_gpu(t, "bf16")
    b = run_gpu(t, "bf16")
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_guard_bands_untouched():
    M, D, H = 257, 320, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=7, device="cuda")
    pad = 512
    bufs, views = {}, {}
    for k, shape in (("Y", (M, D)), ("saved", (M, 3 * H)), ("dX", (M, D)),
                     ("dWgu", (2 * H, D)), ("dWd", (D, H))):
        n = shape[0] * shape[1]
        b = torch.full((n + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
        bufs[k] = b
        views[k] = b[pad:pad + n].view(*shape)
    api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], out=views)
    api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], views["saved"], out=views)
    torch.cuda.synchronize()
    for k, b in bufs.items():
        assert torch.all(b[:pad] == 12345.0) and torch.all(b[-pad:] == 12345.0), k
        assert torch.all(torch.isfinite(views[k].float())), k


def test_grads_finite_and_nonzero():
    t = synthetic.make_inputs(512, 256, 384, "bf16", seed=8, device="cuda")
    g = run_gpu(t, "bf16")
    for k in ("dX", "dWg", "dWu", "dWd"):
        assert np.all(np.isfinite(g[k])), k
        assert np.any(g[k] != 0), k


def test_empty_batch():
    t = synthetic.make_inputs(1, 64, 128, "bf16", seed=0, device="cuda")
    X0 = t["X"][:0]
    Y, saved = api.swiglu_mlp_fwd(X0, t["Wgu"], t["Wd"])
    assert Y.shape == (0, 64) and api.swiglu_mlp_last_launch_count() == 0


def test_device_errors_are_statuses():
    t = synthetic.make_inputs(128, 64, 128, "bf16", seed=0, device="cuda")
    L = api.lib()
    Y = torch.empty(128, 64, dtype=torch.bfloat16, device="cuda")
    saved = torch.empty(128, 3 * 128, dtype=torch.bfloat16, device="cuda")
    ws = api.workspace(128, 64, 128, torch.bfloat16, 0, "cuda")
    p = lambda x: x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    mis = t["X"].data_ptr() + 2
    assert L.swiglu_mlp_fwd(mis, p(t["Wgu"]), p(t["Wd"]), p(Y), p(saved), 128, 64, 128, 0,
                            p(ws), ws.numel(), s) == 2
    assert L.swiglu_mlp_fwd(p(t["X"]), p(t["Wgu"]), p(t["Wd"]), p(Y), p(saved), 128, 64, 128, 0,
                            p(ws), 4, s) == 4
    assert L.swiglu_mlp_fwd(p(t["X"]), p(t["Wgu"]), p(t["Wd"]), p(Y), p(saved), 128, 64, 128, 0,
                            p(ws), ws.numel(), s) == 0
    assert api.swiglu_mlp_query_error(ws) == 0


def test_stalled_pipeline_times_out_cleanly(cta_pairs):
    """Failure detection without a fault: the producer skips one stage, the
    MMA warp's bounded wait runs out, the kernel records a timeout status and
    returns; the context stays usable and the next call is correct."""
    t = synthetic.make_inputs(256, 128, 256, "bf16", seed=9, device="cuda")
    ws = api.workspace(256, 128, 256, torch.bfloat16, 0, "cuda")
    old = api.swiglu_mlp_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        api.swiglu_mlp_inject_stall_once(True)
        assert device_status(lambda: api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], ws=ws), ws) == 6
    finally:
        api.swiglu_mlp_inject_stall_once(False)
        api.swiglu_mlp_set_wait_limit_ns(old)
    g = run_gpu(t, "bf16")
    ws2 = api.workspace(256, 128, 256, torch.bfloat16, 0, "cuda")
    api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], ws=ws2)
    assert api.swiglu_mlp_query_error(ws2) == 0
    check_all(g, run_oracle(t, "bf16"), "bf16")


def test_stalled_tma_dgu_kernel_times_out_cleanly():
    """The same failure, injected into the dG/dU kernel of a backward call (its
    second launch) on SM pairs with D <= 2048, where the epilogue streams G/U
    through TMA slots: the kernel unwinds, reports the timeout, and the next
    backward on fresh buffers is correct."""
    M, D, H = 512, 256, 512
    t = synthetic.make_inputs(M, D, H, "bf16", seed=12, device="cuda")
    old_p = api.swiglu_mlp_set_cta_pairs(2)
    old = api.swiglu_mlp_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        _, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
        ws = api.workspace(M, D, H, torch.bfloat16, 2, "cuda")
        api.swiglu_mlp_inject_stall_once(2)  # dWd, then dG/dU
        assert device_status(
            lambda: api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved, ws=ws), ws) == 6
    finally:
        api.swiglu_mlp_inject_stall_once(False)
        api.swiglu_mlp_set_wait_limit_ns(old)
    try:
        g = run_gpu(t, "bf16")
    finally:
        api.swiglu_mlp_set_cta_pairs(old_p)
    check_all(g, run_oracle(t, "bf16"), "bf16")


# --------------------------------------------------------------------------
# full-size workloads against the oracle: B=8 S=2048 D=1024 H=2816 in full,
# the larger ones on sampled token rows and hidden units
# --------------------------------------------------------------------------
SAMPLED = [
    ("bf16", 8, 4096, 2048, 5632),
    ("f16", 8, 4096, 2048, 5632),
    ("bf16", 8, 8192, 4096, 11008),
]


def _full_size_gpu(t, H):
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    fwd = saved.clone()
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved)
    torch.cuda.synchronize()
    return Y, fwd, saved, dX, dWgu, dWd


@pytest.mark.slow
def test_full_size_full_oracle_b8_s2048_d1024_h2816():
    """Every element of every output at B=8 S=2048 D=1024 H=2816 (bf16)
    against the full oracle (18 M D H fp64 multiply-adds, about a minute)."""
    M, D, H = 8 * 2048, 1024, 2816
    t = synthetic.make_inputs(M, D, H, "bf16", seed=0, device="cuda", kind="device")
    Y, fwd, saved, dX, dWgu, dWd = _full_size_gpu(t, H)
    g = {"Y": f64(Y), "G": f64(fwd[:, :H]), "U": f64(fwd[:, H:2 * H]), "A": f64(fwd[:, 2 * H:]),
         "dG": f64(saved[:, :H]), "dU": f64(saved[:, H:2 * H]), "dX": f64(dX),
         "dWg": f64(dWgu[:H]), "dWu": f64(dWgu[H:]), "dWd": f64(dWd)}
    del fwd, saved
    check_all(g, run_oracle(t, "bf16"), "bf16")


def sample_rows(M, seed):
    """256 seeded token rows, the rows at 128- and 256-row tile seams, the last
    row, and 32 seeded rows in [0, 4096): the first 16 row tiles, where the
    first tiles of the raster order (the stream-K-shared ones, when a GEMM
    shares any) lie."""
    rng = np.random.default_rng(seed)
    seams = [0, 127, 128, 255, 256, 383, 384, 511, 512, 4095, 4096, M - 1]
    return np.unique(np.concatenate([seams, rng.choice(M, 256, replace=False),
                                     rng.choice(min(M, 4096), 32, replace=False)]))


def sample_units(H, seed):
    """128 seeded hidden units, the unit-tile seams and the last unit, and 16
    seeded units among the first 4096 (the first weight-gradient tiles)."""
    rng = np.random.default_rng(seed)
    seams = [0, 63, 64, 127, 128, 255, 256, 511, 512, H - 1]
    return np.unique(np.concatenate([[x for x in seams if x < H],
                                     rng.choice(H, 128, replace=False),
                                     rng.choice(min(H, 4096), 16, replace=False)]))


@pytest.mark.slow
@pytest.mark.parametrize("dtn,B,S,D,H", SAMPLED)
def test_full_size_sampled_parity(dtn, B, S, D, H):
    _sampled_parity(dtn, B, S, D, H)


@pytest.fixture
def wide_tiles():
    """Runs a test with 512-column pair tiles for dWd, dWgu and dX at every
    size (the default takes them by size)."""
    old = api.swiglu_mlp_set_wide_tiles(2)
    yield
    api.swiglu_mlp_set_wide_tiles(old)


@pytest.mark.parametrize("dtn,B,S,D,H", [("bf16", 1, 8192, 1024, 4096), ("f16", 1, 8192, 1024, 4096),
                                         ("bf16", 8, 4096, 2048, 5632)])
def test_wide_tiles_sampled_parity(dtn, B, S, D, H, wide_tiles):
    """512-column tiles for dWd, dWgu and dX against the oracle on the
    sampled rows and units."""
    _sampled_parity(dtn, B, S, D, H)


@pytest.mark.parametrize("M,D,H", [(1000, 200, 392), (513, 648, 776), (4096, 1024, 1000)])
def test_wide_tiles_ragged_parity(M, D, H, wide_tiles):
    """512-column tiles with ragged edges: N not a multiple of 512 (and of
    256), M not a multiple of 256, on SM pairs, against the full oracle."""
    old = api.swiglu_mlp_set_cta_pairs(2)
    try:
        t = synthetic.make_inputs(M, D, H, "bf16", seed=M + D, device="cuda")
        g = run_gpu(t, "bf16")
    finally:
        api.swiglu_mlp_set_cta_pairs(old)
    check_all(g, run_oracle(t, "bf16"), "bf16")


def test_wide_tiles_deterministic_and_close_to_narrow():
    """The 512-column form gives the same bits on every call, and matches
    the 256-column form within accumulation-order rounding (whole tiles sum
    their k-blocks in the same order in both; stream-K-shared tiles split
    at different points)."""
    M, D, H = 8192, 1024, 4096
    t = synthetic.make_inputs(M, D, H, "bf16", seed=61, device="cuda", kind="device")
    outs = {}
    for mode in (2, 2, 0):
        old = api.swiglu_mlp_set_wide_tiles(mode)
        try:
            _, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
            dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved)
            torch.cuda.synchronize()
        finally:
            api.swiglu_mlp_set_wide_tiles(old)
        outs.setdefault(mode, []).append((dX.clone(), dWgu.clone(), dWd.clone()))
    (a, b), (n,) = outs[2], outs[0]
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for x, y in zip(a, n):
        assert oracle.rel_frob(f64(x), f64(y)) <= 2e-3


def _sampled_parity(dtn, B, S, D, H):
    M = B * S
    t = synthetic.make_inputs(M, D, H, dtn, seed=0, device="cuda", kind="device")
    rows = sample_rows(M, M + D)
    cols = sample_units(H, M + H)
    rt = torch.from_numpy(rows).cuda()
    Y, fwd, saved, dX, dWgu, dWd = _full_size_gpu(t, H)
    fwd_rows = fwd.index_select(0, rt).cpu()
    del fwd
    bwd_rows = saved.index_select(0, rt).cpu()
    c = {k: t[k].cpu() for k in ("X", "Wg", "Wu", "Wd", "dY")}
    r = oracle.sampled_rows(c["X"], c["Wg"], c["Wu"], c["Wd"], c["dY"], rows, dt=ODT[dtn])
    q = oracle.sampled_cols(c["X"], c["Wg"], c["Wu"], c["Wd"], c["dY"], cols, dt=ODT[dtn])
    got = {"Y": f64(Y[rt]), "G": f64(fwd_rows[:, :H]), "U": f64(fwd_rows[:, H:2 * H]),
           "A": f64(fwd_rows[:, 2 * H:]), "dG": f64(bwd_rows[:, :H]),
           "dU": f64(bwd_rows[:, H:2 * H]), "dX": f64(dX[rt])}
    for k, v in got.items():
        e = oracle.rel_frob(v, r[k])
        assert e <= TOL[dtn], (k, e)
    for k in ("G", "U", "A", "dG", "dU"):
        f = within_ulp_frac(got[k], r[k], dtn)
        assert f >= 0.99, (k, f)
    ct = torch.from_numpy(cols).cuda()
    e = oracle.rel_frob(f64(dWgu[:H][ct]), q["dWg"]); assert e <= TOL[dtn], ("dWg", e)
    e = oracle.rel_frob(f64(dWgu[H:][ct]), q["dWu"]); assert e <= TOL[dtn], ("dWu", e)
    e = oracle.rel_frob(f64(dWd[:, ct].t()), q["dWdT"]); assert e <= TOL[dtn], ("dWd", e)
    # the sampled rows and units each on their own: no tile is worse than the bound
    for k in ("Y", "dX"):
        per_row = [oracle.rel_frob(got[k][i], r[k][i]) for i in range(len(rows))]
        assert max(per_row) <= 2 * TOL[dtn], (k, rows[int(np.argmax(per_row))], max(per_row))


@pytest.mark.parametrize("S", [1, 2, 16, 64, 256])
def test_nograd_sweep_parity(S):
    D, H = 4096, 11008
    t = synthetic.make_inputs(S, D, H, "bf16", seed=S, device="cuda", kind="device")
    Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    torch.cuda.synchronize()
    rows = np.arange(S) if S <= 16 else np.unique(np.concatenate([[0, S - 1], np.arange(1, S, 17)]))
    c = {k: t[k].cpu() for k in ("X", "Wg", "Wu", "Wd", "dY")}
    r = oracle.sampled_rows(c["X"], c["Wg"], c["Wu"], c["Wd"], c["dY"], rows)
    rt = torch.from_numpy(rows).cuda()
    assert oracle.rel_frob(f64(Y[rt]), r["Y"]) <= 1e-2
    assert within_ulp_frac(f64(A[rt]), r["A"], "bf16") >= 0.99


@pytest.fixture(params=[2, 0], ids=["fused", "two_kernels"])
def ng_mode(request):
    """Runs a test with the few-token no-grad forward as one fused kernel,
    then as two kernels."""
    old = api.swiglu_mlp_set_nograd_fused(request.param)
    yield request.param
    api.swiglu_mlp_set_nograd_fused(old)


@pytest.mark.parametrize("dtn", ["bf16", "f16"])
@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 40, 48, 49, 64, 65, 100, 128])
def test_nograd_small_m_parity(M, dtn, ng_mode):
    """Few-token no-grad path (split contraction, per-tile reduction): ragged
    hidden and feature tiles, several splits per tile, against the oracle and
    against the training forward; two calls give the same bits."""
    D, H = 320, 392
    t = synthetic.make_inputs(M, D, H, dtn, seed=M, device="cuda")
    Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    Y2, A2 = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    Yt, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(A, A2)
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn])
    assert oracle.rel_frob(f64(Y), r["Y"]) <= TOL[dtn]
    assert oracle.rel_frob(f64(A), r["A"]) <= TOL[dtn]
    assert within_ulp_frac(f64(A), r["A"], dtn) >= 0.99
    assert oracle.rel_frob(f64(Y), f64(Yt)) <= TOL[dtn]


@pytest.mark.parametrize("M,D,H", [(1, 4096, 11008), (16, 4096, 11008), (33, 4096, 11008),
                                   (7, 1024, 2816), (64, 2048, 5632), (3, 64, 176),
                                   (16, 8, 8), (5, 320, 392)])
def test_nograd_fused_deterministic_and_matches_oracle(M, D, H):
    """The fused kernel hands out work units dynamically, but every unit's
    partial has a fixed slot and each tile sums its chunks in order: repeated
    calls give the same bits.  Both forms agree with the oracle, and the fused
    one is a single launch."""
    t = synthetic.make_inputs(M, D, H, "bf16", seed=40 + M, device="cuda", kind="device")
    old = api.swiglu_mlp_set_nograd_fused(2)
    try:
        runs = []
        for _ in range(3):
            runs.append(api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"]))
            assert api.swiglu_mlp_last_launch_count() == 1
        api.swiglu_mlp_set_nograd_fused(0)
        Y2, A2 = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
        assert api.swiglu_mlp_last_launch_count() == 2
    finally:
        api.swiglu_mlp_set_nograd_fused(old)
    torch.cuda.synchronize()
    Yf, Af = runs[0]
    for Y, A in runs[1:]:
        assert torch.equal(Y, Yf) and torch.equal(A, Af)
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT["bf16"])
    for got in ((Yf, Af), (Y2, A2)):
        assert oracle.rel_frob(f64(got[0]), r["Y"]) <= TOL["bf16"]
        assert oracle.rel_frob(f64(got[1]), r["A"]) <= TOL["bf16"]
        assert within_ulp_frac(f64(got[1]), r["A"], "bf16") >= 0.99


def test_nograd_fused_reused_workspace_and_mixed_calls():
    """One workspace serves fused calls, two-kernel calls and training calls
    in any order: the ready mask and counters are left clear after each."""
    M, D, H = 16, 1024, 2816
    t = synthetic.make_inputs(M, D, H, "bf16", seed=50, device="cuda", kind="device")
    need = max(api.lib().swiglu_mlp_workspace_bytes(M, D, H, 0, op) for op in (0, 1))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    old = api.swiglu_mlp_set_nograd_fused(2)
    try:
        for step in range(6):
            api.swiglu_mlp_set_nograd_fused(0 if step % 3 == 1 else 2)
            if step == 3:
                api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], ws=ws)
            x = t["X"] if step % 2 == 0 else torch.randn(M, D, device="cuda").bfloat16()
            Y, _ = api.swiglu_mlp_fwd_nograd(x, t["Wgu"], t["Wd"], ws=ws)
            Yr, _ = api.swiglu_mlp_fwd_nograd(x, t["Wgu"], t["Wd"])
            torch.cuda.synchronize()
            assert torch.equal(Y, Yr), step
            assert api.swiglu_mlp_query_error(ws) == 0
    finally:
        api.swiglu_mlp_set_nograd_fused(old)


def test_nograd_fused_unraised_flag_times_out_cleanly():
    """Failure detection of the fused kernel's cross-CTA wait without a fault:
    the first gate/up tile's ready bit is never set, the bounded waits on
    it run out, the kernel records a timeout and returns; the next call on a
    fresh workspace is correct."""
    M, D, H = 16, 320, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=51, device="cuda")
    ws = api.workspace(M, D, H, torch.bfloat16, api.SWIGLU_OP_FWD_NOGRAD, "cuda")
    old_mode = api.swiglu_mlp_set_nograd_fused(2)
    old = api.swiglu_mlp_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        api.swiglu_mlp_inject_stall_once(True)
        assert device_status(
            lambda: api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"], ws=ws), ws) == 6
        Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
        torch.cuda.synchronize()
    finally:
        api.swiglu_mlp_inject_stall_once(False)
        api.swiglu_mlp_set_wait_limit_ns(old)
        api.swiglu_mlp_set_nograd_fused(old_mode)
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT["bf16"])
    assert oracle.rel_frob(f64(Y), r["Y"]) <= TOL["bf16"]
    assert oracle.rel_frob(f64(A), r["A"]) <= TOL["bf16"]


def test_stream_k_shared_tiles_parity_and_determinism(cta_pairs):
    """M=1024, D=512, H=1024 puts every tensor-core GEMM on the stream-K path
    (fewer tiles than SMs: each tile's k-blocks shared by several CTAs, fp32
    partials summed by the last one); results must match the oracle and be
    bitwise reproducible."""
    t = synthetic.make_inputs(1024, 512, 1024, "bf16", seed=12, device="cuda")
    a = run_gpu(t, "bf16")
    b = run_gpu(t, "bf16")
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    check_all(a, run_oracle(t, "bf16"), "bf16")


def test_minimal_workspace_parity(cta_pairs):
    """With the smallest accepted workspace the GEMMs run whole tiles only
    (no stream-K partials): same results within the tolerances, and the
    few-token no-grad call falls back to the two-kernel form."""
    M, D, H = 1024, 512, 1024
    t = synthetic.make_inputs(M, D, H, "bf16", seed=70, device="cuda")
    full = run_gpu(t, "bf16")
    L = api.lib()
    ws_f = api.workspace(M, D, H, torch.bfloat16, api.SWIGLU_OP_FWD, "cuda", minimal=True)
    ws_b = api.workspace(M, D, H, torch.bfloat16, api.SWIGLU_OP_BWD, "cuda", minimal=True)
    assert ws_f.numel() < L.swiglu_mlp_workspace_bytes(M, D, H, 0, api.SWIGLU_OP_BWD)
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], ws=ws_f)
    fs = saved.clone()
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved, ws=ws_b)
    torch.cuda.synchronize()
    assert api.swiglu_mlp_query_error(ws_b) == 0
    small = {"Y": f64(Y), "G": f64(fs[:, :H]), "U": f64(fs[:, H:2 * H]), "A": f64(fs[:, 2 * H:]),
             "dG": f64(saved[:, :H]), "dU": f64(saved[:, H:2 * H]), "dX": f64(dX),
             "dWg": f64(dWgu[:H]), "dWu": f64(dWgu[H:]), "dWd": f64(dWd)}
    check_all(small, run_oracle(t, "bf16"), "bf16")
    for k in small:
        assert oracle.rel_frob(small[k], full[k]) <= 1e-2, k
    # few tokens: the minimal workspace fits the two-kernel form
    tn = synthetic.make_inputs(16, 4096, 11008, "bf16", seed=71, device="cuda", kind="device")
    ws_n = api.workspace(16, 4096, 11008, torch.bfloat16, api.SWIGLU_OP_FWD_NOGRAD, "cuda",
                         minimal=True)
    old = api.swiglu_mlp_set_nograd_fused(2)
    try:
        Yn, _ = api.swiglu_mlp_fwd_nograd(tn["X"], tn["Wgu"], tn["Wd"], ws=ws_n)
        assert api.swiglu_mlp_last_launch_count() in (1, 2)
        Yr, _ = api.swiglu_mlp_fwd_nograd(tn["X"], tn["Wgu"], tn["Wd"])
    finally:
        api.swiglu_mlp_set_nograd_fused(old)
    torch.cuda.synchronize()
    assert oracle.rel_frob(f64(Yn), f64(Yr)) <= 1e-2
