"""The packed-weights form of the few-token no-grad forward
(swiglu_mlp_pack_weights + swiglu_mlp_fwd_nograd_packed), through the C ABI.

The packed copy stores each 16 KB weight block of the few-token kernels
contiguously and pre-swizzled, so the kernels see the same shared-memory
contents as when they load the blocks from the row-major weights with
tensor maps: the outputs must be bitwise equal to swiglu_mlp_fwd_nograd's
two-kernel form.  The layout itself is checked byte for byte against a
numpy restatement of its definition."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic

pytestmark = pytest.mark.gpu

ODT = {"bf16": oracle.BF16, "f16": oracle.F16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


@pytest.fixture(autouse=True)
def _two_kernels():
    old = api.swiglu_mlp_set_nograd_fused(0)
    yield
    api.swiglu_mlp_set_nograd_fused(old)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def pack_reference(Wgu, Wd):
    """The layout's definition, written out: blocks of 128 rows x 64 elements,
    gate/up blocks (64 Wg rows, then the 64 Wu rows of the same units) then
    down blocks (128 Wd rows), each block's 16-byte chunk c of row r at
    position c ^ (r mod 8); zeros past D or H."""
    wgu, wd = _bits(Wgu), _bits(Wd)
    H2, D = wgu.shape
    H = H2 // 2

    def blocks(rows_of, nt, K, nk, src):
        out = np.zeros((nt, nk, 128, 64), np.uint16)
        for t in range(nt):
            for r, row in enumerate(rows_of(t)):
                if row is None:
                    continue
                for kb in range(nk):
                    k0, k1 = kb * 64, min(K, kb * 64 + 64)
                    if k0 < K:
                        out[t, kb, r, :k1 - k0] = src[row, k0:k1]
        chunks = out.reshape(nt, nk, 128, 8, 8)
        sw = np.empty_like(chunks)
        for r in range(128):
            for p in range(8):
                sw[:, :, r, p] = chunks[:, :, r, p ^ (r & 7)]
        return sw.reshape(-1)

    t1, kb1 = -(-H // 64), -(-D // 64)
    t2, kb2 = -(-D // 128), -(-H // 64)
    gu = blocks(lambda t: [(t * 64 + i if t * 64 + i < H else None) for i in range(64)]
                + [(H + t * 64 + i if t * 64 + i < H else None) for i in range(64)],
                t1, D, kb1, wgu)
    dn = blocks(lambda t: [(t * 128 + i if t * 128 + i < D else None) for i in range(128)],
                t2, H, kb2, wd)
    return np.concatenate([gu, dn])


@pytest.mark.parametrize("D,H", [(72, 80), (320, 392), (128, 64)])
def test_packed_layout_matches_its_definition(D, H):
    t = synthetic.make_inputs(1, D, H, "bf16", seed=D + H, device="cuda")
    packed = api.swiglu_mlp_pack_weights(t["Wgu"], t["Wd"])
    torch.cuda.synchronize()
    assert packed.numel() == api.lib().swiglu_mlp_packed_weights_bytes(D, H, 0)
    got = packed.cpu().numpy().view(np.uint16)
    ref = pack_reference(t["Wgu"], t["Wd"])
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtn", ["bf16", "f16"])
@pytest.mark.parametrize("M,D,H", [(1, 320, 392), (5, 320, 392), (16, 320, 392), (17, 320, 392),
                                   (33, 320, 392), (40, 320, 392), (48, 320, 392),
                                   (64, 320, 392), (3, 72, 80),
                                   (1, 4096, 11008), (16, 4096, 11008), (32, 4096, 11008),
                                   (48, 4096, 11008), (64, 4096, 11008)])
def test_packed_forward_bitwise_equals_plain(M, D, H, dtn):
    t = synthetic.make_inputs(M, D, H, dtn, seed=500 + M, device="cuda", kind="device")
    packed = api.swiglu_mlp_pack_weights(t["Wgu"], t["Wd"])
    Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    Yp, Ap = api.swiglu_mlp_fwd_nograd_packed(t["X"], packed, H)
    assert api.swiglu_mlp_last_launch_count() == 2
    torch.cuda.synchronize()
    assert torch.equal(Y, Yp) and torch.equal(A, Ap)


def test_packed_forward_multipliers_and_oracle():
    M, D, H = 7, 320, 392
    t = synthetic.make_inputs(M, D, H, "bf16", seed=77, device="cuda")
    packed = api.swiglu_mlp_pack_weights(t["Wgu"], t["Wd"])
    Y, A = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"], gate_mul=0.5, down_mul=2.0)
    Yp, Ap = api.swiglu_mlp_fwd_nograd_packed(t["X"], packed, H, gate_mul=0.5, down_mul=2.0)
    torch.cuda.synchronize()
    assert torch.equal(Y, Yp) and torch.equal(A, Ap)
    Yp1, Ap1 = api.swiglu_mlp_fwd_nograd_packed(t["X"], packed, H)
    torch.cuda.synchronize()
    c = {k: v.cpu() for k, v in t.items()}
    r = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT["bf16"])
    assert oracle.rel_frob(Yp1.double().cpu().numpy(), r["Y"]) <= 1e-2
    assert oracle.rel_frob(Ap1.double().cpu().numpy(), r["A"]) <= 1e-2


def test_packed_forward_limits():
    D, H = 64, 128
    t = synthetic.make_inputs(65, D, H, "bf16", seed=3, device="cuda")
    packed = api.swiglu_mlp_pack_weights(t["Wgu"], t["Wd"])
    with pytest.raises(api.SwigluError) as e:   # more tokens than the few-token path
        api.swiglu_mlp_fwd_nograd_packed(t["X"], packed, H)
    assert e.value.code == 3
    Y, A = api.swiglu_mlp_fwd_nograd_packed(t["X"][:0], packed, H)   # empty batch
    assert api.swiglu_mlp_last_launch_count() == 0
    assert Y.shape == (0, D) and A.shape == (0, H)
