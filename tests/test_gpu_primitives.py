"""Device primitives through the C ABI: exp2 variants, a one-tile tcgen05 MMA
probe for each operand form the kernels use, and the bounded-wait timeout path."""
import numpy as np
import pytest
import torch

import exact_attention_smem_gb300 as fa
import fa_testing_lib as ft
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    ft.fa_test_get_device_error(clear=True)
    yield
    assert ft.fa_test_get_device_error(clear=True) == 0


def _exp2_dev(x, mode):
    xd = torch.tensor(x, dtype=torch.float32, device="cuda")
    y = torch.empty_like(xd)
    ft.fa_test_exp2(xd, y, mode)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_poly_exp2_device_matches_host_twin_bitwise():
    xs = np.concatenate([np.linspace(-130, 8, 100001, dtype=np.float32),
                         (np.arange(0x8000, 0x10000, dtype=np.uint32) << 16).view(np.float32)])
    xs = xs[~np.isnan(xs)]
    dev = _exp2_dev(xs, 0)
    host = np.array([ft.fa_exp2_poly_host(float(x)) for x in xs], dtype=np.float32)
    assert np.array_equal(dev.view(np.uint32), host.view(np.uint32))
    sel = xs >= -125
    rel = np.abs(dev[sel] / oracle.exp2_exact(xs[sel].astype(np.float64)) - 1)
    assert rel.max() <= 2.0 ** -13


def test_mufu_exp2_accuracy():
    xs = np.linspace(-125, 8, 200001, dtype=np.float32)
    dev = _exp2_dev(xs, 1)
    rel = np.abs(dev / oracle.exp2_exact(xs.astype(np.float64)) - 1)
    assert rel.max() <= 2.0 ** -20


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_mma_probe(mode, N):
    g = torch.Generator().manual_seed(100 + mode * 7 + N)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    B = torch.randn(*((N, 128) if mode == 0 else (128, N)), generator=g).to(torch.bfloat16)
    C = torch.full((128, N), float("nan"), device="cuda")
    ft.fa_test_mma(A.cuda(), B.cuda(), C, mode, N)
    torch.cuda.synchronize()
    a, b = A.double().numpy(), B.double().numpy()
    want = a @ b.T if mode == 0 else (a @ b if mode == 1 else a.T @ b)
    got = C.cpu().double().numpy()
    assert np.abs(got - want).max() <= 1e-3 * max(1.0, np.abs(want).max())


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_mma_fp8_probe(mode, N):
    """kind::f8f6f4 with e4m3 operands: the products of e4m3 values are exact
    in fp32, so a 128-term fp32 sum is within 128 * 2^-24 (< 1e-5) of the
    exact value, relative to the sum of the terms' magnitudes."""
    rng = np.random.default_rng(300 + mode * 7 + N)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    A = rng.choice(codes, (128, 128))
    B = rng.choice(codes, (N, 128))
    C = torch.full((128, N), float("nan"), device="cuda")
    ft.fa_test_mma_fp8(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, mode, N)
    torch.cuda.synchronize()
    a, b = oracle.fp8_e4m3.e4m3_decode(A), oracle.fp8_e4m3.e4m3_decode(B)
    want = a @ b.T
    got = C.cpu().double().numpy()
    scale = (np.abs(a) @ np.abs(b).T).max()
    assert np.abs(got - want).max() <= 1e-5 * scale


def test_tma_and_tmem_round_trips():
    """A TMA load + TMA store of one swizzled tile returns the tile bit for bit;
    a tensor-memory store + load returns every lane's words."""
    src = torch.randn(128, 64, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    dst = torch.zeros_like(src)
    out = torch.zeros(128, 32, dtype=torch.int32, device="cuda")
    ft.fa_test_roundtrip(src, dst, out)
    torch.cuda.synchronize()
    assert ft.fa_test_get_device_error(clear=True) == 0
    assert torch.equal(dst.view(torch.int16), src.view(torch.int16))
    want = torch.arange(128).view(128, 1) * 1000 + torch.arange(32).view(1, 32)
    assert torch.equal(out.cpu(), want.to(torch.int32))


@pytest.mark.parametrize("N", [128])
@pytest.mark.parametrize("mode", [0, 1])
def test_mma_pair_probe(mode, N):
    """cta_group::2: one M=256 MMA chain over a cluster of two CTAs."""
    g = torch.Generator().manual_seed(200 + mode * 7 + N)
    A = torch.randn(256, 128, generator=g).to(torch.bfloat16)
    B = torch.randn(*((N, 128) if mode == 0 else (128, N)), generator=g).to(torch.bfloat16)
    C = torch.full((256, N), float("nan"), device="cuda")
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    ft.fa_test_mma_pair(A.cuda(), B.cuda(), C, flags, mode, N)
    torch.cuda.synchronize()
    assert ft.fa_test_get_device_error(clear=True) == 0
    f = flags.cpu().tolist()
    assert f[0] == 1 and f[1] == 1 and f[2] == f[3], f
    a, b = A.double().numpy(), B.double().numpy()
    want = a @ b.T if mode == 0 else a @ b
    got = C.cpu().double().numpy()
    assert np.abs(got - want).max() <= 1e-3 * max(1.0, np.abs(want).max())


def test_bounded_wait_times_out_instead_of_hanging():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ft.fa_test_wait_timeout(status, 50.0)
    torch.cuda.synchronize()
    assert status.item() == 1
    assert ft.fa_test_get_device_error(clear=True) == 901
