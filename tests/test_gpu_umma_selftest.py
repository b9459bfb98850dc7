"""tcgen05 building blocks (descriptors, swizzled layouts, TMEM operand,
MMA, commit, TMEM loads) checked on one tile against a float64 matmul. The
self-test library uses the same inline-PTX header as the tensor-core
partial kernel."""

import ctypes

import numpy as np
import pytest
import torch

from mla_speculative_decoding_gb300 import build as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probe():
    lib = ctypes.CDLL(B.build_selftest())
    f = lib.mlav_umma_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    return f


def _run(probe, mode, N, variant=0, seed=0):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, 64, generator=g).to(torch.bfloat16) if mode in (0, 1) else \
        torch.randn(64, N, generator=g).to(torch.bfloat16)
    dA, dB = A.cuda(), Bm.cuda()
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, mode, variant, err.data_ptr())
    assert rc == 0, f"probe launch failed: {rc}"
    assert int(err.item()) == 0, "probe wait timed out"
    a = A.double()
    ref = a @ (Bm.double().T if mode in (0, 1) else Bm.double())
    return D.cpu().double(), ref


@pytest.mark.parametrize("N", [32, 64, 128, 256])
@pytest.mark.parametrize("mode", [0, 1])
def test_kmajor_b(probe, mode, N):
    got, ref = _run(probe, mode, N)
    torch.testing.assert_close(got, ref, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("mode", [2, 3])
def test_mnmajor_b(probe, mode, N):
    """MN-major B (the V operand): one of the two stride assignments must be
    right; the kernel uses variant 0 (atom-column stride in the leading
    field)."""
    got, ref = _run(probe, mode, N, variant=0)
    ok0 = torch.allclose(got, ref, rtol=1e-4, atol=1e-3)
    got1, _ = _run(probe, mode, N, variant=1)
    ok1 = torch.allclose(got1, ref, rtol=1e-4, atol=1e-3)
    print(f"mode {mode} N {N}: variant0 {ok0} variant1 {ok1}")
    assert ok0, f"variant 0 wrong (variant 1 {'right' if ok1 else 'also wrong'})"


def test_tma_gather4_rows_and_zero_fill():
    """tile::gather4 through the KV tensor map: 8 scattered rows x 64 columns land
    as 128B-swizzled rows; an out-of-range row reads zeros."""
    lib = ctypes.CDLL(B.build_selftest())
    f = lib.mlav_gather_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p]
    slots = 1000
    g = torch.Generator().manual_seed(3)
    kv = torch.randn(slots, 576, generator=g).to(torch.bfloat16)
    dkv = kv.cuda()
    rows = [5, 999, 0, 17, slots, 512, 3, 770]   # one out-of-range row
    for x in (0, 64, 512):
        out = torch.zeros(1024, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = f(dkv.data_ptr(), slots, (ctypes.c_int * 8)(*rows), x, out.data_ptr(), err.data_ptr())
        assert rc == 0 and int(err.item()) == 0, rc
        raw = out.cpu().view(torch.int16).view(8, 8, 8)  # [row][16B chunk][8 bf16]
        for i, r in enumerate(rows):
            want = (kv[r, x:x + 64].view(torch.int16).view(8, 8) if r < slots
                    else torch.zeros(8, 8, dtype=torch.int16))
            for c in range(8):
                assert torch.equal(raw[i, c ^ (i % 8)], want[c]), (x, i, c)


@pytest.fixture(scope="module")
def pair_probe():
    lib = ctypes.CDLL(B.build_selftest())
    f = lib.mlav_pair_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 3
    return f


@pytest.mark.parametrize("mode,N", [(0, 128), (0, 256), (1, 128), (1, 256), (2, 256)])
def test_cta_pair_mma(pair_probe, mode, N):
    """2-SM MMA (cta_group::2, M = 256) as the four-SM kernel uses it: A rows
    split across the pair (shared memory or TMEM), B's N columns split across
    the pair (K-major or MN-major), commit multicast to both CTAs, each CTA
    reading its 128 rows of D; the pair's allocation result is the same in
    both CTAs."""
    g = torch.Generator().manual_seed(7 * mode + N)
    A = torch.randn(256, 64, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, 64, generator=g).to(torch.bfloat16) if mode in (0, 1) else \
        torch.randn(64, N, generator=g).to(torch.bfloat16)
    dA, dB = A.cuda(), Bm.cuda()
    D = torch.full((256, N), float("nan"), dtype=torch.float32, device="cuda")
    addr = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = pair_probe(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, mode, 1, 0, addr.data_ptr(),
                    cyc.data_ptr(), err.data_ptr())
    assert rc == 0, f"pair probe launch failed: {rc}"
    assert int(err.item()) == 0, "pair probe wait timed out"
    a = addr.cpu().tolist()
    assert a[0] == a[1], f"allocation differs between the CTAs of the pair: {a}"
    ref = A.double() @ (Bm.double().T if mode in (0, 1) else Bm.double())
    torch.testing.assert_close(D.cpu().double(), ref, rtol=1e-4, atol=1e-3)
