"""The tcgen05 building blocks (TMEM alloc, K-major no-swizzle descriptors,
kind::f16 MMA on bf16 and fp16 inputs, commit, tcgen05.ld / st) against a
numpy matmul, before the chunked prefill relies on them."""

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from linear_attention_decode_kda_gb300 import build as gbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("tc") / "libtcselftest.so")
    subprocess.run([gbuild.NVCC, *gbuild.ARCH, *gbuild.FLAGS, "-shared",
                    os.path.join(HERE, "native", "tc_selftest.cu"), "-o", out], check=True)
    l = ctypes.CDLL(out)
    l.tc_selftest.restype = ctypes.c_int
    l.tc_selftest.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    return l


@pytest.mark.parametrize("K,N", [(16, 64), (64, 64), (128, 64), (128, 128), (64, 128)])
@pytest.mark.parametrize("mode", [0, 1, 2, 4, 5, 8, 13, 16, 17, 24, 29, 32, 40, 44, 48, 56])
def test_tcgen05_mma(lib, K, N, mode):
    """Modes (bits): 1 negate A, 2 twice, 4 accumulate onto D0, 8 fp16 (else bf16),
    16 A from TMEM, 32 A and B in the 128-byte swizzled layout (K a multiple of 64)."""
    if mode & 32 and K % 64:
        pytest.skip("the swizzled layout takes 64-element atoms")
    g = torch.Generator().manual_seed(K * 1000 + N * 10 + mode)
    dt = torch.float16 if mode & 8 else torch.bfloat16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    D0 = torch.randn(128, N, generator=g)
    dA, dB, dD0 = A.cuda(), B.cuda(), D0.cuda()
    dD = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest(dA.data_ptr(), dB.data_ptr(), dD0.data_ptr(), dD.data_ptr(), K, N, mode,
                         err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "mbarrier wait timed out"
    P = A.double().numpy() @ B.double().numpy().T
    want = -P if mode & 1 else P
    if mode & 2:
        want = 2 * want
    if mode & 4:
        want = want + D0.double().numpy()
    got = dD.cpu().double().numpy()
    scale = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(got - want)) <= 1e-5 * scale * K, np.max(np.abs(got - want)) / scale
