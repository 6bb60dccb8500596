"""GPU self-test of the tcgen05 helpers: a 128 x N x K MMA from shared-memory
tiles in the no-swizzle core-matrix layouts (K-major and MN-major operands,
bf16 and fp16), compared with a host matmul."""
import ctypes
import os
import subprocess

import pytest
import torch

from kimi_delta_attention_rule_gb300 import build as kbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("tc") / "tc_selftest.so")
    cmd = [kbuild.nvcc()] + kbuild.ARCH + ["-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                                          "-I" + kbuild.CSRC, "-I" + kbuild.INCLUDE,
                                          os.path.join(HERE, "tc_selftest.cu"), "-o", out]
    subprocess.check_call(cmd)
    L = ctypes.CDLL(out)
    L.tc_selftest.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    L.tc_selftest.restype = ctypes.c_int
    return L


def run(lib, N, K, b_mn, f16, mn_swap=0):
    dt = torch.float16 if f16 else torch.bfloat16
    g = torch.Generator().manual_seed(N * 1000 + K)
    A = torch.randn(128, K, generator=g).to(dt)
    Bkn = torch.randn(K, N, generator=g).to(dt)
    Bdev = (Bkn if b_mn else Bkn.t().contiguous()).cuda()
    D = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest(A.cuda().data_ptr(), Bdev.data_ptr(), D.data_ptr(), N, K, b_mn, f16,
                         mn_swap, err.data_ptr())
    assert rc == 0 and int(err.item()) == 0, (rc, int(err.item()))
    ref = A.float() @ Bkn.float()
    return (D.cpu() - ref).abs().max().item() / ref.abs().max().item()


@pytest.mark.parametrize("N,K", [(16, 16), (64, 64), (128, 128), (256, 64)])
@pytest.mark.parametrize("f16", [0, 1])
def test_kmajor(lib, N, K, f16):
    assert run(lib, N, K, 0, f16) < 1e-5


@pytest.mark.parametrize("N,K", [(64, 64), (128, 128)])
def test_mnmajor_b(lib, N, K):
    """LBO = stride along K, SBO = stride along N, as for K-major tiles."""
    errs = {swap: run(lib, N, K, 1, f16, swap) for swap in (0, 1) for f16 in (0, 1)}
    assert run(lib, N, K, 1, 0, 0) < 1e-5 and run(lib, N, K, 1, 1, 0) < 1e-5
    assert run(lib, N, K, 1, 1, 1) > 1e-2  # the other field order reads other data
