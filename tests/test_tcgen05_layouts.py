"""GPU self-test of the tcgen05 helpers: an M x N x K MMA (M = 128 or 64) from
shared-memory tiles in the no-swizzle core-matrix layouts (K-major and
MN-major operands, bf16 and fp16), compared with a host matmul. For M = 64 the
test also pins which TMEM lanes hold the rows of D: rows 16 w .. 16 w + 15 in
lanes 32 w .. 32 w + 15 (the first half of each warp's lane quarter)."""
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
    L.tc_selftest.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p]
    L.tc_selftest.restype = ctypes.c_int
    return L


def M64_LANE(m):
    return 32 * (m // 16) + m % 16


def mma_lanes(lib, M, N, K, a_mn, b_mn, f16, mn_swap=0):
    """(all 128 TMEM lanes x N columns after the MMA, the host product)."""
    dt = torch.float16 if f16 else torch.bfloat16
    g = torch.Generator().manual_seed(M * 7 + N * 1000 + K)
    A = torch.randn(M, K, generator=g).to(dt)
    Bkn = torch.randn(K, N, generator=g).to(dt)
    Adev = (A.t().contiguous() if a_mn else A).cuda()
    Bdev = (Bkn if b_mn else Bkn.t().contiguous()).cuda()
    D = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest(Adev.data_ptr(), Bdev.data_ptr(), D.data_ptr(), M, N, K, a_mn, b_mn,
                         f16, mn_swap, err.data_ptr())
    assert rc == 0 and int(err.item()) == 0, (rc, int(err.item()))
    return D.cpu(), A.float() @ Bkn.float()


def run(lib, N, K, b_mn, f16, mn_swap=0, M=128, a_mn=0):
    D, ref = mma_lanes(lib, M, N, K, a_mn, b_mn, f16, mn_swap)
    if M == 64:
        D = D[[M64_LANE(m) for m in range(64)]]
    return (D - ref).abs().max().item() / ref.abs().max().item()


@pytest.mark.parametrize("N,K", [(16, 16), (64, 64), (128, 128), (256, 64)])
@pytest.mark.parametrize("f16", [0, 1])
def test_kmajor(lib, N, K, f16):
    assert run(lib, N, K, 0, f16) < 1e-5


@pytest.mark.parametrize("N,K", [(64, 64), (128, 128), (192, 64)])
def test_mnmajor_b(lib, N, K):
    """LBO = stride along K, SBO = stride along N, as for K-major tiles."""
    errs = {swap: run(lib, N, K, 1, f16, swap) for swap in (0, 1) for f16 in (0, 1)}
    assert run(lib, N, K, 1, 0, 0) < 1e-5 and run(lib, N, K, 1, 1, 0) < 1e-5
    # the other field order reads other data (which may decode to inf or NaN)
    assert not run(lib, N, K, 1, 1, 1) <= 1e-2


@pytest.mark.parametrize("N,K", [(16, 128), (32, 128), (128, 64)])
def test_m64_lane_map(lib, N, K):
    """M = 64: each row of D is found in exactly the lane the kernels read."""
    D, ref = mma_lanes(lib, 64, N, K, 0, 0, 0)
    scale = ref.abs().max().item()
    found = {}
    for m in range(64):
        errs = (D - ref[m]).abs().max(dim=1).values / scale
        found[m] = int(torch.argmin(errs))
        assert errs[found[m]] < 1e-5, (m, float(errs[found[m]]))
    assert all(found[m] == M64_LANE(m) for m in range(64)), found


@pytest.mark.parametrize("M", [64, 128])
@pytest.mark.parametrize("f16", [0, 1])
def test_mnmajor_a(lib, M, f16):
    """A stored MN-major (K rows of M contiguous elements), same field order."""
    assert run(lib, 64, 64, 0, f16, M=M, a_mn=1) < 1e-5
    assert run(lib, 128, 64, 1, f16, M=M, a_mn=1) < 1e-5
