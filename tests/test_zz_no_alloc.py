"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (it takes its scratch from a static device array in
the library instead of a caller-provided workspace). Checked through the C
ABI against kda_prefill, the entry point that takes a workspace, on two
calls in a row (the second call reuses the array the first one left
behind). This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import build as kbuild, inputs

pytestmark = pytest.mark.gpu
TOL_BF16 = 2e-2


def _noalloc_fn():
    kbuild.build()
    lib = kda.load()
    f = lib.kda_prefill_noalloc
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, I32, I32, I32, I32, I32, I32, P, P, P]
    f.restype = ctypes.c_int
    return f


def _max_rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    rms = float(np.sqrt(np.mean(b ** 2))) or 1.0
    return float(np.max(np.abs(a - b))) / rms


def test_noalloc_matches_workspace_entry_point_twice():
    f = _noalloc_fn()
    dev = torch.device("cuda:0")
    x = inputs.prefill_inputs([150, 77, 0, 64], H=3, io="bf16", seed=31, init="normal")
    q, k, v, g, b = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    init, cu = x.init_state.to(dev), x.cu_seqlens.to(dev)
    ref_out, ref_fin = kda.kda_prefill(q, k, v, g, b, x.scale, init_state=init, cu_seqlens=cu,
                                       chunk=64)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    N, T, H = cu.numel() - 1, q.shape[0], q.shape[1]
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        fin = torch.full((N, H, 128, 128), float("nan"), dtype=torch.float32, device=dev)
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), b.data_ptr(), x.scale,
               init.data_ptr(), cu.data_ptr(), N, T, H, 128, 64, kda.KDA_BF16, out.data_ptr(),
               fin.data_ptr(), stream)
        assert rc == kda.KDA_OK, kda.status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
        assert _max_rel(out, ref_out) <= TOL_BF16
        assert _max_rel(fin, ref_fin) <= TOL_BF16


def test_noalloc_rejects_bad_arguments_like_kda_prefill():
    f = _noalloc_fn()
    # D != 128 is unsupported, before anything is launched
    rc = f(None, None, None, None, None, 1.0, None, None, 1, 64, 2, 64, 64, kda.KDA_BF16, None,
           None, None)
    assert rc == kda.KDA_ERR_UNSUPPORTED


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    f = _noalloc_fn()
    # H=32, T=8192 needs ~312 MB of prepared chunk blocks: far beyond 16 MiB
    need = kda.kda_prefill_workspace_size(1, 8192, 32, 128, 64, kda.KDA_BF16, False)
    assert need > 16 << 20
    rc = f(None, None, None, None, None, 1.0, None, None, 1, 8192, 32, 128, 64, kda.KDA_BF16,
           None, None, None)
    assert rc == kda.KDA_ERR_TOO_LARGE
