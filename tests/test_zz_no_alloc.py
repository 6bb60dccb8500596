"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (it takes its scratch from a static device array in
the library instead of a caller-provided workspace). Checked through the C
ABI against kda_prefill, the entry point that takes a workspace, on two
calls in a row (the second call reuses the array the first one left
behind): both run the same kernels on the same inputs, so their results must
agree bit for bit; one comparison against the fp64 oracle as well. Device
errors are read back with kda_noalloc_status. This file is collected last on
purpose."""
import ctypes

import pytest
import torch

import oracle
import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import build as kbuild, inputs
from tests.parity import TOL_BF16, np32, out_err, rel_err

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    kbuild.build()
    lib = kda.load()
    return lib.kda_prefill_noalloc


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
               fin.data_ptr(), ctypes.c_void_p(stream))
        assert rc == kda.KDA_OK, kda.status_string(rc)
        assert kda.kda_noalloc_status() == kda.KDA_OK
        assert torch.equal(out, ref_out)
        assert torch.equal(fin, ref_fin)
    ro, rf = oracle.prefill(np32(x.q), np32(x.k), np32(x.v), np32(x.g), np32(x.beta), x.scale,
                            init_state=x.init_state.double().numpy(),
                            cu_seqlens=x.cu_seqlens.numpy())
    assert out_err(out, ro) <= TOL_BF16
    assert rel_err(fin.cpu().numpy(), rf) <= TOL_BF16


def test_noalloc_reports_bad_offsets_through_its_status_query():
    """Offsets that go back and forth are flagged on the device; the caller of
    the noalloc entry point reads the flag with kda_noalloc_status (which also
    clears it), and a correct call afterwards reports KDA_OK."""
    _noalloc_fn()
    dev = torch.device("cuda:0")
    T_total, N = 129, 5
    x = inputs.prefill_inputs([T_total], H=1, io="bf16", seed=32)
    q, k, v, g, b = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    cu = torch.tensor([0 if i % 2 == 0 else T_total for i in range(N + 1)], dtype=torch.int32,
                      device=dev)
    out = torch.full_like(q, 7.0)
    kda.kda_prefill_noalloc(q, k, v, g, b, x.scale, cu_seqlens=cu, out=out)
    assert kda.kda_noalloc_status() == kda.KDA_ERR_DEVICE
    assert kda.kda_noalloc_status() == kda.KDA_OK  # the read cleared it
    assert torch.all(out == 7.0)  # the call was skipped as a whole
    good = torch.tensor([0, T_total], dtype=torch.int32, device=dev)
    kda.kda_prefill_noalloc(q, k, v, g, b, x.scale, cu_seqlens=good, out=out)
    assert kda.kda_noalloc_status() == kda.KDA_OK


def test_noalloc_rejects_bad_arguments_like_kda_prefill():
    f = _noalloc_fn()
    # D != 128 is unsupported, before anything is launched
    rc = f(None, None, None, None, None, 1.0, None, None, 1, 64, 2, 64, 64, kda.KDA_BF16, None,
           None, None)
    assert rc == kda.KDA_ERR_UNSUPPORTED


def test_noalloc_runs_the_ring_plan_when_the_full_one_does_not_fit():
    """H=16, T=2048: the full plan needs ~38 MB of prepared blocks, beyond the
    16 MiB array; the call runs the fused schedule with rings (fewer chains
    per group than the modelled best, so more than one group) and agrees bit
    for bit with kda_prefill on a full workspace."""
    f = _noalloc_fn()
    dev = torch.device("cuda:0")
    N, T, H = 1, 2048, 16
    bf = kda.KDA_BF16
    assert kda.kda_prefill_workspace_size(N, T, H, 128, 64, bf, True) > 16 << 20
    plan = kda.kda_prefill_plan(N, T, H, 128, 64, bf, True, 16 << 20)
    assert plan.schedule == kda.KDA_SCHEDULE_FUSED and plan.ring > 0 and plan.groups > 1
    x = inputs.prefill_inputs([T], H=H, io="bf16", seed=33, init="normal")
    q, k, v, g, b = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    init, cu = x.init_state.to(dev), x.cu_seqlens.to(dev)
    ref_out, ref_fin = kda.kda_prefill(q, k, v, g, b, x.scale, init_state=init, cu_seqlens=cu,
                                       chunk=64)
    torch.cuda.synchronize()
    out = torch.full_like(q, float("nan"))
    fin = torch.full((N, H, 128, 128), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), b.data_ptr(), x.scale,
           init.data_ptr(), cu.data_ptr(), N, T, H, 128, 64, bf, out.data_ptr(), fin.data_ptr(),
           ctypes.c_void_p(stream))
    assert rc == kda.KDA_OK, kda.status_string(rc)
    assert kda.kda_noalloc_status() == kda.KDA_OK
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    """Only the per-sequence schedule data can outgrow the array: about two
    million packed sequences. Rejected before anything is launched (the
    pointers are never read)."""
    f = _noalloc_fn()
    N = 2_200_000
    need = kda.kda_prefill_workspace_size_min(N, N, 1, 128, 64, kda.KDA_BF16, True)
    assert need > 16 << 20
    cu = torch.zeros(4, dtype=torch.int32, device="cuda:0")  # not read
    rc = f(None, None, None, None, None, 1.0, None, cu.data_ptr(), N, N, 1, 128, 64,
           kda.KDA_BF16, None, None, None)
    assert rc == kda.KDA_ERR_TOO_LARGE
