"""GPU parity outside the unit-scale draws of the workloads: values v scaled
up to 1e5, initial states with entries of order 1e3 to 1e5, keys of norm 0.5
and queries of norm 4, against the fp64 oracle.

The operator is linear in v and in the initial state, so these inputs are
as valid as the unit-scale ones; the bf16 prefill carries the value side of
its state path (beta v, the pseudo-values, the state operand of the chunk
products) in fp16 and must rescale it rather than overflow. Both bf16
schedules (and the fused one with per-chain rings), the fp32 path and decode
are covered. Metric and bars as in the
other parity tests (relative to the RMS of the oracle's result, so they do
not depend on the scale).
"""
import pytest
import torch

import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import inputs
from tests.parity import (DEV, TOL_BF16, TOL_F32, np32, oracle_prefill, out_err,
                          prefill_schedule, rel_err, run_gpu_prefill)
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kimi_delta_attention_rule_gb300 import build as kbuild
    kbuild.build()
    kda.load()


def scaled_inputs(io, seed, v_scale=1.0, state_std=0.02, k_norm=1.0, q_norm=1.0,
                  lens=(300, 1, 129), H=2, g_mode="standard"):
    """Workload draws with v, the initial state, k and q rescaled; the
    rescaled tensors are rounded to their stored dtype once, and both sides
    read those stored values."""
    x = inputs.prefill_inputs(list(lens), H=H, io=io, seed=seed, init="normal", g_mode=g_mode)
    dt = x.q.dtype
    x.v = (x.v.float() * v_scale).to(dt)
    x.k = (x.k.float() * k_norm).to(dt)
    x.q = (x.q.float() * q_norm).to(dt)
    x.init_state = x.init_state * (state_std / 0.02)
    return x


CASES = [
    dict(v_scale=1e2),
    dict(v_scale=1e4),
    dict(v_scale=1e5),
    dict(state_std=1e3),
    dict(state_std=1e5),
    dict(k_norm=0.5, q_norm=4.0),
    dict(v_scale=1e5, state_std=1e5, k_norm=0.5),
    dict(v_scale=1e-3, state_std=1e5),     # state far larger than the new values
    dict(v_scale=1e5, state_std=1e-4),     # values far larger than the state
]


def _id(c):
    return ",".join("%s=%s" % kv for kv in c.items())


@pytest.mark.parametrize("mode", ["split", "fused", "ring"])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_bf16_prefill_scaled(case, mode):
    x = scaled_inputs("bf16", 201, **case)
    with prefill_schedule(mode):
        out, fin = run_gpu_prefill(x, 64, ws_kind="ring" if mode == "ring" else "fast")
    ro, rf = oracle_prefill(x)
    eo, ef = out_err(out, ro), rel_err(fin.cpu().numpy(), rf)
    assert eo <= TOL_BF16 and ef <= TOL_BF16, (eo, ef)


@pytest.mark.parametrize("case", [dict(v_scale=1e5, state_std=1e5, k_norm=0.5),
                                  dict(v_scale=1e4, g_mode="floor")], ids=_id)
def test_bf16_prefill_scaled_long(case):
    """A long sequence (many chunks of the chain) and a ragged tail."""
    x = scaled_inputs("bf16", 202, lens=(2000,), H=3, **case)
    out, fin = run_gpu_prefill(x, 64)
    ro, rf = oracle_prefill(x)
    eo, ef = out_err(out, ro), rel_err(fin.cpu().numpy(), rf)
    assert eo <= TOL_BF16 and ef <= TOL_BF16, (eo, ef)


@pytest.mark.parametrize("mode", ["split", "fused", "ring"])
@pytest.mark.parametrize("first,then", [(1e-3, 1e4), (1e4, 1e-3), (1.0, 3e4)])
def test_bf16_prefill_value_jump(first, then, mode):
    """The magnitude of v changes by up to 1e7 within a sequence (after 192
    tokens, on a chunk boundary, and again mid-chunk at token 300): the state's
    scale must follow both ways."""
    x = scaled_inputs("bf16", 206, lens=(700, 300), H=2, state_std=1e-4)
    v = x.v.float()
    v[:192] *= first
    v[192:300] *= then
    v[300:700] *= first
    v[700:] *= then
    x.v = v.to(torch.bfloat16)
    with prefill_schedule(mode):
        out, fin = run_gpu_prefill(x, 64, ws_kind="ring" if mode == "ring" else "fast")
    ro, rf = oracle_prefill(x)
    eo, ef = out_err(out, ro), rel_err(fin.cpu().numpy(), rf)
    assert eo <= TOL_BF16 and ef <= TOL_BF16, (eo, ef)
    # the small-valued stretch keeps its own precision (not swamped by the large one)
    lo = slice(0, 192) if first < then else slice(192, 300)
    assert out_err(out[lo], ro[lo]) <= TOL_BF16


def test_bf16_prefill_beyond_range_is_reported():
    """v of order 1e30 (representable in bf16, beyond the ~1e20 the state path
    scales to): an fp16 value overflows, the final state is not finite, and the
    call reports KDA_ERR_RANGE instead of returning quietly; the next call is
    fine."""
    x = scaled_inputs("bf16", 207, v_scale=1e30, lens=(200,), H=2)
    q = x.q.to(DEV)
    ws = kda.prefill_workspace(q, x.cu_seqlens.to(DEV), chunk=64)
    _, fin = kda.kda_prefill(q, x.k.to(DEV), x.v.to(DEV), x.g.to(DEV), x.beta.to(DEV), x.scale,
                             init_state=x.init_state.to(DEV), cu_seqlens=x.cu_seqlens.to(DEV),
                             chunk=64, workspace=ws)
    assert kda.kda_workspace_status(ws) == kda.KDA_ERR_RANGE
    assert not torch.isfinite(fin).all()
    y = scaled_inputs("bf16", 207, v_scale=1e20, lens=(200,), H=2)
    out, fin = run_gpu_prefill(y, 64)
    ro, rf = oracle_prefill(y)
    assert out_err(out, ro) <= TOL_BF16 and rel_err(fin.cpu().numpy(), rf) <= TOL_BF16


def test_bf16_prefill_scaled_snapshots():
    """Snapshots are written in the state's own units (not in a scaled form)."""
    x = scaled_inputs("bf16", 203, v_scale=1e5, state_std=1e3, lens=(300,), H=2)
    snaps = torch.zeros((1, 4, 2, 128, 128), dtype=torch.float32, device=DEV)
    kda.kda_prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), x.g.to(DEV), x.beta.to(DEV), x.scale,
                    init_state=x.init_state.to(DEV), cu_seqlens=x.cu_seqlens.to(DEV), chunk=64,
                    snapshot_interval=64, snapshots=snaps)
    torch.cuda.synchronize()
    for si in range(4):
        P = (si + 1) * 64
        sl = lambda t: np32(t[:P])
        _, rs = oracle.prefill(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), x.scale,
                               init_state=x.init_state.double().numpy())
        assert rel_err(snaps[0, si].cpu().numpy(), rs[0]) <= TOL_BF16, si


@pytest.mark.parametrize("case", CASES[2:7], ids=_id)
def test_f32_prefill_scaled(case):
    x = scaled_inputs("f32", 204, **case)
    out, fin = run_gpu_prefill(x, 16)
    ro, rf = oracle_prefill(x)
    eo, ef = out_err(out, ro), rel_err(fin.cpu().numpy(), rf)
    assert eo <= TOL_F32 and ef <= TOL_F32, (eo, ef)


@pytest.mark.parametrize("io,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
@pytest.mark.parametrize("case", CASES[2:7], ids=_id)
def test_decode_scaled(io, tol, case):
    """T = 4 tokens per sequence through kda_decode, from a scaled state."""
    B, T, H = 4, 4, 2
    x = scaled_inputs(io, 205, lens=[T] * B, H=H, **case)
    shp = (B, T, H, 128)
    pool = x.init_state.clone()
    st = pool.to(DEV)
    out = kda.kda_decode(x.q.view(shp).to(DEV), x.k.view(shp).to(DEV), x.v.view(shp).to(DEV),
                         x.g.view(shp).to(DEV), x.beta.view(B, T, H).to(DEV), x.scale, st)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(x)
    assert out_err(out.reshape(B * T, H, 128), ro) <= tol
    assert rel_err(st.cpu().numpy(), rf) <= tol
