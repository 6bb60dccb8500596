"""Shared helpers of the GPU parity tests: the error metric against the fp64
oracle and the calls that run one prefill on each side.

Error metric (per compared tensor): max |gpu - oracle| / rms(oracle), with
bars 2e-2 for bf16 I/O and 1e-4 for fp32 I/O (outputs and final states).
A bf16 output cannot be closer to the exact value than half a bf16 spacing,
and on these heavy-tailed outputs (max|o| / rms(o) ~ 13) that storage
rounding alone is ~2.6e-2 of the RMS; so for bf16-stored tensors the bar
applies to the error in excess of half a bf16 spacing at the oracle value:
    max_i max(0, |gpu_i - ref_i| - ulp_bf16(ref_i) / 2) / rms(ref).
fp32 tensors (final states, fp32 I/O) use the plain metric.
"""
import contextlib

import numpy as np
import torch

import oracle
import kimi_delta_attention_rule_gb300 as kda

TOL_BF16 = 2e-2
TOL_F32 = 1e-4
DEV = "cuda:0"


def bf16_half_spacing(ref):
    """Half the distance between adjacent bf16 numbers at |ref| (8-bit
    significand: spacing 2^(e - 7) in the binade [2^e, 2^(e+1)))."""
    _, e = np.frexp(np.abs(ref))
    e = np.maximum(e, -125)  # bf16 subnormal spacing floor
    return np.ldexp(1.0, e - 9)


def rel_err(got, ref, stored_bf16=False, ulps=0.5):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    diff = np.abs(got - ref)
    if stored_bf16:
        diff = np.maximum(diff - 2 * ulps * bf16_half_spacing(ref), 0.0)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    if rms == 0.0:
        return float(np.max(diff))
    return float(np.max(diff)) / rms


def out_err(out, ref):
    """Error of an output tensor against the oracle (storage-aware)."""
    return rel_err(np32(out), ref, stored_bf16=(out.dtype == torch.bfloat16))


def np32(t):
    return t.detach().float().cpu().numpy()


def run_gpu_prefill(x, chunk, with_init=True, ws_kind="fast"):
    """One kda_prefill call on x with a workspace of the given kind ("fast",
    "ring", "min": the plan follows from its size)."""
    cu = x.cu_seqlens.to(DEV) if x.cu_seqlens is not None else None
    init = x.init_state.to(DEV) if (with_init and x.init_state is not None) else None
    q = x.q.to(DEV)
    ws = kda.prefill_workspace(q, cu, chunk=chunk, kind=ws_kind)
    out, fin = kda.kda_prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), x.g.to(DEV),
                               x.beta.to(DEV), x.scale, init_state=init, cu_seqlens=cu,
                               chunk=chunk, workspace=ws)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    torch.cuda.synchronize()
    return out, fin


def oracle_prefill(x, with_init=True):
    init = x.init_state.double().numpy() if (with_init and x.init_state is not None) else None
    return oracle.prefill(np32(x.q), np32(x.k), np32(x.v), np32(x.g), np32(x.beta), x.scale,
                          init_state=init, cu_seqlens=x.cu_seqlens.numpy())


def check_prefill(x, chunk, tol, with_init=True):
    out, fin = run_gpu_prefill(x, chunk, with_init)
    ro, rf = oracle_prefill(x, with_init)
    eo, ef = out_err(out, ro), rel_err(fin.cpu().numpy(), rf)
    assert eo <= tol and ef <= tol, (eo, ef)
    return eo, ef


@contextlib.contextmanager
def prefill_schedule(mode):
    """Force the bf16 prefill schedule ("split", "fused" or None for the
    automatic choice) for the calls inside the block. ("ring": the automatic
    choice; the caller passes a ring-sized workspace.)"""
    code = {None: -1, "ring": -1, "split": kda.KDA_SCHEDULE_SPLIT,
            "fused": kda.KDA_SCHEDULE_FUSED}[mode]
    prev = kda.kda_prefill_set_schedule(code)
    try:
        yield
    finally:
        kda.kda_prefill_set_schedule(prev)
