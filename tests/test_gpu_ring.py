"""GPU tests of the bounded-workspace plans of the bf16 prefill.

kda_prefill runs the fastest plan that its workspace holds: one prepared
block per (chunk, head) when the workspace has room for them all, else the
fused schedule with each chain's blocks in a ring (groups of chains, one
cooperative launch per group), with fewer chains per group when even the
modelled best group does not fit. Every plan runs the same arithmetic on the
same blocks, so the results must agree bit for bit with the full-workspace
plan; that plan is compared with the fp64 oracle here as well.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import inputs
from tests.parity import DEV, TOL_BF16, oracle_prefill, out_err, prefill_schedule, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kimi_delta_attention_rule_gb300 import build as kbuild
    kbuild.build()
    kda.load()


def _lens(name):
    if name == "equal":      # 32 chains: one group, fast plan = fused
        return [1500] * 4, 8
    if name == "many":       # 192 chains: fast plan = split, rings in groups
        return [300] * 6, 32
    if name == "packed":     # 160 ragged chains incl. empty ones, longest first
        gen = np.random.default_rng(17)
        return [int(x) for x in gen.integers(0, 900, size=38)] + [0, 1], 4
    return [5, 0, 129, 1], 2  # "tiny": a ring longer than the sequences


def _sizes(x, H):
    N = x.cu_seqlens.numel() - 1
    T = x.q.shape[0]
    return N, T, H


def _run(x, nbytes, snaps=None, per_head_g=False):
    cu = x.cu_seqlens.to(DEV)
    q = x.q.to(DEV)
    g = x.g.to(DEV)
    if per_head_g:
        g = g[..., 0].contiguous()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out, fin = kda.kda_prefill(q, x.k.to(DEV), x.v.to(DEV), g, x.beta.to(DEV), x.scale,
                               init_state=x.init_state.to(DEV), cu_seqlens=cu, chunk=64,
                               workspace=ws, snapshot_interval=128 if snaps is not None else 0,
                               snapshots=snaps)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    torch.cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("name", ["equal", "many", "packed", "tiny"])
def test_ring_plans_agree_bitwise_with_the_full_workspace(name):
    lens, H = _lens(name)
    x = inputs.prefill_inputs(lens, H=H, io="bf16", seed=301, init="normal")
    N, T, H = _sizes(x, H)
    bf = kda.KDA_BF16
    fast_b = kda.kda_prefill_workspace_size(N, T, H, 128, 64, bf, True)
    ring_b = kda.kda_prefill_workspace_size_ring(N, T, H, 128, 64, bf, True)
    min_b = kda.kda_prefill_workspace_size_min(N, T, H, 128, 64, bf, True)
    assert 0 < min_b <= ring_b and min_b <= fast_b
    ref_out, ref_fin = _run(x, fast_b)
    ro, rf = oracle_prefill(x)
    assert out_err(ref_out, ro) <= TOL_BF16 and rel_err(ref_fin.cpu().numpy(), rf) <= TOL_BF16
    nchains = N * H
    budgets = {"ring": ring_b, "min": min_b, "mid": (ring_b + min_b) // 2}
    for kind, nbytes in budgets.items():
        plan = kda.kda_prefill_plan(N, T, H, 128, 64, bf, True, nbytes)
        if nbytes < fast_b:
            assert plan.schedule == kda.KDA_SCHEDULE_FUSED and plan.ring > 0, kind
            assert plan.groups * plan.group_chains >= nchains > (plan.groups - 1) * plan.group_chains
            assert plan.bytes <= nbytes
        if kind == "min" and nbytes < fast_b:
            assert plan.group_chains == 1
        out, fin = _run(x, nbytes)
        assert torch.equal(out, ref_out), kind
        assert torch.equal(fin, ref_fin), kind


def test_ring_plan_with_snapshots_and_per_head_decay():
    """Snapshots every 128 tokens and one decay per token and head, through
    the ring plan with one chain per group: bit for bit the full-workspace
    results."""
    x = inputs.prefill_inputs([700, 3, 260], H=3, io="bf16", seed=302, init="normal")
    N, T, H = _sizes(x, 3)
    bf = kda.KDA_BF16
    res = []
    for nbytes in (kda.kda_prefill_workspace_size(N, T, H, 128, 64, bf, True),
                   kda.kda_prefill_workspace_size_min(N, T, H, 128, 64, bf, True)):
        snaps = torch.full((N, 6, H, 128, 128), 7.0, dtype=torch.float32, device=DEV)
        out, fin = _run(x, nbytes, snaps=snaps, per_head_g=True)
        res.append((out, fin, snaps))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
    # and the full-workspace result against the oracle (every channel of the
    # decay = channel 0, the per-head decay the kernels read)
    x.g = x.g[..., :1].expand_as(x.g).contiguous()
    ro, rf = oracle_prefill(x)
    assert out_err(res[0][0], ro) <= TOL_BF16
    assert rel_err(res[0][1].cpu().numpy(), rf) <= TOL_BF16


@pytest.mark.parametrize("case", ["h64_t2048", "h80_t600_one_packed", "h40_n2_per_head"])
def test_lead_plan_agrees_with_split_and_oracle(case):
    """Chains on more than a third of the SMs but fewer than the SMs less 16,
    all of one length: the full workspace gets the fused schedule with a lead
    (a launch of producers only, then the chains with the remaining SMs
    preparing the rest). Same arithmetic as K1 then K2: bit for bit the split
    results, and within the bf16 tolerance of the oracle."""
    per_head = case.endswith("per_head")
    if case == "h64_t2048":
        N, L, H, packed = 1, 2048, 64, False
    elif case == "h80_t600_one_packed":
        N, L, H, packed = 1, 600, 80, True   # one packed sequence, ragged tail
    else:
        N, L, H, packed = 2, 777, 40, False  # 80 chains, one decay per head
    x = inputs.prefill_inputs([L] * N, H=H, io="bf16", seed=305, init="normal")
    bf = kda.KDA_BF16
    T_arg = N * L if packed else L
    full = kda.kda_prefill_workspace_size(N, T_arg, H, 128, 64, bf, packed)
    plan = kda.kda_prefill_plan(N, T_arg, H, 128, 64, bf, packed, full)
    assert plan.schedule == kda.KDA_SCHEDULE_FUSED and plan.ring == 0
    assert plan.groups == 1 and plan.group_chains == N * H
    assert 0 < plan.lead_items < N * H * ((L + 63) // 64)
    g = x.g[..., 0].contiguous() if per_head else x.g
    args = (x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g.to(DEV), x.beta.to(DEV), x.scale)
    cu = x.cu_seqlens.to(DEV) if packed else None
    res = {}
    S = L // 256  # snapshots every 256 tokens: 8, 2 and 3 of them
    for mode in (None, "split"):
        with prefill_schedule(mode):
            ws = kda.prefill_workspace(args[0], cu, N=N, T=L, chunk=64)
            snaps = torch.full((N, S, H, 128, 128), 7.0, dtype=torch.float32, device=DEV)
            out, fin = kda.kda_prefill(*args, init_state=x.init_state.to(DEV), cu_seqlens=cu,
                                       chunk=64, workspace=ws, N=N, T=L, snapshot_interval=256,
                                       snapshots=snaps)
            assert kda.kda_workspace_status(ws) == kda.KDA_OK
            torch.cuda.synchronize()
            res[mode] = (out, fin, snaps)
    for a_, b_ in zip(res[None], res["split"]):  # outputs, final states, snapshots
        assert torch.equal(a_, b_)
    assert not torch.equal(res[None][2], torch.full_like(res[None][2], 7.0))
    if per_head:
        x.g = x.g[..., :1].expand_as(x.g).contiguous()
    ro, rf = oracle_prefill(x)
    assert out_err(res[None][0], ro) <= TOL_BF16
    assert rel_err(res[None][1].cpu().numpy(), rf) <= TOL_BF16


def test_workspace_below_the_minimum_is_rejected():
    x = inputs.prefill_inputs([300, 40], H=2, io="bf16", seed=303, init="normal")
    N, T, H = _sizes(x, 2)
    bf = kda.KDA_BF16
    min_b = kda.kda_prefill_workspace_size_min(N, T, H, 128, 64, bf, True)
    with pytest.raises(kda.KDAError) as e:
        kda.kda_prefill_plan(N, T, H, 128, 64, bf, True, min_b - 256)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KDAError) as e:
        _run(x, min_b - 256)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG


def test_split_override_has_no_ring_plan():
    """With the two-kernel schedule forced, the only plan is the full one."""
    bf = kda.KDA_BF16
    with prefill_schedule("split"):
        full = kda.kda_prefill_workspace_size(2, 640, 4, 128, 64, bf)
        assert kda.kda_prefill_workspace_size_min(2, 640, 4, 128, 64, bf) == full
        assert kda.kda_prefill_plan(2, 640, 4, 128, 64, bf, False, full).schedule == \
            kda.KDA_SCHEDULE_SPLIT


@pytest.mark.parametrize("lens", [[0, 0, 0], [0]])
def test_no_tokens_copies_initial_to_final_state(lens):
    """Packed sequences that are all empty: no prepared blocks at all; the
    final states equal the initial ones, bit for bit."""
    H = 2
    gen = torch.Generator().manual_seed(304)
    init = (0.02 * torch.randn(len(lens), H, 128, 128, generator=gen)).to(DEV)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32, device=DEV)
    e = torch.empty((0, H, 128), dtype=torch.bfloat16, device=DEV)
    g = torch.empty((0, H, 128), dtype=torch.float32, device=DEV)
    b = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    ws = kda.prefill_workspace(e, cu, chunk=64)
    assert ws.numel() == kda.kda_prefill_workspace_size_min(len(lens), 0, H, 128, 64,
                                                            kda.KDA_BF16, True)
    out, fin = kda.kda_prefill(e, e, e, g, b, 0.1, init_state=init, cu_seqlens=cu, chunk=64,
                               workspace=ws)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    assert torch.equal(fin, init) and out.numel() == 0


@pytest.mark.slow
@pytest.mark.parametrize("workload", ["append_h96", "varlen64_h32_floor"])
def test_ring_plan_full_size_bitwise(workload):
    """The full-size append (H=96, 65,536 tokens after a 32,768-token prefill)
    and packed varlen (64 sequences) workloads: the ring workspace (tens of MB,
    fused schedule in groups) and the full workspace (GBs, split schedule)
    give the same bits, outputs and final states. (Their parity with the oracle
    is sampled in tests/test_gpu_parity.py.)"""
    w = inputs.WORKLOADS[workload]
    if workload == "append_h96":
        P, Ta, H = w["prior"], w["T"], w["H"]
        x = inputs.prefill_inputs([P + Ta], H=H, io="bf16", seed=w["seed"], device=DEV)
        _, init = kda.kda_prefill(x.q[:P], x.k[:P], x.v[:P], x.g[:P], x.beta[:P], x.scale, chunk=64)
        q, k, v, g, b = (t[P:] for t in (x.q, x.k, x.v, x.g, x.beta))
        cu, N, T = None, 1, Ta
    else:
        lens = inputs.varlen_lengths(w["n_seqs"], w["lo"], w["hi"], seed=w["seed"])
        H = w["H"]
        x = inputs.prefill_inputs(lens, H=H, io="bf16", seed=w["seed"], g_mode="floor",
                                  init="normal", device=DEV)
        q, k, v, g, b, init, cu = x.q, x.k, x.v, x.g, x.beta, x.init_state, x.cu_seqlens
        N, T = len(lens), q.shape[0]
    res = []
    for kind in ("fast", "ring"):
        ws = kda.prefill_workspace(q, cu, N=N, T=T, chunk=64, kind=kind)
        res.append(kda.kda_prefill(q, k, v, g, b, x.scale, init_state=init, cu_seqlens=cu,
                                   chunk=64, workspace=ws, N=N, T=T))
        assert kda.kda_workspace_status(ws) == kda.KDA_OK
        del ws
    torch.cuda.synchronize()
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
