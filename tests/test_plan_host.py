"""The bf16 prefill's workspace-plan selection (host logic), run on the CPU
for given device properties through the test entry point
kda_testing_prefill_plan: which plan a workspace size gets, the sizes of the
three queries, the group model, and the schedule override."""
import ctypes

import pytest

import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import build as kbuild

BLOCK = 74368
C = 64
NSM = 152


@pytest.fixture(scope="module")
def plan():
    kbuild.build()
    lib = kda.load()

    def f(N, T, H, varlen=False, kind=0, budget=0, nsm=NSM, coop=1, force=-1):
        info = kda.PrefillPlanInfo()
        rc = lib.kda_testing_prefill_plan(N, T, H, int(varlen), nsm, coop, force, kind, budget,
                                          ctypes.byref(info))
        return rc, info
    return f


def pad256(x):
    return (x + 255) // 256 * 256


def test_fastest_plan_few_chains_is_fused_one_block_per_chunk(plan):
    rc, p = plan(1, 8192, 32, kind=1)
    assert rc == kda.KDA_OK
    slots = 8192 // C
    assert p.schedule == kda.KDA_SCHEDULE_FUSED and p.ring == 0
    assert p.groups == 1 and p.group_chains == 32
    assert p.bytes == 256 + pad256(slots * 32 * 4) + slots * 32 * BLOCK


def test_fastest_plan_many_chains_is_split(plan):
    """More chains than the SMs less 16 (2 x 96 = 192): K1 then K2."""
    rc, p = plan(2, 65536, 96, kind=1)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT and p.lead_items == 0
    assert p.bytes == 256 + 2 * 1024 * 96 * BLOCK


def _lead_model(nchains, L, nsm=NSM):
    """The schedule model with the paces measured on GB300 (K1 6.1 us per block
    and K2 1.58 us per chunk alone; 6.3 and 2.15 inside the fused kernel)."""
    blocks = nchains * L
    lead = blocks - (nsm - nchains) / 6.3 * L * 2.15
    t_split = blocks * 6.1 / nsm + L * 1.58
    t_lead = max(lead, 0) * 6.3 / nsm + L * 2.15
    return max(lead, 0), t_lead < 0.97 * t_split


def test_fastest_plan_mid_chain_count_has_a_lead(plan):
    """64 chains of 1,024 chunks: the fused schedule with a lead. The rest
    after the lead is what the 88 other SMs prepare while the chains run
    (88 / 6.3 us x 1,024 chunks x 2.15 us ~ 30,750 blocks), so the chains never
    wait for a block that is not in the lead or made in time."""
    rc, p = plan(1, 65536, 64, kind=1)
    blocks = 1024 * 64
    lead, chosen = _lead_model(64, 1024)
    assert chosen
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_FUSED and p.ring == 0
    assert p.groups == 1 and p.group_chains == 64
    assert abs(p.lead_items - lead) <= 1 and 0 < p.lead_items < blocks
    assert p.bytes == 256 + pad256(blocks * 4) + blocks * BLOCK
    # the same count of chains as 2 sequences x 32 heads
    rc, p2 = plan(2, 65536, 32, kind=1)
    assert p2.schedule == kda.KDA_SCHEDULE_FUSED and p2.lead_items == p.lead_items


@pytest.mark.parametrize("N,T,H", [(1, 65536, 96), (1, 65536, 112), (1, 8192, 96), (2, 8192, 40),
                                   (1, 16384, 64), (1, 2048, 64), (2, 777, 40), (1, 600, 80),
                                   (1, 640, 51), (3, 64, 40)])
def test_lead_plan_follows_the_model(plan, N, T, H):
    rc, p = plan(N, T, H, kind=1)
    L = (T + 63) // 64
    lead, chosen = _lead_model(N * H, L)
    assert rc == kda.KDA_OK
    if 3 * N * H <= NSM:
        assert p.schedule == kda.KDA_SCHEDULE_FUSED and p.lead_items == 0
    elif chosen:
        assert p.schedule == kda.KDA_SCHEDULE_FUSED and abs(p.lead_items - lead) <= 1
        assert p.groups == 1 and p.group_chains == N * H
    else:
        assert p.schedule == kda.KDA_SCHEDULE_SPLIT and p.lead_items == 0


def test_lead_only_when_modelled_faster(plan):
    # 128 chains leave 24 producers: the lead plan models no faster than split
    rc, p = plan(1, 65536, 128, kind=1)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT
    # 137 chains: more than the SMs less 16
    rc, p = plan(1, 65536, 137, kind=1)
    assert p.schedule == kda.KDA_SCHEDULE_SPLIT and p.lead_items == 0
    # 64 chains of 32 chunks: lead
    rc, p = plan(1, 2048, 64, kind=1)
    assert p.schedule == kda.KDA_SCHEDULE_FUSED and 0 < p.lead_items < 32 * 64
    # packed sequences of unknown lengths: no lead
    rc, p = plan(2, 65536, 32, varlen=True, kind=1)
    assert p.schedule == kda.KDA_SCHEDULE_SPLIT and p.lead_items == 0
    # one packed sequence: its length is known
    rc, p = plan(1, 65536, 64, varlen=True, kind=1)
    assert p.schedule == kda.KDA_SCHEDULE_FUSED and p.lead_items > 0
    # the override: split, or fused without a lead
    rc, p = plan(1, 65536, 64, kind=1, force=0)
    assert p.schedule == kda.KDA_SCHEDULE_SPLIT and p.lead_items == 0
    rc, p = plan(1, 65536, 64, kind=1, force=1)
    assert p.schedule == kda.KDA_SCHEDULE_FUSED and p.lead_items == 0
    # ring plans have no lead
    rc, p = plan(1, 65536, 64, kind=2)
    assert p.ring == 16 and p.lead_items == 0


def test_ring_plan_does_not_grow_with_the_length(plan):
    sizes = set()
    for T in (4096, 8192, 65536, 1 << 20):
        rc, p = plan(1, T, 32, kind=2)
        assert rc == kda.KDA_OK and p.ring == 16 and p.group_chains == 32 and p.groups == 1
        sizes.add(p.bytes)
    # per chain: its ring flags and its progress counter, a 128-byte line each
    assert sizes == {256 + 32 * 2 * 128 + 32 * 16 * BLOCK}


def test_group_model_many_chains(plan):
    """2,048 chains of equal length: groups of the modelled best size, about
    SMs x 1.83 / (1.83 + 6.3) ~ 34 chains, every chain in exactly one group."""
    rc, p = plan(64, 16384, 32, kind=2)
    assert rc == kda.KDA_OK
    assert 30 <= p.group_chains <= 38
    assert (p.groups - 1) * p.group_chains < 64 * 32 <= p.groups * p.group_chains


def test_smallest_plan_is_one_chain_per_group(plan):
    rc, p = plan(2, 8192, 8, kind=3)
    assert rc == kda.KDA_OK
    assert p.group_chains == 1 and p.groups == 16 and p.ring == 16
    assert p.bytes == 256 + 2 * 128 + 16 * BLOCK


def test_budget_selects_the_plan(plan):
    N, T, H = 1, 8192, 32
    _, fast = plan(N, T, H, kind=1)
    _, ring = plan(N, T, H, kind=2)
    _, small = plan(N, T, H, kind=3)
    assert small.bytes < ring.bytes < fast.bytes
    # the full workspace (or more): the fastest plan
    for b in (fast.bytes, fast.bytes + 12345):
        rc, p = plan(N, T, H, budget=b)
        assert rc == kda.KDA_OK and p.ring == 0 and p.bytes == fast.bytes
    # from the ring size up to just below the full size: the best ring plan
    for b in (ring.bytes, fast.bytes - 1):
        rc, p = plan(N, T, H, budget=b)
        assert rc == kda.KDA_OK and p.ring == 16 and p.group_chains == ring.group_chains
    # below the ring size: fewer chains per group, never above the budget,
    # and more chains with more bytes
    prev = 0
    for b in range(small.bytes, ring.bytes, (ring.bytes - small.bytes) // 7):
        rc, p = plan(N, T, H, budget=b)
        assert rc == kda.KDA_OK and p.ring == 16
        assert 1 <= p.group_chains < ring.group_chains and p.bytes <= b
        assert p.group_chains >= prev
        prev = p.group_chains
    # below the smallest plan: rejected
    rc, _ = plan(N, T, H, budget=small.bytes - 1)
    assert rc == kda.KDA_ERR_INVALID_ARG


def test_packed_sequences_add_the_schedule(plan):
    """With cu_seqlens the workspace also holds the chunk schedule (2 N + 2
    int32), and the slots are T_total / C + N."""
    N, T, H = 5, 1000, 4
    rc, p = plan(N, T, H, varlen=True, kind=1)
    slots = (T + C - 1) // C + N
    base = 256 + pad256((2 * N + 2) * 4)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_FUSED
    assert p.bytes == base + pad256(slots * H * 4) + slots * H * BLOCK


def test_override_and_device_without_cooperative_launch(plan):
    # split forced: no ring plan; the smallest plan is the split one
    rc, p = plan(1, 8192, 32, kind=2, force=kda.KDA_SCHEDULE_SPLIT)
    assert rc == kda.KDA_ERR_INVALID_ARG
    rc, p = plan(1, 8192, 32, kind=3, force=kda.KDA_SCHEDULE_SPLIT)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT
    # fused forced with many chains: fused, in groups
    rc, p = plan(1, 65536, 96, kind=1, force=kda.KDA_SCHEDULE_FUSED)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_FUSED and p.groups > 1
    # no cooperative launches: never fused
    rc, p = plan(1, 8192, 32, kind=1, coop=0)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT
    rc, p = plan(1, 8192, 32, kind=2, coop=0)
    assert rc == kda.KDA_ERR_INVALID_ARG


def test_no_tokens_needs_no_blocks(plan):
    rc, p = plan(3, 0, 2, varlen=True, kind=3)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT
    assert p.bytes == 256 + pad256((2 * 3 + 2) * 4)


def test_invalid_arguments(plan):
    assert plan(1, 64, 2, kind=4)[0] == kda.KDA_ERR_INVALID_ARG
    assert plan(1, 64, 2, force=2)[0] == kda.KDA_ERR_INVALID_ARG
    assert plan(-1, 64, 2)[0] == kda.KDA_ERR_INVALID_ARG
    assert plan(1, 64, 2, kind=1, nsm=0)[0] == kda.KDA_ERR_INVALID_ARG
