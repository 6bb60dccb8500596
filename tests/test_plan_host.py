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
    rc, p = plan(1, 65536, 96, kind=1)
    assert rc == kda.KDA_OK and p.schedule == kda.KDA_SCHEDULE_SPLIT
    assert p.bytes == 256 + 1024 * 96 * BLOCK


def test_ring_plan_does_not_grow_with_the_length(plan):
    sizes = set()
    for T in (4096, 8192, 65536, 1 << 20):
        rc, p = plan(1, T, 32, kind=2)
        assert rc == kda.KDA_OK and p.ring == 16 and p.group_chains == 32 and p.groups == 1
        sizes.add(p.bytes)
    assert sizes == {256 + pad256(32 * 17 * 4) + 32 * 16 * BLOCK}


def test_group_model_many_chains(plan):
    """2,048 chains of equal length: groups of the modelled best size, about
    SMs x 1.6 / (1.6 + 6.8) ~ 29 chains, every chain in exactly one group."""
    rc, p = plan(64, 16384, 32, kind=2)
    assert rc == kda.KDA_OK
    assert 25 <= p.group_chains <= 33
    assert (p.groups - 1) * p.group_chains < 64 * 32 <= p.groups * p.group_chains


def test_smallest_plan_is_one_chain_per_group(plan):
    rc, p = plan(2, 8192, 8, kind=3)
    assert rc == kda.KDA_OK
    assert p.group_chains == 1 and p.groups == 16 and p.ring == 16
    assert p.bytes == 256 + 256 + 16 * BLOCK


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
