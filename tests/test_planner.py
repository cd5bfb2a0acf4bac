"""The placement planner (whead_plan_query), on the host: no GPU is needed.

The planner splits W into 16-row groups, gives each CTA a run of them and places each group in one tier
("Weights That Stay", Fig. 1: each SM keeps its shard of W on chip; Fig. 12: the split of that shard over the
on-chip tiers). The kernel trusts its work lists completely, so these tests check them structurally on many
shapes, and check the placements of the pages' workloads against the ones whead_plan_info reported on a
GB300 (152 SMs, 232,448 bytes of opt-in shared memory per block).
"""
import itertools

import pytest

from speculative_decoding_serial_gb300 import whead as wh

GB300 = dict(sm_count=152, smem_optin=232448)
MARKOV, RECURRENT = 0, 1


@pytest.fixture(scope="module", autouse=True)
def library():
    from speculative_decoding_serial_gb300 import build
    build.build()


# (V, r, kind, max_B, e4m3) -> (grid, groups per CTA, shared, tensor, register, streamed groups per CTA)
MEASURED = [
    ((4096, 64, MARKOV, 1, False), (6, 43, 43, 0, 0, 0)),
    ((151936, 256, MARKOV, 1, False), (152, 63, 27, 32, 4, 0)),
    ((151936, 256, RECURRENT, 1, False), (152, 63, 27, 32, 4, 0)),
    ((151936, 256, MARKOV, 2, False), (152, 63, 27, 32, 4, 0)),
    ((151936, 256, MARKOV, 4, False), (152, 63, 26, 32, 5, 0)),
    ((151936, 256, MARKOV, 8, False), (152, 63, 24, 32, 7, 0)),
    ((151936, 256, MARKOV, 16, False), (152, 63, 20, 32, 0, 11)),
    ((248064, 256, MARKOV, 1, False), (152, 102, 27, 32, 8, 35)),
    ((248064, 256, MARKOV, 4, False), (152, 102, 24, 32, 8, 38)),
    ((151936, 256, MARKOV, 1, True), (152, 63, 53, 10, 0, 0)),
    ((248064, 256, MARKOV, 1, True), (152, 102, 52, 50, 0, 0)),
    ((248064, 256, MARKOV, 4, True), (152, 102, 47, 55, 0, 0)),
]


@pytest.mark.parametrize("shape,want", MEASURED)
def test_placements_of_the_pages_workloads(shape, want):
    V, r, kind, B, e4m3 = shape
    p = wh.plan_query(V, r, kind, max_B=B, B=B, e4m3=e4m3, **GB300)
    got = (p["grid"], p["groups_per_cta"], p["smem_groups"], p["tmem_groups"], p["rf_groups"], p["stream_groups"])
    assert got == want
    assert p["threads"] == 384 and p["sm_count"] == 152


@pytest.mark.parametrize("shape,want", MEASURED)
def test_the_pages_workloads_load_through_the_ring(shape, want):
    """The kernel streams the shard through its shared-memory slots when there is a shared tier and at most 64
    tensor-memory and register groups to stage; every workload of the pages qualifies (the small head has nothing
    to stage; a head that did not qualify would load those groups through registers instead)."""
    V, r, kind, B, e4m3 = shape
    p = wh.plan_query(V, r, kind, max_B=B, B=B, e4m3=e4m3, **GB300)
    staged = p["tmem_groups"] + p["rf_groups"]
    assert p["smem_groups"] >= 1 and staged <= 64


def test_headline_placement_bytes():
    p = wh.plan_query(151936, 256, MARKOV, max_B=1, B=1, **GB300)
    assert p["smem_bytes"] == 227856 and p["tmem_cols"] == 512


def check_plan(p, V, r, kind, e4m3, sm_count, smem_optin):
    kb = r // 128 if e4m3 else r // 64
    G, ng = p["grid"], p["groups_per_cta"]
    ns, nt, nr, nst = p["smem_groups"], p["tmem_groups"], p["rf_groups"], p["stream_groups"]
    assert 1 <= G <= min(sm_count, 256) and 1 <= ng <= 255
    assert G * ng * 16 >= V                      # every row of W belongs to some CTA
    assert ns + nt + nr + nst == ng
    assert p["smem_bytes"] <= smem_optin
    assert ns * kb * 2048 < p["smem_bytes"]       # the shared tier fits beside the rest of the layout
    if nt:
        cols = p["tmem_cols"]
        assert cols in (32, 64, 128, 256, 512) and cols >= ((nt - 1) // 4 + 1) * 16 * kb
    rf_mask = p["rf_warp_mask"]
    assert not rf_mask & 1                        # warp 0 runs the exchange and keeps no register group
    tiers = {}
    tmem_slots = set()
    for w, entries in enumerate(p["work_lists"]):
        assert len(entries) <= 32
        rf_here = [e for e in entries if e[1] == wh.TIER_RF]
        if (rf_mask >> w) & 1:
            assert len(rf_here) == 1              # a register warp holds exactly one group
        else:
            assert not rf_here
        for j, tier, col in entries:
            assert j not in tiers                 # each group is processed by exactly one warp
            tiers[j] = tier
            if tier == wh.TIER_TMEM:
                assert not (rf_mask >> w) & 1
                assert col + 16 * kb <= p["tmem_cols"]
                slot = (w % 4, col)               # the warp's lane quadrant and its first column
                assert slot not in tmem_slots
                tmem_slots.add(slot)
    assert sorted(tiers) == list(range(ng))
    # the tiers are contiguous runs of local groups: shared, tensor memory, registers, streamed
    bounds = [(0, ns, wh.TIER_SMEM), (ns, ns + nt, wh.TIER_TMEM), (ns + nt, ns + nt + nr, wh.TIER_RF),
              (ns + nt + nr, ng, wh.TIER_STREAM)]
    for lo, hi, tier in bounds:
        assert all(tiers[j] == tier for j in range(lo, hi))
    if kind == RECURRENT:
        assert not (rf_mask >> p["ah_warp"]) & 1
    # the shard load's ring: every warp takes its staged (tensor-memory and register) groups out of the shared
    # slots in work-list order, and the slot of staged group k is refilled only after group k - n_smem has left
    # it, so each warp's staged groups must come in increasing order for the ring to always move on
    for entries in p["work_lists"]:
        staged = [j for j, tier, _ in entries if tier in (wh.TIER_TMEM, wh.TIER_RF)]
        assert staged == sorted(staged)


SHAPES = list(itertools.product(
    [16, 1000, 4097, 20011, 151936, 248064],      # V
    [64, 128, 192, 256],                          # r
    [MARKOV, RECURRENT],
    [1, 3, 8, 16],                                # batch size (both plans)
    [(152, 232448), (132, 232448), (80, 101376), (16, 232448)],
))


@pytest.mark.parametrize("V,r,kind,B,dev", SHAPES)
def test_work_lists_are_a_valid_placement(V, r, kind, B, dev):
    sm_count, optin = dev
    try:
        p = wh.plan_query(V, r, kind, max_B=B, B=B, sm_count=sm_count, smem_optin=optin)
    except wh.WheadError as e:
        # only shapes whose shard does not fit even with streaming, or that need more than 255 groups per CTA
        assert e.code == wh.ERR_UNSUPPORTED
        assert (V + 15) // 16 > 255 * min(sm_count, 256) or optin < 110000
        return
    check_plan(p, V, r, kind, False, sm_count, optin)


@pytest.mark.parametrize("V,r,B", list(itertools.product([1000, 151936, 248064], [128, 256], [1, 2, 4])))
def test_e4m3_work_lists_are_a_valid_placement(V, r, B):
    p = wh.plan_query(V, r, MARKOV, max_B=B, B=B, e4m3=True, **GB300)
    check_plan(p, V, r, MARKOV, True, **GB300)


def test_recurrent_slice_goes_to_a_least_loaded_warp():
    # tier costs of the planner: tensor memory 5, registers 5, shared memory 6, streamed 9
    cost = {wh.TIER_TMEM: 5, wh.TIER_RF: 5, wh.TIER_SMEM: 6, wh.TIER_STREAM: 9}
    for V, B in ((151936, 1), (151936, 4), (248064, 1), (20011, 3)):
        p = wh.plan_query(V, 256, RECURRENT, max_B=B, B=B, **GB300)
        load = [sum(cost[t] for _, t, _ in entries) for entries in p["work_lists"]]
        free = [w for w in range(12) if not (p["rf_warp_mask"] >> w) & 1]
        assert p["ah_warp"] in free
        assert load[p["ah_warp"]] == min(load[w] for w in free)


def test_larger_batches_use_the_sixteen_walk_plan():
    small = wh.plan_query(151936, 256, MARKOV, max_B=16, B=8, **GB300)
    large = wh.plan_query(151936, 256, MARKOV, max_B=16, B=16, **GB300)
    assert small["rf_groups"] == 7 and large["rf_groups"] == 0   # register groups only for one n8 half
    assert large["stream_groups"] > 0


@pytest.mark.parametrize("args,code", [
    (dict(V=1000, r=100), wh.ERR_UNSUPPORTED),
    (dict(V=1 << 24, r=64), wh.ERR_UNSUPPORTED),
    (dict(V=1000, r=64, max_B=2, B=3), wh.ERR_INVALID_ARG),
    (dict(V=1000, r=64, max_B=17, B=1), wh.ERR_INVALID_ARG),
    (dict(V=1000, r=64, kind=2), wh.ERR_INVALID_ARG),
    (dict(V=0, r=64), wh.ERR_INVALID_ARG),
    (dict(V=1000, r=64, max_B=8, B=8, e4m3=True), wh.ERR_UNSUPPORTED),
    (dict(V=1000, r=192, e4m3=True), wh.ERR_UNSUPPORTED),
    (dict(V=1000, r=64, sm_count=0), wh.ERR_INVALID_ARG),
])
def test_invalid_and_unsupported_shapes(args, code):
    a = dict(kind=MARKOV, max_B=1, B=1, sm_count=152, smem_optin=232448)
    a.update(args)
    V, r = a.pop("V"), a.pop("r")
    kind = a.pop("kind")
    with pytest.raises(wh.WheadError) as e:
        wh.plan_query(V, r, kind, **a)
    assert e.value.code == code
