"""Pins for the plan definition: properties that any valid plan must have."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("seed,grouped", [(s, g) for s in range(8) for g in (False, True)])
def test_pieces_partition_every_page_in_logical_order(seed, grouped):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    bs = int(rng.choice([16, 32, 64]))
    L = rng.integers(0, 3000, B)
    Hkv = int(rng.integers(1, 5))
    RB = int(rng.integers(1, 5))
    G = RB if grouped else 1
    W = int(rng.integers(1, 400)) * G
    mbps = int(-(-L.max() // bs)) + 1
    pl = oracle.plan(L, bs=bs, Hkv=Hkv, max_context_len=int(L.max()), max_blocks_per_seq=mbps,
                     row_blocks=RB, warps=W, group_size=G)
    X = Hkv * RB
    assert pl["positions"] == X // G * int(pl["pages"].sum())
    # warp shares are contiguous, cover [0, N) and differ in size by at most one
    st = pl["warp_starts"]
    assert st[0] == 0 and st[-1] == pl["positions"]
    sizes = np.diff(st)
    assert sizes.min() >= 0 and sizes.max() - sizes.min() <= 1
    # every page of every segment lies in exactly one piece; pieces of a
    # segment come in ascending warp order and are consecutive
    by_seg = {}
    for pc in pl["pieces"]:
        by_seg.setdefault(pc["segment"], []).append(pc)
    for b in range(B):
        for q in range(X):
            s = b * X + q
            got = by_seg.get(s, [])
            if pl["pages"][b] == 0:
                assert not got
                continue
            assert [p["warp"] for p in got] == sorted(p["warp"] for p in got)
            pos = 0
            for p in got:
                assert p["pages"][0] == pos
                pos = p["pages"][1]
            assert pos == pl["pages"][b]
            assert (len(got) == 1) == got[0]["complete"]
            # a grouped worker g*G + i only ever takes row block i
            assert all(p["warp"] % G == q % G for p in got)
    slots = [p["slot"] for p in pl["pieces"]]
    assert len(set(slots)) == len(slots) and max(slots, default=0) < pl["slots"]


def test_grouped_workers_of_a_group_share_their_pages():
    # the G workers of a group take the same page runs, one row block each
    pl = oracle.plan([300, 5, 900], bs=64, Hkv=1, max_context_len=900, max_blocks_per_seq=15,
                     row_blocks=4, warps=12, group_size=4)
    runs = {}
    for p in pl["pieces"]:
        runs.setdefault((p["warp"] // 4, p["segment"] // 4), set()).add((p["pages"], p["segment"] % 4))
    for key, v in runs.items():
        assert {rb for _, rb in v} == {0, 1, 2, 3}
        assert len({pg for pg, _ in v}) == 1
    assert pl["slots"] == (3 * 1 + 3) * 4


def test_plan_flags_invalid_requests():
    pl = oracle.plan([10, -1, 300, 40], bs=16, Hkv=2, max_context_len=256, max_blocks_per_seq=3, warps=5)
    assert pl["flags"].tolist() == [0, 1, 1, 0]
    assert pl["pages"].tolist() == [1, 0, 0, 3]
    assert pl["prefix"].tolist() == [0, 1, 1, 1]
    assert pl["total_pages"] == 4


def test_plan_depends_only_on_lengths():
    L = [100, 7, 4000]
    a = oracle.plan(L, bs=16, Hkv=4, max_context_len=4000, max_blocks_per_seq=300, warps=64)
    b = oracle.plan(list(L), bs=16, Hkv=4, max_context_len=4000, max_blocks_per_seq=300, warps=64)
    assert a["pieces"] == b["pieces"]
    one = oracle.plan(L, bs=16, Hkv=1, max_context_len=4000, max_blocks_per_seq=300, warps=1)
    assert all(p["complete"] for p in one["pieces"]) and len(one["pieces"]) == 3


def test_merged_work_pages_keep_the_table_limit_in_blocks():
    # work pages of two 16-token blocks: pages count 32 tokens, but a request is
    # valid only while its 16-token blocks fit the table row (5 here); 90 tokens
    # need 6 blocks although ceil(90 / 32) = 3 pages would fit ceil(5 / 2)
    pl = oracle.plan([90, 80, 17, 0], bs=32, block_size=16, Hkv=1, max_context_len=1000, max_blocks_per_seq=5)
    assert pl["flags"].tolist() == [1, 0, 0, 0]
    assert pl["pages"].tolist() == [0, 3, 1, 0]
    assert pl["prefix"].tolist() == [0, 0, 3, 4]
    same = oracle.plan([90, 80, 17, 0], bs=16, Hkv=1, max_context_len=1000, max_blocks_per_seq=5)
    assert same["flags"].tolist() == pl["flags"].tolist()
