"""Pins for the plan definition: properties that any valid plan must have."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("seed", range(6))
def test_plan_covers_every_page_once_in_logical_order(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    bs = int(rng.choice([16, 32, 64]))
    L = rng.integers(0, 5000, B)
    Hkv = int(rng.integers(1, 9))
    mbps = int(-(-L.max() // bs)) + 1
    pl = oracle.plan(L, bs=bs, Hkv=Hkv, max_context_len=int(L.max()), max_blocks_per_seq=mbps,
                     target_ctas=int(rng.integers(1, 3000)), min_pages=int(rng.integers(1, 40)))
    assert pl["num_units"] == len(pl["units"]) == int(pl["splits"].sum()) * Hkv
    seen = {}
    for u, (b, h, s, p0, p1) in enumerate(pl["units"]):
        assert u == pl["offsets"][b] * Hkv + h * pl["splits"][b] + s
        assert 0 <= p0 <= p1 <= pl["pages"][b]
        seen.setdefault((b, h), []).append((s, p0, p1))
    for b in range(B):
        for h in range(Hkv):
            parts = sorted(seen[(b, h)])
            assert [p[0] for p in parts] == list(range(pl["splits"][b]))
            # consecutive, ascending, covering [0, P_b)
            pos = 0
            for _, p0, p1 in parts:
                assert p0 == pos
                pos = p1
            assert pos == -(-L[b] // bs)
    # every request gets at least one unit, and no unit is empty unless its
    # request has no pages
    assert all(p1 > p0 or pl["pages"][b] == 0 for (b, h, s, p0, p1) in pl["units"])


def test_plan_flags_invalid_requests():
    pl = oracle.plan([10, -1, 300, 40], bs=16, Hkv=2, max_context_len=256, max_blocks_per_seq=3,
                     target_ctas=100, min_pages=1)
    assert pl["flags"].tolist() == [0, 1, 1, 0]
    assert pl["pages"].tolist() == [1, 0, 0, 3]
    assert pl["splits"].tolist()[1:3] == [1, 1]


def test_plan_depends_only_on_lengths():
    L = [100, 7, 4000]
    a = oracle.plan(L, bs=16, Hkv=4, max_context_len=4000, max_blocks_per_seq=300, target_ctas=64, min_pages=2)
    b = oracle.plan(list(L), bs=16, Hkv=4, max_context_len=4000, max_blocks_per_seq=300, target_ctas=64, min_pages=2)
    assert a["units"] == b["units"]
    forced = oracle.plan(L, bs=16, Hkv=1, max_context_len=4000, max_blocks_per_seq=300,
                         target_ctas=64, min_pages=2, forced_pages=1)
    assert forced["splits"].tolist() == [7, 1, 250]
