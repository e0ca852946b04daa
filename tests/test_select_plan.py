"""Host-side launch plan of the selection kernels (kvo_plan_select): rows per
thread, CTAs per group, the ticket kernel's grid and the cluster kernel's
cluster size, for the four roofline workloads' shapes on a 152-SM GB300 and
for random shapes (properties every plan must have)."""
import random

import pytest

from sparse_kv_cache_landmark_gb300 import kvo
from sparse_kv_cache_landmark_gb300.kvo import KvoError

SMS = 152


def _ceil(a, b):
    return -(-a // b)


def test_llama_layer_keeps_the_ticket_kernel():
    # 16 requests x 8 KV heads, (32768 - 512) / 32 = 1008 blocks each
    p = kvo.plan_select([1008] * 128, SMS)
    assert p == {"rows_per_thread": 1, "ctas_per_group": 4, "ctas": 512, "cluster_ctas": 0}
    assert kvo.plan_select([1008] * 128, SMS, impl=2)["cluster_ctas"] == 4
    assert kvo.plan_select([1008] * 128, SMS, impl=0)["cluster_ctas"] == 0


def test_wide_budget_layer_uses_clusters_of_eight():
    # 8 x 8 groups of (262144 - 512) / 64 = 4088 blocks: 512-row CTAs fit one wave
    p = kvo.plan_select([4088] * 64, SMS)
    assert p == {"rows_per_thread": 2, "ctas_per_group": 8, "ctas": 512, "cluster_ctas": 8}
    assert kvo.plan_select([4088] * 64, SMS, impl=0)["cluster_ctas"] == 0


def test_long_context_layer_keeps_the_ticket_kernel():
    # 64 x 8 groups of 2032 .. 4080 blocks: 1024-row CTAs, more than one wave
    blocks = [2032 + (2048 * i) // 511 for i in range(512)]
    p = kvo.plan_select(blocks, SMS)
    assert p["rows_per_thread"] == 4 and p["ctas_per_group"] == 4
    assert p["ctas"] == sum(_ceil(c, 1024) for c in blocks) and p["ctas"] > 4 * SMS
    assert p["cluster_ctas"] == 0
    assert kvo.plan_select(blocks, SMS, impl=2)["cluster_ctas"] == 4


def test_fragmentation_layer_cannot_use_clusters():
    # 32 x 8 groups of 65536 - 512 token blocks: 64 CTAs per group
    p = kvo.plan_select([65024] * 256, SMS, impl=2)
    assert p["rows_per_thread"] == 4 and p["ctas_per_group"] == 64 and p["cluster_ctas"] == 0


def test_random_plans_are_consistent():
    rng = random.Random(7)
    for _ in range(300):
        G = rng.randint(1, 600)
        hi = rng.choice([8, 300, 1100, 5000, 40000])
        blocks = [rng.randint(0, hi) for _ in range(G)]
        sms = rng.choice([1, 16, 152])
        plans = {impl: kvo.plan_select(blocks, sms, impl) for impl in (0, 1, 2)}
        p = plans[1]
        rows = 256 * p["rows_per_thread"]
        assert p["rows_per_thread"] in (1, 2, 4)
        assert all(q["rows_per_thread"] == p["rows_per_thread"] for q in plans.values())
        assert p["ctas"] == sum(_ceil(c, rows) for c in blocks)
        assert p["ctas_per_group"] == max(_ceil(c, rows) for c in blocks)
        assert plans[0]["cluster_ctas"] == 0
        S = max(1, p["ctas_per_group"])
        # impl 2: a cluster per group exactly when a group's CTAs fit one
        assert plans[2]["cluster_ctas"] == (S if S <= 8 else 0)
        # impl 1: clusters only where impl 2 would use them and the groups are long
        if p["cluster_ctas"]:
            assert p["cluster_ctas"] == plans[2]["cluster_ctas"] and max(blocks) > 1024
            assert p["ctas"] <= 4 * sms


def test_plan_select_checks_its_arguments():
    for args in (([], SMS, 1), ([10], 0, 1), ([10], SMS, 3), ([10, -1], SMS, 1)):
        with pytest.raises(KvoError):
            kvo.plan_select(*args)
