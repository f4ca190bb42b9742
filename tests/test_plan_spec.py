"""Invariants of the written split-KV plan specification (oracle/plan_spec.py).

The chunking constants are design choices with no counterpart on the pages;
these tests pin the specification against the properties it promises.
"""

import math
import random

import pytest

from oracle.plan_spec import plan_spec


def _cases():
    rnd = random.Random(11)
    out = []
    for _ in range(60):
        B = rnd.randint(1, 40)
        Hkv = rnd.choice([1, 2, 4, 8])
        ps = rnd.choice([16, 32])
        ql = [rnd.randint(1, 6) for _ in range(B)]
        kv = [max(ql[b], rnd.randint(1, 20000)) for b in range(B)]
        if rnd.random() < 0.3:
            kv[0] = 131072
        W = rnd.choice([-1, -1, 0, 5, 4095])
        out.append((kv, ql, 8 * Hkv, Hkv, ps, W, rnd.choice([4, 152]), rnd.choice([1, 2, 4]),
                    256, rnd.random() < 0.8))
    return out


@pytest.mark.parametrize("case", _cases())
def test_plan_covers_every_visited_page_once(case):
    kv, ql, Hq, Hkv, ps, W, sms, waves, mct, frozen = case
    p = plan_spec(kv, ql, Hq, Hkv, 128, ps, W, sms, waves, mct, frozen)
    B = len(kv)
    covered = {}
    for (b, hk, ci, lo, hi) in p["items"]:
        assert lo < hi
        covered.setdefault((b, hk), []).append((ci, lo, hi))
    for b in range(B):
        n, L = kv[b], ql[b]
        first_key = max(0, n - L - W) if (W >= 0 and frozen) else 0
        want = list(range(first_key // ps, math.ceil(n / ps)))
        for hk in range(Hkv):
            ch = sorted(covered[(b, hk)])
            assert [c for c, _, _ in ch] == list(range(p["n_chunks"][b]))
            pages = [pg for _, lo, hi in ch for pg in range(lo, hi)]
            assert pages == want
            assert all(hi - lo <= p["chunk_pages"] for _, lo, hi in ch)


@pytest.mark.parametrize("case", _cases())
def test_plan_chunk_is_minimal_under_the_target(case):
    kv, ql, Hq, Hkv, ps, W, sms, waves, mct, frozen = case
    p = plan_spec(kv, ql, Hq, Hkv, 128, ps, W, sms, waves, mct, frozen)
    B, T = len(kv), waves * sms
    npg = [hi - lo for lo, hi in zip(p["page_lo"], p["page_hi"])]
    c = p["chunk_pages"]
    c_min = math.ceil(mct / ps)
    G = Hq // Hkv
    mma = G * max(ql) >= 8
    tiles = [math.ceil(G * q / 16) if mma else 1 for q in ql]
    ctas = [Hkv * t for t in tiles]
    if sum(ctas) >= T:
        # no uniform split: only requests past the first wave of resident CTAs are
        # cut, into at most k = slots // (their CTAs) chunks of >= min(c_min, np) pages
        assert c == max(npg)
        slots = (3 if mma else 2) * sms
        order, first, acc = p["order"], 0, 0
        while first < B and acc + ctas[order[first]] <= slots:
            acc += ctas[order[first]]
            first += 1
        tail = order[first:]
        rest = sum(ctas[b] for b in tail)
        k = slots // rest if rest else 1
        assert all(p["n_chunks"][b] == 1 for b in order[:first])
        for b in tail:
            n = p["n_chunks"][b]
            if k <= 1:
                assert n == 1
                continue
            assert 1 <= n <= k
            lens = [hi - lo for (bb, hk, ci, lo, hi) in p["items"] if bb == b and hk == 0]
            assert all(x >= min(c_min, npg[b]) for x in lens[:-1])
            if n < k:   # fewer pages than k, or the c_min floor bound the chunk
                assert npg[b] < k or math.ceil(npg[b] / k) < min(c_min, npg[b])
        return
    ctas_at = lambda cc: Hkv * sum(t * math.ceil(x / cc) for t, x in zip(tiles, npg))
    assert Hkv * sum(math.ceil(x / c) for x in npg) == len(p["items"]) and ctas_at(c) <= T
    c_lo = min(c_min, max(npg))
    assert c >= c_lo
    if c > c_lo:
        assert ctas_at(c - 1) > T


@pytest.mark.parametrize("case", _cases()[:20])
def test_plan_order_partials_and_workspace(case):
    kv, ql, Hq, Hkv, ps, W, sms, waves, mct, frozen = case
    p = plan_spec(kv, ql, Hq, Hkv, 128, ps, W, sms, waves, mct, frozen)
    npg = [hi - lo for lo, hi in zip(p["page_lo"], p["page_hi"])]
    seq = [it[0] for it in p["items"]]
    firsts = list(dict.fromkeys(seq))
    assert firsts == p["order"]
    assert all(npg[a] >= npg[b] for a, b in zip(firsts, firsts[1:]))
    rows = 0
    for b in range(len(kv)):
        if p["n_chunks"][b] > 1:
            assert p["part_base"][b] == rows
            rows += p["n_chunks"][b] * ql[b] * Hq
        else:
            assert p["part_base"][b] == -1
    assert p["partial_rows"] == rows
    if rows:
        assert p["workspace_bytes"] == math.ceil(rows * 128 * 4 / 256) * 256 + rows * 4
    else:
        assert p["workspace_bytes"] == 0


def test_plan_tail_requests_are_cut_into_one_round():
    """32 requests of ~4096 keys with 1-3 tiles: the longest-first prefix fills the
    3 x 152 resident slots, the rest is cut into 456 // (its CTAs) chunks each."""
    ql = [1 + (b % 6) for b in range(32)]
    kv = [4096 + 16 * (31 - b) for b in range(32)]
    p = plan_spec(kv, ql, 64, 8, 128, 16, 4095, 152, 2, 256)
    ctas = [8 * math.ceil(8 * q / 16) for q in ql]
    acc, first = 0, 0
    for b in p["order"]:
        if acc + ctas[b] > 456:
            break
        acc += ctas[b]
        first += 1
    tail = p["order"][first:]
    k = 456 // sum(ctas[b] for b in tail)
    assert k > 1 and all(p["n_chunks"][b] == k for b in tail)
    assert all(p["n_chunks"][b] == 1 for b in p["order"][:first])


def test_plan_skewed_long_request_is_split():
    kv = [131072] + [2048] * 15
    p = plan_spec(kv, [1] * 16, 64, 8, 128, 32, -1, 152, 2, 256)
    assert p["n_chunks"][0] > 1 and p["order"][0] == 0
    assert len(p["items"]) <= 2 * 152


def test_plan_single_tile_requests_are_cut_to_a_share_of_the_slot_load():
    """Tensor-core kernel, one 16-row tile per request, whole requests by the CTA target
    (64 x 8 CTAs >= 2 x 152): every chunk holds at most 3/5 of a resident slot's average
    load (A = Hkv * sum np / (3 * 152) pages), rounded up to whole parts, and a request
    of several tiles (q_len 3) is left whole by this rule."""
    kv = [512 + 120 * b for b in range(64)]
    p = plan_spec(kv, [1] * 64, 64, 8, 128, 16, -1, 152, 2, 256)
    npg = [math.ceil(x / 16) for x in kv]
    A = 8 * sum(npg) / (3 * 152)
    long = [b for b, n in enumerate(npg) if n > 0.6 * A]
    assert long
    for b in long:
        parts = math.ceil(npg[b] / (0.6 * A))
        assert p["n_chunks"][b] == parts and parts >= 2
    assert max(hi - lo for (_, _, _, lo, hi) in p["items"]) <= math.ceil(0.6 * A)
    # (the shortest requests are cut by the tail rule, which this rule leaves alone)
    p3 = plan_spec(kv, [3] * 64, 64, 8, 128, 16, -1, 152, 2, 256)   # 24 rows: 2 tiles
    assert all(p3["n_chunks"][b] == 1 for b in long)
