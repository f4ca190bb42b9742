"""The C++ planner against the written plan specification, bit for bit (CPU only).

Plans are built with PKA_PLAN_HOST_ONLY, so no GPU is needed.
"""

import random

import pytest

from oracle.plan_spec import plan_spec
from paged_kv_attention_32_gb300 import _lib as L
from paged_kv_attention_32_gb300 import api


def _cases():
    rnd = random.Random(23)
    cases = []
    for _ in range(40):
        B = rnd.randint(1, 48)
        Hkv = rnd.choice([1, 2, 4, 8])
        G = rnd.choice([1, 2, 4, 8])
        ps = rnd.choice([16, 32, 64])
        packed = rnd.random() < 0.5
        ql = [rnd.randint(1, 6) if packed else 1 for _ in range(B)]
        kv = [max(ql[b], rnd.randint(1, 30000)) for b in range(B)]
        if rnd.random() < 0.3:
            kv[rnd.randrange(B)] = 131072
        W = rnd.choice([-1, -1, 0, 7, 4095])
        cases.append(dict(kv=kv, ql=ql, packed=packed, Hq=G * Hkv, Hkv=Hkv, ps=ps, W=W,
                          sms=rnd.choice([8, 132, 152]), waves=rnd.choice([1, 2, 4]),
                          mct=rnd.choice([128, 256, 512]), frozen=rnd.random() < 0.8,
                          causal=rnd.random() < 0.5, mma_min_rows=rnd.choice([4, 8, 16])))
    wide = random.Random(29)
    for _ in range(10):   # more than 64 query rows per KV head (tensor-core kernel, many tiles)
        B = wide.randint(1, 24)
        G = wide.choice([16, 32, 64, 128])
        packed = wide.random() < 0.5
        ql = [wide.randint(1, 6) if packed else 1 for _ in range(B)]
        kv = [max(ql[b], wide.randint(1, 20000)) for b in range(B)]
        cases.append(dict(kv=kv, ql=ql, packed=packed, Hq=G * wide.choice([1, 2]), Hkv=1, ps=16,
                          W=wide.choice([-1, 4095]), sms=152, waves=2, mct=256,
                          frozen=True, causal=True, mma_min_rows=8))
        if wide.random() < 0.5:
            cases[-1]["Hkv"] = 2
            cases[-1]["Hq"] = G * 2
    one_tile = random.Random(31)
    for G, mmr, mct in [(8, 8, 256), (4, 4, 256), (8, 8, 4096), (16, 8, 256)]:
        # the tensor-core kernel with one 16-row tile per request, whole requests by
        # the CTA target: long requests are cut to a share of a resident slot's load
        B = 64
        kv = [one_tile.randint(512, 8192) for _ in range(B)]
        cases.append(dict(kv=kv, ql=[1] * B, packed=False, Hq=G * 8, Hkv=8, ps=16, W=-1,
                          sms=152, waves=2, mct=mct, frozen=True, causal=False,
                          mma_min_rows=mmr))
    # equal lengths: the longest-first order keeps tied requests in request order
    for kv, sms, waves in [([4096] * 40, 152, 2), ([1000, 4096] * 30, 152, 2),
                           ([5000] * 12, 64, 2), ([300, 300, 9000, 9000, 300] * 4, 16, 4)]:
        B = len(kv)
        cases.append(dict(kv=kv, ql=[1] * B, packed=False, Hq=32, Hkv=8, ps=16, W=-1, sms=sms,
                          waves=waves, mct=256, frozen=True, causal=False, mma_min_rows=1))
    return cases


@pytest.mark.parametrize("c", _cases())
def test_native_plan_matches_spec(c):
    ps = c["ps"]
    C = max(-(-n // ps) for n in c["kv"])
    indptr = None
    if c["packed"]:
        indptr = [0]
        for q in c["ql"]:
            indptr.append(indptr[-1] + q)
    plan = api.paged_decode_plan(
        c["kv"], num_qo_heads=c["Hq"], num_kv_heads=c["Hkv"], page_size=ps,
        max_pages_per_seq=C, num_pages=10 ** 6, qo_indptr=indptr, q_len=1,
        causal=c["causal"], window_left=c["W"], freeze_seq_lens=c["frozen"], num_sms=c["sms"],
        split_waves=c["waves"], min_chunk_tokens=c["mct"], mma_min_rows=c["mma_min_rows"],
        host_only=True)
    got = plan.export()
    info = plan.info
    want = plan_spec(c["kv"], c["ql"], c["Hq"], c["Hkv"], 128, ps, c["W"], c["sms"], c["waves"],
                     c["mct"], c["frozen"], c["mma_min_rows"])
    assert got["items"] == [tuple(x) for x in want["items"]]
    assert got["n_chunks"] == want["n_chunks"]
    assert got["part_base"] == want["part_base"]
    assert got["page_lo"] == want["page_lo"]
    assert got["page_hi"] == want["page_hi"]
    assert got["order"] == want["order"]
    assert info["chunk_pages"] == want["chunk_pages"]
    assert info["partial_rows"] == want["partial_rows"]
    assert info["workspace_bytes"] == want["workspace_bytes"]


def test_kernel_choice_follows_rows_per_kv_head():
    import torch

    def kernel(G, L, mma_min_rows=0, dtype=torch.bfloat16):
        p = api.paged_decode_plan([100] * 2, num_qo_heads=G, num_kv_heads=1, page_size=16,
                                  max_pages_per_seq=8, num_pages=100, q_len=L, num_sms=8,
                                  mma_min_rows=mma_min_rows, host_only=True, dtype=dtype)
        return p.info["kernel"], p.info["rows_per_cta"]
    assert kernel(1, 1) == (1, 1)       # default threshold 1 row: the tensor-core kernel
    assert kernel(4, 1) == (1, 4)
    assert kernel(2, 1, dtype=torch.float16) == (1, 2)
    assert kernel(8, 1, mma_min_rows=16) == (0, 8)
    assert kernel(8, 2) == (1, 16)
    assert kernel(4, 3, mma_min_rows=16) == (1, 12)   # 9..15 rows exceed one CUDA-core warp
    assert kernel(4, 1, mma_min_rows=4) == (1, 4)
    assert kernel(4, 1, mma_min_rows=8) == (0, 4)
    assert kernel(2, 1, mma_min_rows=4, dtype=torch.float16) == (0, 2)


def test_plan_update_equals_a_fresh_plan():
    """paged_decode_plan_update rebuilds in place: the same arrays as a new plan for the
    new batch (size, lengths, packed offsets), and a failed update leaves the plan as it was."""
    kw = dict(num_qo_heads=16, num_kv_heads=2, page_size=16, max_pages_per_seq=600,
              num_pages=10 ** 6, num_sms=16, causal=True, window_left=300, host_only=True)
    p = api.paged_decode_plan([100, 3000, 50], qo_indptr=[0, 2, 5, 6], **kw)
    for seq, ind in [([4000, 20, 20, 6000, 7], [0, 1, 4, 5, 8, 9]), ([9000], [0, 3])]:
        p.update(seq, qo_indptr=ind)
        fresh = api.paged_decode_plan(seq, qo_indptr=ind, **kw)
        assert p.export() == fresh.export()
        assert p.info == fresh.info and p.workspace_bytes == fresh.workspace_bytes
    before = p.export()
    with pytest.raises(L.PkaError):
        p.update([5, 5], qo_indptr=[0, 6, 7])   # kv_len < q_len
    assert p.export() == before


def test_planner_tunables_from_the_environment(monkeypatch):
    """A descriptor field left 0 takes PKA_SPLIT_WAVES / PKA_MIN_CHUNK_TOKENS /
    PKA_MMA_MIN_ROWS when set to a positive integer; an explicit field wins; a bad
    value falls back to the default; the plan reports what it used."""
    import torch
    from paged_kv_attention_32_gb300 import api
    seq = torch.tensor([4000, 300, 50], dtype=torch.int32)
    kw = dict(num_qo_heads=8, num_kv_heads=2, page_size=16, max_pages_per_seq=256,
              num_pages=1000, q_len=1, num_sms=8, host_only=True)
    monkeypatch.setenv("PKA_SPLIT_WAVES", "5")
    monkeypatch.setenv("PKA_MIN_CHUNK_TOKENS", "512")
    monkeypatch.setenv("PKA_MMA_MIN_ROWS", "8")
    info = api.paged_decode_plan(seq, **kw).info
    assert (info["split_waves"], info["min_chunk_tokens"]) == (5, 512)
    assert info["kernel"] == 0                      # group of 4 rows < 8: CUDA-core kernel
    info = api.paged_decode_plan(seq, split_waves=3, **kw).info
    assert info["split_waves"] == 3
    monkeypatch.setenv("PKA_SPLIT_WAVES", "abc")
    monkeypatch.setenv("PKA_MIN_CHUNK_TOKENS", "0")
    monkeypatch.delenv("PKA_MMA_MIN_ROWS")
    info = api.paged_decode_plan(seq, **kw).info
    assert (info["split_waves"], info["min_chunk_tokens"], info["kernel"]) == (2, 256, 1)


def test_an_empty_batch_is_rejected_by_name():
    """A decode plan needs at least one request; an empty length array is reported as
    such (not as a NULL pointer), and nothing is built."""
    with pytest.raises(L.PkaError, match="batch_size"):
        api.paged_decode_plan([], num_qo_heads=8, num_kv_heads=2, page_size=16,
                              max_pages_per_seq=4, num_pages=100, num_sms=8, host_only=True)
