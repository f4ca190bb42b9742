"""Paged decode on the GPU against the fp64 oracle (element by element)."""

import numpy as np
import pytest
import torch

from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

from helpers import assert_close, oracle_decode, row_mask, run_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"

# Oracle-sized copies of the four decode workloads: same structure (GQA group,
# page size, q_len mix, causal/window/sinks), fewer and shorter requests, still
# spanning many 16-token units and a ragged last page.
SMALL = {
    "tiny": wl.TINY_DECODE,
    "llama3_8b": wl.shrink(wl.LLAMA3_8B_DECODE, batch=6, kv_len_range=(512, 2100),
                           pool_pages=1000, table_width=160, return_lse=True),
    "skewed": wl.shrink(wl.SKEWED_DECODE, batch=5, fixed_first_kv_len=12000,
                        kv_len_range=(1024, 4096), table_width=400),
    "spec": wl.shrink(wl.SPEC_DECODE, batch=6, kv_len_range=(2048, 6000), table_width=400),
}


# decode kernel of a test case: the default (the tensor-core kernel), or the CUDA-core one
# (kept for groups of up to 8 rows per KV head when mma_min_rows is set above them)
KERNELS = {"default": {}, "cuda_core": dict(mma_min_rows=16)}


@pytest.mark.parametrize("name,kernel", [(n, k) for n in SMALL for k in KERNELS
                                         if not (n == "spec" and k == "cuda_core")])
@pytest.mark.parametrize("seed", [0, 1])
def test_decode_matches_oracle(name, seed, kernel):
    inp = wl.make_decode_inputs(SMALL[name], seed=seed, device=DEV)
    out, lse, plan = run_decode(inp, **KERNELS[kernel])
    assert plan.info["kernel"] == (0 if kernel == "cuda_core" else 1)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", ["llama3_8b", "skewed"])
def test_decode_split_kv_path(name, kernel):
    """Few SMs in the plan force a split of the long requests: partials merged in the run."""
    inp = wl.make_decode_inputs(SMALL[name], seed=3, device=DEV)
    out, lse, plan = run_decode(inp, num_sms=32, split_waves=2, min_chunk_tokens=128,
                                **KERNELS[kernel])
    assert plan.info["num_split"] > 0
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("name,sms,kernel", [
    ("spec", 148, "default"), ("skewed", 148, "default"), ("skewed", 48, "default"),
    ("llama3_8b", 64, "default"), ("llama3_8b", 64, "cuda_core"),
    ("llama3_8b", 1024, "cuda_core")])
def test_decode_split_merge_by_the_last_chunk(name, sms, kernel):
    """Split partials are merged inside the decode kernels: the chunk CTA of a (request,
    KV head, tile) group that counts last combines the group's rows (spec: <= 3 chunks
    over packed causal rows, three tiles; skewed: 19 chunks, merged with 16 threads per
    row, or 6, with 8; llama3_8b: both kernels, and the CUDA-core one with up to 17 chunks
    at a planned 1024 SMs).  Run twice, so that the counters left by the first run (reset to
    zero by each group's last CTA) serve the second."""
    inp = wl.make_decode_inputs(SMALL[name], seed=5, device=DEV)
    from helpers import decode_plan_for
    plan = decode_plan_for(inp, num_sms=sms, split_waves=2, min_chunk_tokens=128,
                           **KERNELS[kernel])
    ex = plan.export()
    assert max(ex["n_chunks"]) > 1
    ref_o, ref_l = oracle_decode(inp)
    for _ in range(2):
        out, lse, _ = run_decode(inp, plan=plan)
        assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "skewed"])
def test_decode_both_kernels_on_narrow_groups(name, kernel):
    """4- and 8-row groups on either kernel (the tensor-core one pads the rows to 16)."""
    inp = wl.make_decode_inputs(SMALL[name], seed=4, device=DEV)
    out, lse, plan = run_decode(inp, **KERNELS[kernel])
    assert plan.info["kernel"] == (0 if kernel == "cuda_core" else 1)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("G,L,causal,W,sinks,kernel", [
    (4, 2, True, -1, False, "cuda_core"),   # 8 rows, causal multi-token
    (4, 2, True, -1, False, "default"),
    (2, 3, False, 40, True, "cuda_core"),   # dense mask with a window, sinks
    (2, 3, False, 40, True, "default"),
    (1, 1, False, 0, True, "cuda_core"),    # window 0: only the diagonal key
    (1, 1, False, 0, True, "default"),
    (8, 8, True, 100, True, "default"),     # 64 rows, four m16 tiles
    (4, 8, True, 33, True, "default"),      # 32 rows, two m16 tiles
    (8, 3, False, -1, False, "default"),    # 24 rows, dense mask
    (4, 3, True, 17, False, "cuda_core"),   # 12 rows: the tensor-core kernel whatever is asked
])
def test_decode_masks_and_groups(G, L, causal, W, sinks, kernel):
    w = wl.DecodeWorkload(name="masks", batch=5, num_qo_heads=2 * G, num_kv_heads=2,
                          head_dim=128, page_size=16, kv_len_range=(L, 700), q_len_range=(L, L),
                          causal=causal, window_left=W, sinks=sinks)
    inp = wl.make_decode_inputs(w, seed=5, device=DEV)
    out, lse, plan = run_decode(inp, **KERNELS[kernel])
    assert plan.info["kernel"] == (0 if kernel == "cuda_core" and G * L <= 8 else 1)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("G,L,packed,split", [
    (8, 3, False, False),   # 24 rows: two tiles, the second half empty
    (8, 6, True, True),     # up to 48 rows, requests with 1..3 live tiles, split chunks
    (8, 8, False, True),    # 64 rows: four tiles
    (4, 5, True, False),    # 20 rows, packed lengths 1..5
])
def test_decode_wide_groups(G, L, packed, split):
    """17-64 rows per KV head: one mma CTA per live 16-row tile of every item."""
    w = wl.DecodeWorkload(name="wide", batch=7, num_qo_heads=2 * G, num_kv_heads=2, head_dim=128,
                          page_size=16, kv_len_range=(L, 1500),
                          q_len_range=(1, L) if packed else (L, L), packed_q=packed, causal=True,
                          window_left=300 if split else -1, sinks=True)
    inp = wl.make_decode_inputs(w, seed=12, device=DEV)
    kw = dict(num_sms=48, split_waves=2, min_chunk_tokens=128) if split else {}
    out, lse, plan = run_decode(inp, **kw)
    assert plan.info["kernel"] == 1
    if split:
        assert plan.info["num_split"] > 0
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("G,L,packed,split", [
    (3, 7, False, False),   # 21 rows: a 16-row tile and a 5-row tail (tokens 5-6 of the request)
    (7, 3, False, True),    # 21 rows, split chunks
    (6, 4, False, False),   # 24 rows: a tail of exactly 8
    (5, 5, False, False),   # 25 rows: a 9-row tail on the 16-row step
    (1, 9, False, True),    # 9 rows in one tile
    (3, 2, False, False),   # 6 rows: the transposed step alone
    (5, 7, True, True),     # packed 1..7 tokens: 5..35 rows, tails of every size
])
def test_decode_tile_tails(G, L, packed, split):
    """Tiles whose live rows cross token boundaries at every tail size: a tile of at most
    8 live rows takes the transposed step (the rows' key ranges and their q rows offset by
    the tile), a wider one the 16-row step."""
    w = wl.DecodeWorkload(name="tails", batch=6, num_qo_heads=2 * G, num_kv_heads=2,
                          head_dim=128, page_size=16, kv_len_range=(L, 1200),
                          q_len_range=(1, L) if packed else (L, L), packed_q=packed, causal=True,
                          window_left=200 if split else 37, sinks=True)
    inp = wl.make_decode_inputs(w, seed=31, device=DEV)
    kw = dict(num_sms=40, split_waves=2, min_chunk_tokens=128) if split else {}
    out, lse, plan = run_decode(inp, **kw)
    if split:
        assert plan.info["num_split"] > 0
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("Hq,Hkv,L,packed,split", [
    (128, 1, 1, False, False),   # MQA, 128 heads: 8 tiles per item
    (128, 1, 1, False, True),    #   ... with split chunks and the merge
    (64, 1, 6, True, True),      # 64 heads x packed q_len 1..6: up to 384 rows, 24 tiles
    (16, 2, 16, False, False),   # G = 8 x q_len 16: 128 rows, causal
])
def test_decode_more_than_64_rows_per_kv_head(Hq, Hkv, L, packed, split):
    """Groups wider than four 16-row tiles (cudnn_batch_decode_with_kv_cache allows any
    num_heads_qo >= num_heads_kv and any q_len_per_req): one mma CTA per tile."""
    w = wl.DecodeWorkload(name="wider", batch=4, num_qo_heads=Hq, num_kv_heads=Hkv,
                          head_dim=128, page_size=16, kv_len_range=(L, 1300),
                          q_len_range=(1, L) if packed else (L, L), packed_q=packed,
                          causal=L > 1, window_left=400 if split else -1, sinks=split)
    inp = wl.make_decode_inputs(w, seed=22, device=DEV)
    kw = dict(num_sms=64, split_waves=2, min_chunk_tokens=128) if split else {}
    out, lse, plan = run_decode(inp, **kw)
    assert plan.info["kernel"] == 1 and plan.info["rows_per_cta"] > 64
    if split:
        assert plan.info["num_split"] > 0
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("in_dtype,out_dtype", [
    (torch.float16, None), (torch.float16, torch.float32), (torch.bfloat16, torch.float32),
    (torch.bfloat16, torch.float16)])
@pytest.mark.parametrize("name,mma", [("llama3_8b", 16), ("llama3_8b", 0), ("spec", 0),
                                      ("skewed", 16)])
def test_decode_input_and_output_dtypes(in_dtype, out_dtype, name, mma):
    """fp16 q/K/V (cudnn_batch_decode_with_kv_cache takes float16 or bfloat16) and
    out_dtype bf16 / f16 / fp32 (batch_decode_with_paged_kv_cache, out_dtype), on the
    CUDA-core kernel (4 and 8 rows: mma_min_rows 16), the tensor-core kernel (the
    default) and the split + merge path."""
    inp = wl.make_decode_inputs(SMALL[name], seed=14, device=DEV, dtype=in_dtype)
    kw = dict(out_dtype=out_dtype, num_sms=32, split_waves=2, min_chunk_tokens=128)
    if mma:
        kw["mma_min_rows"] = mma
    out, lse, plan = run_decode(inp, **kw)
    assert out.dtype == (in_dtype if out_dtype is None else out_dtype)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_page_size_64_and_bmm2_scale():
    w = wl.DecodeWorkload(name="ps64", batch=4, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                          page_size=64, kv_len_range=(1, 900), bmm2_scale=0.5)
    inp = wl.make_decode_inputs(w, seed=6, device=DEV)
    out, lse, _ = run_decode(inp)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_live_lengths_unfrozen_plan():
    """A plan that does not freeze the lengths reads them at run time (<= planned)."""
    w = wl.shrink(wl.SPEC_DECODE, batch=4, kv_len_range=(300, 1500), table_width=120,
                  window_left=200)
    inp = wl.make_decode_inputs(w, seed=7, device=DEV)
    plan_lens = inp["seq_lens_kv"].clone()
    live = plan_lens - torch.tensor([0, 5, 17, 100], dtype=torch.int32, device=DEV)
    from helpers import decode_plan_for
    plan = decode_plan_for(inp, freeze_seq_lens=False, num_sms=8, split_waves=2)
    inp2 = dict(inp, seq_lens_kv=live)
    out, lse = api.paged_decode_run(plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                    inp["block_tables"], seq_lens_kv=live, sinks=inp["sinks"])
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle_decode(inp2)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_strided_query_and_combined_kv():
    """q as a slice of a wider buffer; K and V interleaved in one pool tensor."""
    w = wl.shrink(wl.TINY_DECODE, batch=3)
    inp = wl.make_decode_inputs(w, seed=8, device=DEV)
    q = inp["q"]
    wide = torch.zeros((q.shape[0], q.shape[1] * 3, 128), dtype=q.dtype, device=DEV)
    wide[:, 8:16] = q
    qs = wide[:, 8:16]
    P, H, ps, D = inp["k_pages"].shape
    comb = torch.stack([inp["k_pages"], inp["v_pages"]], dim=1).contiguous()   # [P, 2, H, ps, D]
    kview, vview = comb[:, 0], comb[:, 1]
    from helpers import decode_plan_for
    plan = decode_plan_for(inp)
    out, lse = api.paged_decode_run(plan, qs, kview, vview, inp["block_tables"])
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_plan_update_reuses_and_grows():
    """One plan re-planned for three batches: 2 requests, then 40 (outgrows the plan's
    device buffer: reallocated), then 5 (fits: reused)."""
    from helpers import decode_plan_for
    plan = None
    for seed, batch in [(15, 2), (16, 40), (17, 5)]:
        w = wl.shrink(SMALL["llama3_8b"], batch=batch, pool_pages=7000)
        inp = wl.make_decode_inputs(w, seed=seed, device=DEV)
        if plan is None:
            plan = decode_plan_for(inp, num_sms=16)
        else:
            plan.update(inp["seq_lens_kv"].cpu())
        out, lse, _ = run_decode(inp, plan=plan)
        ref_o, ref_l = oracle_decode(inp)
        assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("G,ps,kernel", [(4, 256, "cuda_core"), (4, 256, "default"),
                                         (8, 256, "default"), (16, 128, "default")])
def test_decode_largest_page_sizes(G, ps, kernel):
    """page_size up to 256 (16 TMA units per page), GQA group 4, 8 and 16 rows."""
    w = wl.DecodeWorkload(name="bigpage", batch=3, num_qo_heads=2 * G, num_kv_heads=2,
                          head_dim=128, page_size=ps, kv_len_range=(1, 2000), causal=True)
    inp = wl.make_decode_inputs(w, seed=18, device=DEV)
    out, lse, _ = run_decode(inp, **KERNELS[kernel])
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("G,ps,kernel", [(4, 48, "cuda_core"), (4, 48, "default"),
                                         (8, 80, "default"), (2, 208, "cuda_core"),
                                         (2, 208, "default")])
def test_decode_page_sizes_not_powers_of_two(G, ps, kernel):
    """Any multiple of 16 is a page size: 3, 5 and 13 TMA units per page, with split
    requests whose chunks end inside the unit runs of such pages."""
    w = wl.DecodeWorkload(name="oddpage", batch=3, num_qo_heads=2 * G, num_kv_heads=2,
                          head_dim=128, page_size=ps, kv_len_range=(1, 2000), causal=True,
                          sinks=True)
    inp = wl.make_decode_inputs(w, seed=20 + ps, device=DEV)
    out, lse, plan = run_decode(inp, **KERNELS[kernel])
    assert plan.info["num_split"] > 0
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_single_request_single_key():
    """The degenerate decode: one request, one key -> O is that key's value row (bmm2 1)."""
    w = wl.DecodeWorkload(name="one", batch=1, num_qo_heads=4, num_kv_heads=1, head_dim=128,
                          page_size=16, kv_len_range=(1, 1))
    inp = wl.make_decode_inputs(w, seed=19, device=DEV)
    out, lse, _ = run_decode(inp)
    page = int(inp["block_tables"][0, 0])
    v0 = inp["v_pages"][page, 0, 0].float()
    assert torch.equal(out[0].float(), v0.expand(4, 128))
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_sink_minus_infinity_is_no_sink():
    inp = wl.make_decode_inputs(SMALL["spec"], seed=20, device=DEV)
    out_a, lse_a, _ = run_decode(dict(inp, sinks=torch.full_like(inp["sinks"], -float("inf"))))
    out_b, lse_b, _ = run_decode(dict(inp, sinks=None))
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


def test_decode_graph_capture_replays_eagerly_equal():
    inp = wl.make_decode_inputs(SMALL["skewed"], seed=9, device=DEV)
    from helpers import decode_plan_for
    plan = decode_plan_for(inp, num_sms=32, split_waves=2)
    assert plan.info["num_split"] > 0   # the graph holds the decode and its dependent merge
    out = torch.empty_like(inp["q"])
    lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=DEV)
    ws = torch.empty(max(plan.workspace_bytes, 1), dtype=torch.uint8, device=DEV)
    args = (plan, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_tables"])
    api.paged_decode_run(*args, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone(), lse.clone()
    out.zero_()
    lse.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            api.paged_decode_run(*args, out=out, lse=lse, workspace=ws, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])


# --------------------------------------------------------------------------
# Full-size workloads, in the launch configuration bench.py times: sampled
# requests (longest, shortest, a middle one) against the oracle.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,kernel", [("llama3_8b", "default"), ("llama3_8b", "cuda_core"),
                                         ("skewed", "default"), ("spec", "default")])
def test_decode_full_size_sampled(name, kernel):
    w = wl.DECODE_WORKLOADS[name]
    inp = wl.make_decode_inputs(w, seed=0, device=DEV)
    out, lse, plan = run_decode(inp, return_lse=True, **KERNELS[kernel])
    seq = inp["seq_lens_kv"].cpu().numpy()
    order = np.argsort(-seq, kind="stable")
    reqs = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    ref_o, ref_l = oracle_decode(inp, requests=reqs)
    rows = row_mask(inp, reqs)
    assert_close(out, lse, ref_o, ref_l, rows=rows)
    assert torch.isfinite(out.float()).all()


def test_decode_long_single_tile_requests_cut_by_slot_load():
    """64 requests of U[512, 8192] keys with 8 query heads per KV head (one 16-row tile per
    request): the CTA target leaves them whole, and the plan cuts those longer than 3/5 of a
    resident slot's average load into chunks merged in the kernel.  Sampled requests (the
    longest, the shortest, the middle) against the oracle."""
    w = wl.DecodeWorkload(name="cut", batch=64, num_qo_heads=64, num_kv_heads=8, head_dim=128,
                          page_size=16, kv_len_range=(512, 8192), pool_pages=40000,
                          table_width=512, return_lse=True)
    inp = wl.make_decode_inputs(w, seed=33, device=DEV)
    out, lse, plan = run_decode(inp, num_sms=152)
    assert plan.info["kernel"] == 1 and plan.info["num_split"] > 0
    assert plan.info["num_items"] > 64 * 8
    seq = inp["seq_lens_kv"].cpu().numpy()
    order = np.argsort(-seq, kind="stable")
    reqs = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    ref_o, ref_l = oracle_decode(inp, requests=reqs)
    assert_close(out, lse, ref_o, ref_l, rows=row_mask(inp, reqs))


def test_decode_many_short_requests():
    """2048 requests of 1-64 keys (4096 CTAs, ragged single pages), sampled requests."""
    w = wl.shrink(wl.TINY_DECODE, batch=2048, kv_len_range=(1, 64), pool_pages=2048 * 4 + 64,
                  table_width=4)
    inp = wl.make_decode_inputs(w, seed=31, device=DEV)
    out, lse, plan = run_decode(inp, return_lse=True)
    reqs = [0, 1, 777, 1500, 2047]
    ref_o, ref_l = oracle_decode(inp, requests=reqs)
    assert_close(out, lse, ref_o, ref_l, rows=row_mask(inp, reqs))
    assert torch.isfinite(out.float()).all()
