"""Scores that climb across the keys, against the fp64 oracle.

Every test draws keys whose component along one direction grows with the key's
position and queries that point along it (``workloads.climbing_keys`` /
``aligned_queries``), so each row's running maximum rises from one key tile to
the next:

* prefill: the row max moves by more than 2^8 (log2 units) after the first
  64-key tile, which is when the prefill kernel rescales O held in tensor
  memory (after waiting for the P V of the previous tile);
* decode: a split request's chunks end with partial base-2 LSEs more than 20
  apart, so the merge weights them by factors below 2^-20.

The sm_scale / scale conventions, the bottom-right causal diagonal and the
windows are those of batch_prefill and cudnn_batch_decode_with_kv_cache; the
oracle is the plain softmax over each row's keys.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

from helpers import LSE_ATOL, O_ATOL, O_RTOL, assert_close, decode_plan_for, oracle_decode

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)
KEY_TILE = 64          # keys per prefill K/V tile
RESCALE_STEP = 8.0     # the prefill rescales O when the row max grows by more than this (log2)


def _indptr(lens):
    return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _climbing_prefill(lq, lk, Hq, Hkv, D, dtype, seed, slope):
    g = torch.Generator(device="cpu").manual_seed(seed)
    u = wl.unit_direction(D, g)
    qi, ki = _indptr(lq), _indptr(lk)
    pos = torch.cat([torch.arange(n) for n in lk])     # key position inside its request
    k = wl.climbing_keys(pos, Hkv, u, slope, g).to(dtype).to("cuda")
    v = torch.randn((int(ki[-1]), Hkv, D), generator=g).to(dtype).to("cuda")
    q = wl.aligned_queries(int(qi[-1]), Hq, u, g).to(dtype).to("cuda")
    return q, k, v, qi, ki


def _prefill_rescale_events(q, k, qi, ki, Hkv, sm_scale, causal, window_left):
    """(row, head, key tile) triples past a row's first visible 64-key tile at which
    that tile's largest visible score, in log2 units, exceeds the running reference
    maximum by more than 2^8: each is a tile where the kernel's lazy rule rescales O."""
    qf, kf = _f64(q), _f64(k)
    Hq = qf.shape[1]
    G = Hq // Hkv
    events = 0
    for b in range(len(qi) - 1):
        q0, q1, k0, k1 = int(qi[b]), int(qi[b + 1]), int(ki[b]), int(ki[b + 1])
        Lq, Lk = q1 - q0, k1 - k0
        for h in range(Hq):
            s = sm_scale * LOG2E * (qf[q0:q1, h] @ kf[k0:k1, h // G].T)
            for i in range(Lq):
                lo, hi = oracle.decode_row_key_range(Lk, Lq, i, causal, window_left)
                ref = -math.inf
                for t in range(lo // KEY_TILE, -(-hi // KEY_TILE)):
                    a, z = max(lo, t * KEY_TILE), min(hi, (t + 1) * KEY_TILE)
                    mx = s[i, a:z].max()
                    if mx > ref + RESCALE_STEP:
                        events += t > lo // KEY_TILE and ref > -math.inf
                        ref = mx
    return events


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal,W", [(True, -1), (True, 100), (False, -1), (False, 300)])
def test_prefill_lazy_rescale(D, dtype, causal, W):
    """Row maxima that climb by ~11-14 (log2) per 64-key tile: O in tensor memory is
    rescaled at nearly every tile.  With the window, the rows whose window starts at
    key 64t + 63 see a single (the lowest) score in their first tile."""
    lq = [300, 1, 700, 129]
    lk = [300, 1, 700, 200] if causal else [420, 5, 700, 129]
    sm_scale = 0.5
    q, k, v, qi, ki = _climbing_prefill(lq, lk, 4, 2, D, dtype, seed=100 + D, slope=0.25)
    events = _prefill_rescale_events(q, k, qi, ki, 2, sm_scale, causal, W)
    assert events > 300, events
    plan = api.batch_prefill_plan(qi, ki, num_qo_heads=4, num_kv_heads=2, causal=causal,
                                  return_lse=True, dtype=dtype, head_dim=D, sm_scale=sm_scale,
                                  window_left=W, output_scale=0.75)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    name = "f16" if dtype == torch.float16 else "bf16"
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v),
                                        qi.numpy(), ki.numpy(), 2, causal=causal,
                                        sm_scale=sm_scale, output_scale=0.75, window_left=W,
                                        dtype=name)
    assert_close(out, lse, ref_o, ref_l)


def test_prefill_lazy_rescale_variable_window():
    """Per-query bounds (fixed shape) over climbing keys: row i sees the last key of
    64-key tile i // 64 - 3 (its lowest score, alone in that tile), then every key up to
    i, so the later tiles raise the row max past 2^8."""
    B, S, Hq, Hkv, D = 2, 320, 4, 2, 128
    g = torch.Generator(device="cpu").manual_seed(120)
    u = wl.unit_direction(D, g)
    pos = torch.arange(S).repeat(B)
    k = wl.climbing_keys(pos, Hkv, u, 0.25, g).to(torch.bfloat16).to("cuda")
    v = torch.randn((B * S, Hkv, D), generator=g).to(torch.bfloat16).to("cuda")
    q = wl.aligned_queries(B * S, Hq, u, g).to(torch.bfloat16).to("cuda")
    i = np.arange(S)
    st = np.tile(np.maximum(0, (i // KEY_TILE - 2) * KEY_TILE - 1), (B, 1)).astype(np.int32)
    en = np.tile(i, (B, 1)).astype(np.int32)
    plan = api.batch_prefill_plan_fixed(B, S, S, num_qo_heads=Hq, num_kv_heads=Hkv,
                                        mask_type="variable_window", sm_scale=0.5,
                                        variable_window_token_starts=st,
                                        variable_window_token_ends=en, return_lse=True)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    ind = np.arange(B + 1) * S
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), ind,
                                        ind, Hkv, sm_scale=0.5, window_starts=st, window_ends=en)
    assert_close(out, lse, ref_o, ref_l)


# --------------------------------------------------------------------------
# decode: split partials whose LSEs lie far apart
# --------------------------------------------------------------------------

DECODE_CASES = {
    # 4 rows per KV head (the tensor-core kernel by default; the CUDA-core one below)
    "llama3_8b": wl.shrink(wl.LLAMA3_8B_DECODE, batch=4, kv_len_range=(1500, 2100),
                           pool_pages=700, table_width=160, return_lse=True),
    # tensor-core kernel (8 rows), one long request
    "skewed": wl.shrink(wl.SKEWED_DECODE, batch=3, fixed_first_kv_len=2600,
                        kv_len_range=(600, 1200), table_width=100),
    # tensor-core kernel, packed causal rows, window and sinks
    "spec": wl.shrink(wl.SPEC_DECODE, batch=4, kv_len_range=(1200, 2400), window_left=1500,
                      table_width=160),
}


def _chunk_lse_spread(inp, plan):
    """Largest spread (max - min) of the chunk LSEs of one (row, head) of a split
    request: the base-2 log-sum-exp of the row's visible keys in each chunk."""
    ex = plan.export()
    ps = inp["page_size"]
    qf = _f64(inp["q"])
    kp = inp["k_pages"]
    bt = inp["block_tables"].cpu().numpy()
    seq = inp["seq_lens_kv"].cpu().numpy()
    Hq = qf.shape[1]
    G = Hq // inp["num_kv_heads"]
    ind = (inp["qo_indptr"].cpu().numpy() if inp["qo_indptr"] is not None
           else np.arange(len(seq) + 1) * inp["q_len"])
    scale = 1.0 / math.sqrt(qf.shape[2])
    spread = 0.0
    for b, nch in enumerate(ex["n_chunks"]):
        if nch < 2:
            continue
        n, L = int(seq[b]), int(ind[b + 1] - ind[b])
        i, h = L - 1, 0
        lo, hi = oracle.decode_row_key_range(n, L, i, inp["causal"], inp["window_left"])
        keys = np.arange(lo, hi)
        kk = _f64(kp[torch.as_tensor(bt[b, keys // ps], dtype=torch.long), h // G,
                     torch.as_tensor(keys % ps, dtype=torch.long)])
        s = scale * LOG2E * (kk @ qf[ind[b] + i, h])
        lses = []
        for (rb, hk, ci, plo, phi) in ex["items"]:
            if rb != b or hk != 0:
                continue
            sel = (keys >= plo * ps) & (keys < phi * ps)
            if sel.any():
                m = s[sel].max()
                lses.append(m + math.log2(np.exp2(s[sel] - m).sum()))
        spread = max(spread, max(lses) - min(lses))
    return spread


@pytest.mark.parametrize("name,mma_min_rows", [(n, 0) for n in DECODE_CASES] +
                         [("llama3_8b", 16)])   # the last: the CUDA-core kernel
def test_decode_split_partials_far_apart(name, mma_min_rows):
    inp = wl.make_climbing_decode_inputs(DECODE_CASES[name], seed=130, device="cuda", slope=1.0)
    plan = decode_plan_for(inp, num_sms=64, split_waves=2, min_chunk_tokens=128,
                           mma_min_rows=mma_min_rows)
    assert plan.info["kernel"] == (0 if mma_min_rows == 16 else 1)
    assert plan.info["num_split"] > 0
    spread = _chunk_lse_spread(inp, plan)
    assert spread > 20.0, spread
    out, lse = api.paged_decode_run(plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                    inp["block_tables"], sinks=inp["sinks"])
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)
