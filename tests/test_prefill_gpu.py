"""Ragged causal prefill (tcgen05 kernel) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

from helpers import LSE_ATOL, O_ATOL, O_RTOL

pytestmark = pytest.mark.gpu


def _rand(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda", dtype=dtype)


def _indptr(lens):
    return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)


def _check(out, lse, ref_o, ref_l):
    o = out.float().cpu().numpy()
    ok = np.abs(o - ref_o) <= O_ATOL + O_RTOL * np.abs(ref_o)
    assert ok.all(), f"max err {np.abs(o - ref_o).max():.4g} at {np.argwhere(~ok)[:4].tolist()}"
    if lse is not None:
        l = lse.cpu().numpy().astype(np.float64)
        assert (np.abs(l - ref_l) <= LSE_ATOL).all(), f"LSE err {np.abs(l - ref_l).max():.4g}"


def _run(lq, lk, Hq, Hkv, causal=True, seed=0, dtype=torch.bfloat16, out_dtype=None, D=128,
         **kw):
    qi, ki = _indptr(lq), _indptr(lk)
    q = _rand((int(qi[-1]), Hq, D), seed + 1, dtype)
    k = _rand((int(ki[-1]), Hkv, D), seed + 2, dtype)
    v = _rand((int(ki[-1]), Hkv, D), seed + 3, dtype)
    plan = api.batch_prefill_plan(qi, ki, num_qo_heads=Hq, num_kv_heads=Hkv, causal=causal,
                                  return_lse=True, dtype=dtype, out_dtype=out_dtype, head_dim=D,
                                  **kw)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    assert out.dtype == (dtype if out_dtype is None else out_dtype)
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v),
                                        qi.numpy(), ki.numpy(), Hkv, causal=causal,
                                        dtype="f16" if dtype == torch.float16 else "bf16", **kw)
    _check(out, lse, ref_o, ref_l)


def test_prefill_fused_qkv_views():
    """q, k and v as head slices of one fused [total, Hq + 2 Hkv, D] projection output
    (strided tokens, K and V at other base pointers with the same strides)."""
    lens = [70, 129, 3]
    qi = _indptr(lens)
    Hq, Hkv, D = 4, 2, 128
    qkv = _rand((int(qi[-1]), Hq + 2 * Hkv, D), 91)
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    plan = api.batch_prefill_plan(qi, qi, num_qo_heads=Hq, num_kv_heads=Hkv, return_lse=True)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q.contiguous()), wl.bf16_bits(k.contiguous()),
                                        wl.bf16_bits(v.contiguous()), qi.numpy(), qi.numpy(), Hkv,
                                        causal=True)
    _check(out, lse, ref_o, ref_l)


def test_prefill_smallest():
    _run([1, 5, 130], [1, 5, 130], 4, 2)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (6, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_matches_oracle(Hq, Hkv, causal):
    lens = [1, 5, 127, 128, 129, 300, 513]
    _run(lens, lens, Hq, Hkv, causal=causal, seed=10, output_scale=0.75)


def test_prefill_bottom_right_causal_with_longer_kv():
    _run([3, 130, 64], [40, 200, 64], 4, 2, seed=20, sm_scale=0.05)


@pytest.mark.parametrize("W", [0, 5, 127, 128, 300])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_window_left(W, causal):
    """Plain sliding window: row i keeps keys from Lk - Lq + i - W on; tiles left of
    every row's window are skipped, partly covered ones masked per row."""
    lq = [1, 130, 300, 513]
    lk = [1, 200, 300, 700] if causal else [5, 130, 410, 513]
    _run(lq, lk, 8, 2, causal=causal, seed=30 + W, window_left=W)


@pytest.mark.parametrize("W", [-1, 40])
def test_prefill_zero_scale_is_a_mean_over_visible_keys(W):
    """sm_scale = 0: every visible key gets the same weight, so O is the mean of the
    visible V rows; masked keys must still get none (their -inf score times 0 would
    otherwise give NaN)."""
    _run([1, 130, 257], [1, 200, 300], 4, 2, seed=45, sm_scale=0.0, window_left=W)


def test_prefill_window_odd_group():
    _run([257, 64], [400, 64], 6, 2, seed=40, window_left=60)


def _fixed_case(B, Sq, Sk, Hq, Hkv, seed, **kw):
    q = _rand((B, Sq, Hq, 128), seed + 1)
    k, v = _rand((B, Sk, Hkv, 128), seed + 2), _rand((B, Sk, Hkv, 128), seed + 3)
    plan = api.batch_prefill_plan_fixed(B, Sq, Sk, num_qo_heads=Hq, num_kv_heads=Hkv,
                                        return_lse=True, **kw)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    assert out.shape == (B, Sq, Hq, 128) and lse.shape == (B, Sq, Hq)
    mask = kw.get("mask_type", "causal")
    okw = dict(causal=mask == "causal", window_left=kw.get("window_left", -1))
    if mask == "variable_window":
        okw = dict(window_starts=kw["variable_window_token_starts"],
                   window_ends=kw["variable_window_token_ends"])
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q.flatten(0, 1)), wl.bf16_bits(k.flatten(0, 1)),
                                        wl.bf16_bits(v.flatten(0, 1)), np.arange(B + 1) * Sq,
                                        np.arange(B + 1) * Sk, Hkv, **okw)
    _check(out.flatten(0, 1), lse.flatten(0, 1), ref_o, ref_l)


@pytest.mark.parametrize("mask,W", [("causal", -1), ("dense", -1), ("causal", 100),
                                    ("dense", 37)])
def test_prefill_fixed_shape(mask, W):
    """[B, S, H, D] storage without offset tensors, Sq < Sk (bottom-right diagonal)."""
    _fixed_case(3, 200, 333, 8, 2, seed=50, mask_type=mask, window_left=W)


@pytest.mark.parametrize("Hq,Hkv,seed", [(8, 2, 60), (6, 2, 61)])
def test_prefill_variable_window(Hq, Hkv, seed):
    """Per-query inclusive key bounds: random spans, some of a single key, some far
    left of the diagonal, over several 64-key tiles."""
    B, Sq, Sk = 3, 260, 400
    g = np.random.default_rng(seed)
    a, b = g.integers(0, Sk, size=(B, Sq)), g.integers(0, Sk, size=(B, Sq))
    st, en = np.minimum(a, b).astype(np.int32), np.maximum(a, b).astype(np.int32)
    en[:, ::7] = st[:, ::7]                      # single-key rows
    _fixed_case(B, Sq, Sk, Hq, Hkv, seed=seed, mask_type="variable_window",
                variable_window_token_starts=st, variable_window_token_ends=en)


@pytest.mark.parametrize("D,out_dtype", [(128, None), (128, torch.float32), (256, None)])
def test_prefill_variable_window_reordered_rows(D, out_dtype):
    """Row i sees [i - U(0, 511), i] (the bench's variable_window shape, smaller): the
    planner groups rows of similar windows into tiles (rows ordered by last key in
    bands of four tiles, by first key inside a band), so the kernel gathers Q rows
    and scatters O / LSE rows through the row order."""
    B, S, Hq, Hkv = 2, 1024, 4, 2
    g = np.random.default_rng(100 + D)
    i = np.arange(S)
    st = (i - g.integers(0, 512, size=(B, S))).clip(0, None).astype(np.int32)
    en = np.tile(i, (B, 1)).astype(np.int32)
    q = _rand((B, S, Hq, D), 101)
    k, v = _rand((B, S, Hkv, D), 102), _rand((B, S, Hkv, D), 103)
    plan = api.batch_prefill_plan_fixed(B, S, S, num_qo_heads=Hq, num_kv_heads=Hkv,
                                        mask_type="variable_window", head_dim=D,
                                        variable_window_token_starts=st,
                                        variable_window_token_ends=en, return_lse=True,
                                        out_dtype=out_dtype)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q.flatten(0, 1)), wl.bf16_bits(k.flatten(0, 1)),
                                        wl.bf16_bits(v.flatten(0, 1)), np.arange(B + 1) * S,
                                        np.arange(B + 1) * S, Hkv, window_starts=st, window_ends=en)
    _check(out.flatten(0, 1), lse.flatten(0, 1), ref_o, ref_l)


@pytest.mark.parametrize("dtype,out_dtype", [(torch.float16, None), (torch.float16, torch.float32),
                                             (torch.bfloat16, torch.float32),
                                             (torch.bfloat16, torch.float16)])
def test_prefill_input_and_output_dtypes(dtype, out_dtype):
    """fp16 q/k/v (kind::f16 MMAs on half operands) and out_dtype (batch_prefill)."""
    lens = [1, 127, 300, 513]
    _run(lens, lens, 8, 2, seed=70, dtype=dtype, out_dtype=out_dtype, window_left=200)


@pytest.mark.parametrize("causal,W", [(True, -1), (False, -1), (True, 100)])
def test_prefill_head_dim_256(causal, W):
    """head_dim 256 (batch_prefill allows D = 128 or 256): 64-key tiles, one head per CTA."""
    lq = [1, 64, 65, 127, 300, 513]
    lk = [1, 64, 100, 127, 400, 513] if causal else [9, 64, 65, 200, 300, 513]
    _run(lq, lk, 4, 2, causal=causal, seed=80, D=256, window_left=W, output_scale=0.5)


@pytest.mark.parametrize("dtype,out_dtype", [(torch.float16, torch.float32), (torch.bfloat16, None)])
def test_prefill_head_dim_256_dtypes_and_odd_group(dtype, out_dtype):
    _run([200, 37], [260, 37], 6, 2, seed=81, D=256, dtype=dtype, out_dtype=out_dtype)


def test_prefill_head_dim_256_variable_window():
    B, Sq, Sk = 2, 150, 230
    g = np.random.default_rng(82)
    a, b = g.integers(0, Sk, size=(B, Sq)), g.integers(0, Sk, size=(B, Sq))
    st, en = np.minimum(a, b).astype(np.int32), np.maximum(a, b).astype(np.int32)
    q = _rand((B, Sq, 4, 256), 83)
    k, v = _rand((B, Sk, 2, 256), 84), _rand((B, Sk, 2, 256), 85)
    plan = api.batch_prefill_plan_fixed(B, Sq, Sk, num_qo_heads=4, num_kv_heads=2,
                                        mask_type="variable_window", head_dim=256,
                                        variable_window_token_starts=st,
                                        variable_window_token_ends=en, return_lse=True)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle.batch_prefill(wl.bf16_bits(q.flatten(0, 1)), wl.bf16_bits(k.flatten(0, 1)),
                                        wl.bf16_bits(v.flatten(0, 1)), np.arange(B + 1) * Sq,
                                        np.arange(B + 1) * Sk, 2, window_starts=st, window_ends=en)
    _check(out.flatten(0, 1), lse.flatten(0, 1), ref_o, ref_l)


@pytest.mark.parametrize("D", [128, 256])
def test_prefill_empty_and_single_row_requests(D):
    """Requests with no rows and no keys, and one-row one-key requests, among others."""
    _run([0, 1, 0, 200, 1], [0, 1, 0, 230, 5], 4, 2, seed=90, D=D)


@pytest.mark.parametrize("window", [-1, 4095])
def test_prefill_one_long_request(window):
    """One 32768-token causal request: a query tile visits up to 512 key tiles and the
    K/V token coordinates pass 2^15; with and without a 4096-key window.  Sampled rows
    (both ends of tiles, the middle, the last rows) and heads against the oracle."""
    n, Hq, Hkv, D = 32768, 8, 2, 128
    q, k, v = _rand((n, Hq, D), 40), _rand((n, Hkv, D), 41), _rand((n, Hkv, D), 42)
    ind = _indptr([n])
    plan = api.batch_prefill_plan(ind, ind, num_qo_heads=Hq, num_kv_heads=Hkv, causal=True,
                                  return_lse=True, window_left=window)
    out, lse = api.batch_prefill_run(plan, q, k, v)
    torch.cuda.synchronize()
    plan.check()
    rows = [0, 1, 127, 128, 4095, 4096, 4097, 16383, 16384, 32639, 32640, 32767]
    heads = [0, 3, 7]
    ro, rl = oracle.prefill_request(0, wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v),
                                    ind.numpy(), ind.numpy(), Hkv, heads=heads, rows=rows,
                                    window_left=window)
    got_o, got_l = out.float().cpu().numpy(), lse.cpu().numpy()
    for h in heads:
        d = np.abs(got_o[rows, h] - ro[rows, h])
        assert (d <= O_ATOL + O_RTOL * np.abs(ro[rows, h])).all(), d.max()
        assert (np.abs(got_l[rows, h] - rl[rows, h]) <= LSE_ATOL).all()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("D", [128, 256])
def test_prefill_full_size_sampled(D):
    """The ragged prefill workload at full size (as bench.py times it, head_dim 128 and
    the 256 line), sampled rows."""
    import dataclasses
    w = wl.RAGGED_PREFILL
    if D != w.head_dim:
        w = dataclasses.replace(w, head_dim=D)
    inp = wl.make_prefill_inputs(w, seed=0, device="cuda")
    ind = inp["qo_indptr"].cpu()
    plan = api.batch_prefill_plan(ind, ind, num_qo_heads=w.num_qo_heads,
                                  num_kv_heads=w.num_kv_heads, return_lse=True, head_dim=D)
    out, lse = api.batch_prefill_run(plan, inp["q"], inp["k"], inp["v"])
    torch.cuda.synchronize()
    plan.check()
    lens = inp["lens"].tolist()
    b = int(np.argmax(lens))
    n = lens[b]
    rows = sorted({0, 1, 127, 128, n // 2, n - 129, n - 1})
    heads = [0, 5, 31]
    qb, kb, vb = wl.bf16_bits(inp["q"]), wl.bf16_bits(inp["k"]), wl.bf16_bits(inp["v"])
    ro, rl = oracle.prefill_request(b, qb, kb, vb, ind.numpy(), ind.numpy(), w.num_kv_heads,
                                    heads=heads, rows=rows)
    base = int(ind[b])
    got_o = out[base:base + n].float().cpu().numpy()
    got_l = lse[base:base + n].cpu().numpy()
    for h in heads:
        d = np.abs(got_o[rows, h] - ro[rows, h])
        assert (d <= O_ATOL + O_RTOL * np.abs(ro[rows, h])).all(), d.max()
        assert (np.abs(got_l[rows, h] - rl[rows, h]) <= LSE_ATOL).all()
    assert torch.isfinite(out.float()).all()
