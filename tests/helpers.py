"""Shared test plumbing: call the CUDA path through the binding, call the
oracle on the same inputs, compare with the tolerances of the parity bar."""

import numpy as np
import torch

import oracle
from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

# bf16 O: |gpu - ref| <= ATOL + RTOL * |ref|;  fp32 base-2 LSE: |gpu - ref| <= LSE_ATOL
O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


def decode_plan_for(inp, **kw):
    w_tables = inp["block_tables"]
    kw.setdefault("dtype", inp["q"].dtype)
    seq = inp["seq_lens_kv"].cpu()
    args = dict(num_qo_heads=inp["q"].shape[1], num_kv_heads=inp["num_kv_heads"],
                page_size=inp["page_size"], max_pages_per_seq=w_tables.shape[1],
                num_pages=inp["k_pages"].shape[0], causal=inp["causal"],
                window_left=inp["window_left"], return_lse=True,
                bmm2_scale=inp["bmm2_scale"])
    if inp["qo_indptr"] is not None:
        args["qo_indptr"] = inp["qo_indptr"].cpu()
    else:
        args["q_len"] = inp["q_len"]
    args.update(kw)
    return api.paged_decode_plan(seq, **args)


def run_decode(inp, plan=None, **kw):
    plan = plan or decode_plan_for(inp, **kw)
    out, lse = api.paged_decode_run(plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                    inp["block_tables"], seq_lens_kv=inp["seq_lens_kv"],
                                    sinks=inp["sinks"])
    torch.cuda.synchronize()
    plan.check()
    return out, lse, plan


def oracle_decode(inp, requests=None, window_left=None):
    dtype = "f16" if inp["q"].dtype == torch.float16 else "bf16"
    q_len = inp["q_len"] if inp["q_len"] is not None else 1
    indptr = inp["qo_indptr"].cpu().numpy() if inp["qo_indptr"] is not None else None
    bt = inp["block_tables"].cpu().numpy()
    need = None
    if requests is not None:   # only copy the pages the sampled requests use
        ps = inp["page_size"]
        need = set()
        seq = inp["seq_lens_kv"].cpu().numpy()
        for b in requests:
            need.update(int(x) for x in bt[b, : -(-int(seq[b]) // ps)])
    kp, vp = inp["k_pages"], inp["v_pages"]
    if need is not None:
        ids = sorted(need)
        remap = {p: i for i, p in enumerate(ids)}
        idx = torch.tensor(ids, dtype=torch.long, device=kp.device)
        kbits = wl.bf16_bits(kp.index_select(0, idx))
        vbits = wl.bf16_bits(vp.index_select(0, idx))
        bt = np.vectorize(lambda p: remap.get(int(p), -1))(bt)
    else:
        kbits, vbits = wl.bf16_bits(kp), wl.bf16_bits(vp)
    sinks = inp["sinks"].cpu().double().numpy() if inp["sinks"] is not None else None
    return oracle.paged_decode(
        wl.bf16_bits(inp["q"]), kbits, vbits, bt, inp["seq_lens_kv"].cpu().numpy(),
        inp["num_kv_heads"], inp["page_size"], qo_indptr=indptr, q_len=q_len,
        causal=inp["causal"], window_left=inp["window_left"] if window_left is None else window_left,
        scale=None, bmm2_scale=inp["bmm2_scale"], sinks=sinks, requests=requests, dtype=dtype)


def row_mask(inp, requests):
    """Boolean mask over packed query rows belonging to `requests`."""
    total = inp["q"].shape[0]
    m = np.zeros(total, dtype=bool)
    if inp["qo_indptr"] is not None:
        ind = inp["qo_indptr"].cpu().numpy()
    else:
        L = inp["q_len"]
        ind = np.arange(len(inp["seq_lens_kv"]) + 1) * L
    for b in requests:
        m[ind[b]:ind[b + 1]] = True
    return m


def assert_close(out, lse, ref_o, ref_lse, rows=None):
    o = out.float().cpu().numpy()
    if rows is not None:
        o, ref_o = o[rows], ref_o[rows]
    err = np.abs(o - ref_o)
    bound = O_ATOL + O_RTOL * np.abs(ref_o)
    bad = err > bound
    assert not bad.any(), (f"O mismatch at {np.argwhere(bad)[:5].tolist()}: "
                           f"max err {err.max():.4g}")
    if lse is not None and ref_lse is not None:
        l = lse.cpu().numpy().astype(np.float64)
        rl = ref_lse
        if rows is not None:
            l, rl = l[rows], rl[rows]
        lerr = np.abs(l - rl)
        assert (lerr <= LSE_ATOL).all(), f"LSE max err {lerr.max():.4g}"
    return float(err.max())
