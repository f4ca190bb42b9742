"""paged_decode_step_host: one decode step from host buffers (copies in, re-plan
on the step's lengths, run, copies out; or host arrays used in place) returns the
bytes paged_decode_run
returns on device copies of the same inputs, step after step, and matches the
oracle."""

import pytest
import torch

from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

from helpers import assert_close, decode_plan_for, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"

LLAMA = wl.shrink(wl.LLAMA3_8B_DECODE, batch=6, kv_len_range=(512, 2100), pool_pages=1000,
                  table_width=160, return_lse=True)
SPEC = wl.shrink(wl.SPEC_DECODE, batch=6, kv_len_range=(2048, 6000), table_width=400)


def _make_io(inp, out_dtype, in_place=False):
    """Pinned host buffers sized for the batch in ``inp``, with device staging, or
    (``in_place``) with every device slot given its pinned host tensor itself."""
    q, bt, seq = inp["q"], inp["block_tables"], inp["seq_lens_kv"]
    rows = q.shape[:2]
    host = dict(
        q_host=torch.empty(q.shape, dtype=q.dtype).pin_memory(),
        block_tables_host=torch.empty(bt.shape, dtype=torch.int32).pin_memory(),
        seq_lens_kv_host=torch.empty(seq.shape, dtype=torch.int32).pin_memory(),
        out_host=torch.empty(q.shape, dtype=out_dtype).pin_memory(),
        lse_host=torch.empty(rows, dtype=torch.float32).pin_memory(),
        qo_indptr_host=(None if inp["qo_indptr"] is None else
                        torch.empty(inp["qo_indptr"].shape, dtype=torch.int32).pin_memory()))
    if in_place:
        dev = dict(q_dev=host["q_host"], block_tables_dev=host["block_tables_host"],
                   seq_lens_kv_dev=host["seq_lens_kv_host"], out_dev=host["out_host"],
                   lse_dev=host["lse_host"])
    else:
        dev = dict(q_dev=torch.empty_like(q), block_tables_dev=torch.empty_like(bt),
                   seq_lens_kv_dev=torch.empty_like(seq),
                   out_dev=torch.empty(q.shape, dtype=out_dtype, device=DEV),
                   lse_dev=torch.empty(rows, dtype=torch.float32, device=DEV))
    return api.DecodeHostIO(**host, **dev)


def _fill(io, inp):
    """Write one step's inputs into the leading rows of the host buffers."""
    t = io.tensors
    B, tq = inp["seq_lens_kv"].numel(), inp["q"].shape[0]
    t["q_host"][:tq].copy_(inp["q"].cpu())
    t["block_tables_host"][:B].copy_(inp["block_tables"].cpu())
    t["seq_lens_kv_host"][:B].copy_(inp["seq_lens_kv"].cpu())
    if inp["qo_indptr"] is not None:
        t["qo_indptr_host"][:B + 1].copy_(inp["qo_indptr"].cpu())
    return B, tq


def _next_step(inp, seed, batch):
    """The next step's batch over the same pools: the first ``batch`` requests with
    shorter lengths (their table rows stay valid) and new queries."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    seq = inp["seq_lens_kv"][:batch].cpu()
    L = (torch.full((batch,), inp["q_len"], dtype=torch.int32) if inp["qo_indptr"] is None
         else (inp["qo_indptr"][1:batch + 1] - inp["qo_indptr"][:batch]).cpu())
    cut = torch.randint(0, 400, (batch,), generator=g, dtype=torch.int32)
    seq = torch.maximum(seq - cut, L)
    nxt = dict(inp, seq_lens_kv=seq.to(DEV), block_tables=inp["block_tables"][:batch])
    if inp["qo_indptr"] is not None:
        nxt["qo_indptr"] = inp["qo_indptr"][:batch + 1]
    tq = int(L.sum())
    q = torch.randn((tq,) + tuple(inp["q"].shape[1:]), generator=g).to(inp["q"].dtype)
    nxt["q"] = q.to(DEV)
    return nxt


def _run_reference(inp, **kw):
    plan = decode_plan_for(inp, **kw)
    out, lse = api.paged_decode_run(plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                    inp["block_tables"], seq_lens_kv=inp["seq_lens_kv"],
                                    sinks=inp["sinks"])
    torch.cuda.synchronize()
    plan.check()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("name,kw", [
    ("llama3_8b", {}),
    ("spec", dict(freeze_seq_lens=False, num_sms=32, split_waves=2, min_chunk_tokens=128)),
])
def test_step_host_equals_run_step_after_step(name, kw, in_place):
    """Staged (device copies) or in place (the kernels read q, tables and live lengths
    and write O and the LSE in pinned host memory): the same bytes either way."""
    w = LLAMA if name == "llama3_8b" else SPEC
    inp = wl.make_decode_inputs(w, seed=21, device=DEV)
    out_dtype = inp["q"].dtype
    io = _make_io(inp, out_dtype, in_place)
    plan = decode_plan_for(inp, **kw)
    split_seen = False
    for step, batch in enumerate([inp["seq_lens_kv"].numel(), 4, 5]):
        cur = inp if step == 0 else _next_step(inp, seed=100 + step, batch=batch)
        B, tq = _fill(io, cur)
        out_h, lse_h = api.paged_decode_step_host(plan, io, cur["k_pages"], cur["v_pages"],
                                                  sinks=cur["sinks"], batch_size=B)
        plan.check()
        split_seen = split_seen or plan.info["num_split"] > 0
        ref_o, ref_l = _run_reference(cur, **kw)
        assert torch.equal(out_h[:tq], ref_o), f"step {step}: O differs from paged_decode_run"
        assert torch.equal(lse_h[:tq], ref_l), f"step {step}: LSE differs from paged_decode_run"
        o_or, l_or = oracle_decode(cur)
        assert_close(out_h[:tq], lse_h[:tq], o_or, l_or)
    if kw:   # the split path ran, with a workspace the binding grew on demand
        assert split_seen and io.workspace is not None


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("name,kw", [
    ("llama3_8b", {}),
    ("spec", dict(freeze_seq_lens=False, num_sms=32, split_waves=2, min_chunk_tokens=128)),
])
def test_prepared_step_equals_run_step_after_step(name, kw, in_place):
    """DecodeStep (the step call marshalled once, then repeated on new host contents):
    each call re-plans on the step's lengths and returns the bytes paged_decode_run
    returns on device copies of the same inputs; a packed batch whose rows outgrow the
    io is refused before the call."""
    w = LLAMA if name == "llama3_8b" else SPEC
    inp = wl.make_decode_inputs(w, seed=25, device=DEV)
    io = _make_io(inp, inp["q"].dtype, in_place)
    plan = decode_plan_for(inp, **kw)
    B = inp["seq_lens_kv"].numel()
    step = api.DecodeStep(plan, io, inp["k_pages"], inp["v_pages"], sinks=inp["sinks"])
    for k in range(3):
        cur = inp if k == 0 else _next_step(inp, seed=200 + k, batch=B)
        _, tq = _fill(io, cur)
        out_h, lse_h = step()
        plan.check()
        ref_o, ref_l = _run_reference(cur, **kw)
        assert torch.equal(out_h[:tq], ref_o), f"step {k}: O differs from paged_decode_run"
        assert torch.equal(lse_h[:tq], ref_l), f"step {k}: LSE differs from paged_decode_run"
    o_or, l_or = oracle_decode(cur)
    assert_close(out_h[:tq], lse_h[:tq], o_or, l_or)
    if kw:
        assert io.workspace is not None and plan.info["num_split"] > 0
        ind = io.tensors["qo_indptr_host"]
        saved = int(ind[B])
        ind[B] = io.tensors["q_host"].shape[0] + 1
        with pytest.raises(ValueError):
            step()
        ind[B] = saved


@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float16, torch.float32),
                                               (torch.bfloat16, torch.float16)])
def test_step_host_input_and_output_types(in_dtype, out_dtype):
    """Half inputs and fp32 / fp16 outputs: the copies move the plan's element
    sizes (2-byte q in, 4- or 2-byte O out)."""
    inp = wl.make_decode_inputs(LLAMA, seed=23, device=DEV, dtype=in_dtype)
    io = _make_io(inp, out_dtype)
    plan = decode_plan_for(inp, out_dtype=out_dtype)
    B, tq = _fill(io, inp)
    out_h, lse_h = api.paged_decode_step_host(plan, io, inp["k_pages"], inp["v_pages"],
                                              sinks=inp["sinks"], batch_size=B)
    plan.check()
    assert out_h.dtype == out_dtype
    ref_plan = decode_plan_for(inp, out_dtype=out_dtype)
    ref_o, ref_l = api.paged_decode_run(ref_plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                        inp["block_tables"], seq_lens_kv=inp["seq_lens_kv"],
                                        sinks=inp["sinks"])
    torch.cuda.synchronize()
    assert torch.equal(out_h[:tq], ref_o.cpu()) and torch.equal(lse_h[:tq], ref_l.cpu())
    o_or, l_or = oracle_decode(inp)
    assert_close(out_h[:tq], lse_h[:tq], o_or, l_or)


def test_step_host_rejects_a_batch_larger_than_the_buffers():
    inp = wl.make_decode_inputs(LLAMA, seed=22, device=DEV)
    small = dict(inp, q=inp["q"][:3], block_tables=inp["block_tables"][:3],
                 seq_lens_kv=inp["seq_lens_kv"][:3])
    io = _make_io(small, inp["q"].dtype)
    plan = decode_plan_for(small)
    with pytest.raises(ValueError):
        api.paged_decode_step_host(plan, io, inp["k_pages"], inp["v_pages"], batch_size=6)


def test_step_host_refuses_unpinned_memory_in_place():
    """Through the C ABI: a host array that is not page-locked, given as its own device
    array, is refused before anything runs (the kernels could not address it)."""
    import ctypes
    from paged_kv_attention_32_gb300 import _lib as L
    inp = wl.make_decode_inputs(LLAMA, seed=24, device=DEV)
    io = _make_io(inp, inp["q"].dtype)
    _fill(io, inp)
    plan = decode_plan_for(inp)
    q_plain = io.tensors["q_host"].clone()        # pageable host memory
    c = L.DecodeHostIO.from_buffer_copy(io.c)
    c.q_host = c.q_dev = q_plain.data_ptr()
    ws_need = ctypes.c_size_t()
    rc = L.lib().paged_decode_step_host(
        plan.handle, inp["seq_lens_kv"].numel(), ctypes.byref(c), inp["k_pages"].data_ptr(),
        inp["v_pages"].data_ptr(), inp["k_pages"].stride(0), inp["k_pages"].stride(1), None,
        None, 0, ctypes.byref(ws_need), 1, torch.cuda.current_stream().cuda_stream)
    assert rc == L.PKA_ERR_INVALID_ARG
    assert "page-locked" in L.lib().pka_last_error().decode()
