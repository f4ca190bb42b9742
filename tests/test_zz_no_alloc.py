"""paged_decode_run_noalloc: the decode entry point for callers that cannot
allocate device memory (code inside an allocator hook, or a process whose
device memory is a fixed pool it does not control).  It keeps its work list
and split-KV partials in a fixed array inside the library.  Checked through
the C ABI against paged_decode_run on two calls in a row, against the fp64
oracle (also with live lengths shorter than planned), and for the report of a
wait that gave up, read through paged_decode_plan_check on a host-only plan.
This file is collected last on purpose."""

import ctypes

import pytest
import torch

from paged_kv_attention_32_gb300 import _lib as L
from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

from helpers import LSE_ATOL, O_ATOL, O_RTOL, assert_close, decode_plan_for, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc(plan, inp, out, lse):
    q, kp, vp, bt = inp["q"], inp["k_pages"], inp["v_pages"], inp["block_tables"]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def ptr(t):
        return ctypes.c_void_p(0 if t is None else t.data_ptr())

    return L.lib().paged_decode_run_noalloc(
        plan.handle, ptr(q), q.stride(0), q.stride(1), ptr(kp), ptr(vp), kp.stride(0),
        kp.stride(1), ptr(bt), bt.stride(0), ptr(inp["seq_lens_kv"]), ptr(inp["sinks"]),
        ptr(out), ptr(lse), stream)


@pytest.mark.parametrize("name", ["skewed", "spec"])
def test_noalloc_matches_paged_decode_run_twice(name):
    small = {
        "skewed": wl.shrink(wl.SKEWED_DECODE, batch=5, fixed_first_kv_len=12000,
                            kv_len_range=(1024, 4096), table_width=400),
        "spec": wl.shrink(wl.SPEC_DECODE, batch=6, kv_len_range=(2048, 6000), table_width=400),
    }[name]
    for seed in (11, 12):   # two calls in a row, different inputs
        inp = wl.make_decode_inputs(small, seed=seed, device="cuda")
        ref_plan = decode_plan_for(inp, num_sms=128, split_waves=2)
        host_plan = decode_plan_for(inp, num_sms=128, split_waves=2, host_only=True)
        assert host_plan.info["num_split"] > 0          # the partials go through the scratch
        ref_o, ref_l = api.paged_decode_run(ref_plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                            inp["block_tables"], sinks=inp["sinks"])
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full(inp["q"].shape[:2], float("nan"), device="cuda")
        rc = _noalloc(host_plan, inp, out, lse)
        assert rc == L.PKA_OK, L.lib().pka_last_error()
        torch.cuda.synchronize()
        diff = (out.float() - ref_o.float()).abs()
        assert bool((diff <= O_ATOL + O_RTOL * ref_o.float().abs()).all())
        assert bool(((lse - ref_l).abs() <= LSE_ATOL).all())


def test_noalloc_rejects_plans_beyond_its_scratch():
    # a host-only plan whose split partials alone exceed the 16 MiB scratch
    plan = api.paged_decode_plan([131072] * 2, num_qo_heads=64, num_kv_heads=1, page_size=16,
                                 max_pages_per_seq=8192, num_pages=20000, q_len=1,
                                 num_sms=152, split_waves=32, host_only=True)
    assert plan.workspace_bytes > 16 << 20
    q = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    pages = torch.zeros((1, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((2, 8192), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    inp = {"q": q, "k_pages": pages, "v_pages": pages, "block_tables": bt,
           "seq_lens_kv": None, "sinks": None}
    rc = _noalloc(plan, inp, out, None)
    assert rc == L.PKA_ERR_WORKSPACE_TOO_SMALL
    assert b"16777216" in L.lib().pka_last_error()


@pytest.mark.parametrize("name,mma_min_rows", [("llama3_8b", 0), ("llama3_8b", 16),
                                               ("spec", 0)])
def test_noalloc_matches_the_oracle(name, mma_min_rows):
    """Frozen lengths (llama3_8b shape, split; the tensor-core kernel, the default, and the
    CUDA-core one) and live lengths shorter than planned (spec shape: causal rows, window,
    sinks)."""
    w = {"llama3_8b": wl.shrink(wl.LLAMA3_8B_DECODE, batch=5, kv_len_range=(512, 2100),
                                pool_pages=1000, table_width=160, return_lse=True),
         "spec": wl.shrink(wl.SPEC_DECODE, batch=5, kv_len_range=(600, 2600), window_left=700,
                           table_width=200)}[name]
    inp = wl.make_decode_inputs(w, seed=21, device="cuda")
    frozen = name == "llama3_8b"
    plan = decode_plan_for(inp, num_sms=32 if frozen else 128, split_waves=2,
                           min_chunk_tokens=128, host_only=True, freeze_seq_lens=frozen,
                           mma_min_rows=mma_min_rows)
    assert plan.info["kernel"] == (0 if mma_min_rows == 16 else 1)
    assert plan.info["num_split"] > 0
    if not frozen:
        cut = torch.tensor([0, 7, 100, 333, 1], dtype=torch.int32, device="cuda")
        inp = dict(inp, seq_lens_kv=inp["seq_lens_kv"] - cut)
    out = torch.full_like(inp["q"], float("nan"))
    lse = torch.full(inp["q"].shape[:2], float("nan"), device="cuda")
    assert _noalloc(plan, inp, out, lse) == L.PKA_OK, L.lib().pka_last_error()
    torch.cuda.synchronize()
    plan.check()
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)


def test_noalloc_reports_a_wait_that_gave_up():
    """The kernels' bounded wait, run on the status word of the fixed scratch (the word
    a host-only plan's check reads), is reported once as PKA_ERR_DEVICE_TIMEOUT and
    cleared; the next no-allocation decode still matches paged_decode_run."""
    w = wl.shrink(wl.SKEWED_DECODE, batch=4, fixed_first_kv_len=9000, kv_len_range=(1024, 3000),
                  table_width=300)
    inp = wl.make_decode_inputs(w, seed=23, device="cuda")
    host_plan = decode_plan_for(inp, num_sms=64, split_waves=2, host_only=True)
    host_plan.check()   # nothing pending
    api.wait_timeout_probe(limit_ns=20_000_000, plan=host_plan)
    with pytest.raises(L.PkaError) as exc:
        host_plan.check()
    assert exc.value.code == L.PKA_ERR_DEVICE_TIMEOUT
    host_plan.check()   # the read cleared it
    ref_plan = decode_plan_for(inp, num_sms=64, split_waves=2)
    ref_o, ref_l = api.paged_decode_run(ref_plan, inp["q"], inp["k_pages"], inp["v_pages"],
                                        inp["block_tables"], sinks=inp["sinks"])
    out = torch.full_like(inp["q"], float("nan"))
    lse = torch.full(inp["q"].shape[:2], float("nan"), device="cuda")
    assert _noalloc(host_plan, inp, out, lse) == L.PKA_OK, L.lib().pka_last_error()
    torch.cuda.synchronize()
    host_plan.check()
    diff = (out.float() - ref_o.float()).abs()
    assert bool((diff <= O_ATOL + O_RTOL * ref_o.float().abs()).all())
    assert bool(((lse - ref_l).abs() <= LSE_ATOL).all())
