"""The device status word: kernels report instead of trapping.  The bounded wait
every kernel uses gives up, reports, and leaves the context usable (a warp waits on
a barrier phase nothing completes); paged_decode_check_tables reports a block-table
entry outside the pool among the entries a run reads."""
import pytest
import torch

from helpers import assert_close, decode_plan_for, oracle_decode, run_decode
from paged_kv_attention_32_gb300 import _lib as L
from paged_kv_attention_32_gb300 import api
from paged_kv_attention_32_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_wait_gives_up_and_sets_the_timeout_bit():
    status = api.wait_timeout_probe(limit_ns=20_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) & 1 == 1


def test_plan_check_reports_a_wait_timeout_then_runs_normally():
    w = wl.shrink(wl.LLAMA3_8B_DECODE, batch=3, kv_len_range=(300, 900), pool_pages=400,
                  table_width=64, return_lse=True)
    inp = wl.make_decode_inputs(w, seed=21, device=DEV)
    plan = decode_plan_for(inp, num_sms=16)
    api.wait_timeout_probe(limit_ns=20_000_000, plan=plan)
    with pytest.raises(L.PkaError) as exc:
        plan.check()
    assert exc.value.code == L.PKA_ERR_DEVICE_TIMEOUT
    plan.check()   # the word was cleared by the read
    # the context and the plan still work
    out, lse, _ = run_decode(inp, plan=plan)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)
    plan.check()


def test_probe_rejects_limits_outside_the_documented_range():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bad in (0, 999_999, 2_000_000_001):
        with pytest.raises(L.PkaError):
            api.wait_timeout_probe(limit_ns=bad, status=status)


@pytest.mark.parametrize("name", ["llama3_8b", "spec"])
def test_check_tables_reports_a_page_outside_the_pool(name):
    base = {"llama3_8b": wl.shrink(wl.LLAMA3_8B_DECODE, batch=3, kv_len_range=(300, 900),
                                   pool_pages=400, table_width=64, return_lse=True),
            "spec": wl.shrink(wl.SPEC_DECODE, batch=3, kv_len_range=(2048, 3000),
                              table_width=400)}[name]
    inp = wl.make_decode_inputs(base, seed=22, device=DEV)
    plan = decode_plan_for(inp, num_sms=16)
    plan.check_tables(inp["block_tables"])
    plan.check()                                   # a valid table passes
    P = inp["k_pages"].shape[0]
    bad = inp["block_tables"].clone()
    bad[1, int(inp["seq_lens_kv"][1].item() - 1) // inp["page_size"]] = P + 3   # a visited page
    plan.check_tables(bad)
    with pytest.raises(L.PkaError) as exc:
        plan.check()
    assert exc.value.code == L.PKA_ERR_DEVICE_BOUNDS
    plan.check()                                   # the report was cleared
    # entries the run does not read (past the request's pages) are not checked
    loose = inp["block_tables"].clone()
    n1 = (int(inp["seq_lens_kv"][1].item()) + inp["page_size"] - 1) // inp["page_size"]
    if n1 < loose.shape[1]:
        loose[1, n1:] = -7
        plan.check_tables(loose)
        plan.check()
    out, lse, _ = run_decode(inp, plan=plan)
    ref_o, ref_l = oracle_decode(inp)
    assert_close(out, lse, ref_o, ref_l)
