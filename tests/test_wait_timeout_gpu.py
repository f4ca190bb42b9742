"""The bounded wait every kernel uses gives up, reports, and leaves the context
usable (no trap, no hang): a warp waits on a barrier phase nothing completes."""
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
