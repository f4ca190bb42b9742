"""The C-ABI library loads, exports every function include/pka.h declares, and
rejects invalid arguments on the host (no GPU needed for any of this)."""

import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_attention_32_gb300 import _lib as L
from paged_kv_attention_32_gb300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pka.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M))
                  - {"if", "defined"})


def test_header_declares_the_binding_symbols():
    assert set(_declared()) == set(L.EXPORTED)


@pytest.mark.parametrize("name", _declared())
def test_library_exports_symbol(name):
    lib = ctypes.CDLL(L.LIB_PATH)
    assert hasattr(lib, name)


def test_version_string():
    assert b"sm_103a" in L.lib().pka_version()


def _plan(**kw):
    args = dict(num_qo_heads=8, num_kv_heads=2, page_size=16, max_pages_per_seq=20,
                num_pages=100, num_sms=8, host_only=True)
    args.update(kw)
    seq = args.pop("seq", [100, 50])
    return api.paged_decode_plan(seq, **args)


@pytest.mark.parametrize("kw,code", [
    (dict(num_qo_heads=6, num_kv_heads=4), L.PKA_ERR_INVALID_ARG),      # Hq % Hkv
    (dict(head_dim=64), L.PKA_ERR_UNSUPPORTED),                         # D != 128
    (dict(page_size=8), L.PKA_ERR_UNSUPPORTED),
    (dict(seq=[100, 0]), L.PKA_ERR_INVALID_ARG),                        # kv_len 0
    (dict(seq=[3, 50], q_len=4), L.PKA_ERR_INVALID_ARG),                # kv_len < q_len
    (dict(seq=[400, 50]), L.PKA_ERR_INVALID_ARG),                       # > C * page_size
    (dict(q_len=2, max_q_len=3), L.PKA_ERR_INVALID_ARG),                # fixed: max != q_len
    (dict(qo_indptr=[0, 2, 5], max_q_len=2), L.PKA_ERR_INVALID_ARG),    # above capacity
    (dict(qo_indptr=[0, 2, 5], q_len=3, max_q_len=4), L.PKA_ERR_INVALID_ARG),  # alias clash
    (dict(qo_indptr=[1, 2, 5]), L.PKA_ERR_INVALID_ARG),
    (dict(qo_indptr=[0, 2, 2]), L.PKA_ERR_INVALID_ARG),                 # empty packed request
    (dict(window_left=-2), L.PKA_ERR_INVALID_ARG),
    (dict(num_qo_heads=256, num_kv_heads=1, q_len=257, seq=[300, 300]),
     L.PKA_ERR_UNSUPPORTED),                                            # 65792 rows per KV head
])
def test_plan_rejects(kw, code):
    with pytest.raises(L.PkaError) as ei:
        _plan(**kw)
    assert ei.value.code == code


@pytest.mark.parametrize("Hq,Hkv,q_len,tiles", [(128, 1, 1, 8), (64, 1, 2, 8), (16, 2, 16, 8),
                                                (256, 1, 4, 64)])
def test_plan_accepts_wide_groups(Hq, Hkv, q_len, tiles):
    """More than 64 query rows per KV head (MQA with many heads, long q_len_per_req):
    the tensor-core kernel with one CTA per 16-row tile of each work item."""
    p = _plan(num_qo_heads=Hq, num_kv_heads=Hkv, q_len=q_len, seq=[100, 50])
    info = p.info
    assert info["kernel"] == L.PKA_KERNEL_MMA
    assert -(-info["rows_per_cta"] // 16) == tiles


def test_plan_accepts_packed_and_reports_total_rows():
    p = _plan(qo_indptr=[0, 2, 5], causal=True)
    assert p.info["total_q"] == 5


def test_run_rejects_host_only_plan_and_null_pointers():
    p = _plan()
    rc = L.lib().paged_decode_run(p.handle, None, 0, 0, None, None, 0, 0, None, 0, None, None,
                                  None, None, None, 0, None)
    assert rc == L.PKA_ERR_INVALID_ARG


def test_step_host_checks_its_arguments_before_any_device_work():
    """paged_decode_step_host: a NULL io, a host-only plan and NULL buffers are
    rejected on the host, and the plan is left as it was (not re-planned)."""
    p = _plan()
    before = p.export()
    seq = (ctypes.c_int32 * 2)(300, 20)
    io = L.DecodeHostIO(seq_lens_kv_host=ctypes.cast(seq, ctypes.c_void_p).value,
                        bt_row_stride=20)
    ws = ctypes.c_size_t(0)
    lib = L.lib()
    assert lib.paged_decode_step_host(p.handle, 2, None, None, None, 0, 0, None, None, 0,
                                      ctypes.byref(ws), 1, None) == L.PKA_ERR_INVALID_ARG
    assert lib.paged_decode_step_host(p.handle, 2, ctypes.byref(io), None, None, 0, 0, None,
                                      None, 0, ctypes.byref(ws), 1, None) == L.PKA_ERR_INVALID_ARG
    assert b"HOST_ONLY" in lib.pka_last_error()
    assert p.export() == before


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), L.PKA_ERR_UNSUPPORTED),
    (dict(window_left=-2), L.PKA_ERR_INVALID_ARG),
    (dict(num_qo_heads=6, num_kv_heads=4), L.PKA_ERR_INVALID_ARG),
])
def test_prefill_plan_rejects(kw, code):
    args = dict(num_qo_heads=8, num_kv_heads=2, host_only=True)
    args.update(kw)
    with pytest.raises(L.PkaError) as ei:
        api.batch_prefill_plan([0, 10, 30], [0, 10, 30], **args)
    assert ei.value.code == code


def test_prefill_plan_rejects_causal_kv_shorter_than_q():
    with pytest.raises(L.PkaError):
        api.batch_prefill_plan([0, 10], [0, 5], num_qo_heads=2, num_kv_heads=1, host_only=True)


def test_prefill_tiles_heaviest_first():
    p = api.batch_prefill_plan([0, 300, 310], [0, 300, 310], num_qo_heads=4, num_kv_heads=1,
                               host_only=True)
    # 3 q-tiles for request 0 + 1 for request 1, one CTA per query head each
    assert p.num_tiles == (3 + 1) * 4


def test_merge_rejects_bad_head_dim():
    rc = L.lib().attn_merge_lse(None, None, 1, 1, 1, 6, None, 0, None, None)
    assert rc == L.PKA_ERR_INVALID_ARG


def test_prefill_fixed_plan_tiles_and_bound_checks():
    """Fixed-shape prefill: B * ceil(Sq / 128) q-tiles per query head; variable_window
    bounds must satisfy 0 <= start <= end < Sk and come only with that mask."""
    p = api.batch_prefill_plan_fixed(2, 200, 300, num_qo_heads=8, num_kv_heads=2, host_only=True)
    assert p.num_tiles == 2 * 2 * 8
    st = np.zeros((2, 200), np.int32)
    en = np.full((2, 200), 299, np.int32)
    api.batch_prefill_plan_fixed(2, 200, 300, num_qo_heads=8, num_kv_heads=2,
                                 mask_type="variable_window", variable_window_token_starts=st,
                                 variable_window_token_ends=en, host_only=True)
    bad = [dict(mask_type="variable_window", variable_window_token_starts=st,
                variable_window_token_ends=en + 1),
           dict(mask_type="variable_window", variable_window_token_starts=st + 5,
                variable_window_token_ends=en * 0 + 4),
           dict(mask_type="variable_window"),
           dict(mask_type="causal", variable_window_token_starts=st, variable_window_token_ends=en)]
    for kw in bad:
        with pytest.raises(L.PkaError) as ei:
            api.batch_prefill_plan_fixed(2, 200, 300, num_qo_heads=8, num_kv_heads=2,
                                         host_only=True, **kw)
        assert ei.value.code == L.PKA_ERR_INVALID_ARG
