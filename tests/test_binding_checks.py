"""The Python binding rejects layouts the C ABI cannot see (checked on the host,
before any call into the library): a strided head dimension, V laid out unlike K,
non-dense page slots or table rows, non-contiguous outputs."""
import pytest
import torch

from paged_kv_attention_32_gb300 import api

BF = torch.bfloat16


def _decode_plan():
    seq = torch.tensor([40, 17], dtype=torch.int32)
    return api.paged_decode_plan(seq, num_qo_heads=4, num_kv_heads=2, page_size=16,
                                 max_pages_per_seq=4, num_pages=8, q_len=1, num_sms=8,
                                 host_only=True)


def _decode_inputs():
    q = torch.zeros((2, 4, 128), dtype=BF)
    k = torch.zeros((8, 2, 16, 128), dtype=BF)
    v = torch.zeros((8, 2, 16, 128), dtype=BF)
    bt = torch.zeros((2, 4), dtype=torch.int32)
    return q, k, v, bt


def test_decode_rejects_a_strided_head_dimension():
    plan = _decode_plan()
    q, k, v, bt = _decode_inputs()
    q_bad = torch.zeros((2, 4, 256), dtype=BF)[:, :, ::2]
    with pytest.raises(ValueError, match="dense last"):
        api.paged_decode_run(plan, q_bad, k, v, bt)


def test_decode_rejects_v_strided_unlike_k():
    plan = _decode_plan()
    q, k, _, bt = _decode_inputs()
    v_wide = torch.zeros((8, 3, 16, 128), dtype=BF)[:, :2]   # another page stride
    v_other = torch.zeros((8, 2, 16, 128 * 2), dtype=BF)[..., :128]   # another slot stride
    with pytest.raises(ValueError):
        api.paged_decode_run(plan, q, k, v_other, bt)
    with pytest.raises(ValueError, match="shape and strides of k"):
        api.paged_decode_run(plan, q, k, v_wide, bt)


def test_decode_rejects_non_dense_page_slots_and_table_rows():
    plan = _decode_plan()
    q, _, _, bt = _decode_inputs()
    k = torch.zeros((8, 2, 16, 256), dtype=BF)[..., :128]   # slot stride 256, not 128
    with pytest.raises(ValueError, match="dense rows"):
        api.paged_decode_run(plan, q, k, k, bt)
    q, k, v, _ = _decode_inputs()
    bt_bad = torch.zeros((2, 8), dtype=torch.int32)[:, ::2]
    with pytest.raises(ValueError, match="block_tables"):
        api.paged_decode_run(plan, q, k, v, bt_bad)


def test_decode_rejects_non_contiguous_outputs():
    plan = _decode_plan()
    q, k, v, bt = _decode_inputs()
    out = torch.zeros((4, 2, 128), dtype=BF).transpose(0, 1)
    with pytest.raises(ValueError, match="out must be contiguous"):
        api.paged_decode_run(plan, q, k, v, bt, out=out)


def test_prefill_rejects_bad_layouts():
    qi = torch.tensor([0, 5, 9], dtype=torch.int32)
    plan = api.batch_prefill_plan(qi, qi, num_qo_heads=4, num_kv_heads=2, host_only=True)
    q = torch.zeros((9, 4, 128), dtype=BF)
    k = torch.zeros((9, 2, 128), dtype=BF)
    with pytest.raises(ValueError, match="dense last"):
        api.batch_prefill_run(plan, q, torch.zeros((9, 2, 256), dtype=BF)[..., ::2], k)
    with pytest.raises(ValueError, match="shape and strides of k"):
        api.batch_prefill_run(plan, q, k, torch.zeros((9, 3, 128), dtype=BF)[:, :2])
    with pytest.raises(ValueError, match="lse must be contiguous"):
        api.batch_prefill_run(plan, q, k, k, lse=torch.zeros((4, 9)).t())


def test_host_io_wants_host_and_device_tensors_where_stated():
    """DecodeHostIO: host buffers on the CPU, staging buffers on the device, int32
    tables and lengths, matching host/device shapes (checked before any CUDA use)."""
    q = torch.zeros((2, 4, 128), dtype=BF)
    bt = torch.zeros((2, 4), dtype=torch.int32)
    seq = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        api.DecodeHostIO(q_host=q, block_tables_host=bt, seq_lens_kv_host=seq, out_host=q.clone(),
                         q_dev=q.clone(), block_tables_dev=bt.clone(), out_dev=q.clone())
    with pytest.raises(ValueError, match="int32"):
        api.DecodeHostIO(q_host=q, block_tables_host=bt.long(), seq_lens_kv_host=seq,
                         out_host=q.clone(), q_dev=q.clone(), block_tables_dev=bt.clone(),
                         out_dev=q.clone())


def test_host_io_in_place_needs_pinned_memory():
    """A device slot of DecodeHostIO may be its host tensor only when that is pinned
    (checked before any GPU work; plain CPU tensors are never pinned)."""
    q = torch.zeros((4, 8, 128), dtype=torch.bfloat16)
    bt = torch.zeros((4, 4), dtype=torch.int32)
    seq = torch.ones(4, dtype=torch.int32)
    out = torch.zeros_like(q)
    with pytest.raises(ValueError, match="pinned"):
        api.DecodeHostIO(q_host=q, block_tables_host=bt, seq_lens_kv_host=seq, out_host=out,
                         q_dev=q, block_tables_dev=bt, out_dev=out)
