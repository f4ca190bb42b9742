"""Python binding of the C ABI, same names as ``include/pka.h``.

Argument marshalling only: tensors are turned into device pointers, strides
and sizes, outputs are allocated with torch when the caller passes none, and
every computation happens in ``libpka.so``.  There is no CPU path.
"""

import ctypes
import math

import torch

from . import _lib as L


def _stream(stream):
    """cudaStream_t as an int (ctypes passes ints to void* parameters as is)."""
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


_DTYPES = {torch.bfloat16: L.PKA_DTYPE_BF16, torch.float16: L.PKA_DTYPE_F16,
           torch.float32: L.PKA_DTYPE_F32}
_TORCH = {v: k for k, v in _DTYPES.items()}


def _dtype_codes(dtype, out_dtype):
    """(input code, output code) of torch dtypes; the output defaults to the input type."""
    if dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"q/K/V dtype must be bfloat16 or float16, got {dtype}")
    out_dtype = dtype if out_dtype is None else out_dtype
    if out_dtype not in _DTYPES:
        raise ValueError(f"out_dtype must be bfloat16, float16 or float32, got {out_dtype}")
    return _DTYPES[dtype], _DTYPES[out_dtype]


def _check_inputs(plan, *tensors):
    want = _TORCH[plan.desc.dtype]
    for t in tensors:
        if t.dtype != want:
            raise ValueError(f"the plan was made for {want} inputs, got {t.dtype}")


def _check_layout(q, k, v, out=None, lse=None, paged=False):
    """What the C ABI assumes but cannot see: the head dim dense (stride 1), V
    laid out like K (the ABI takes one set of K/V strides), a paged pool's slots
    dense rows of D, and contiguous outputs."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a dense last (head) dimension")
    if tuple(v.stride()) != tuple(k.stride()) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("v must have the shape and strides of k")
    if paged and k.stride(2) != k.shape[3]:
        raise ValueError("each page's slots must be dense rows of head_dim elements")
    for name, t in (("out", out), ("lse", lse)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def _host_i32(x):
    """Contiguous host int32 array (kept alive by the caller) and its pointer."""
    if x is None:
        return None, None
    if (isinstance(x, torch.Tensor) and x.dtype == torch.int32 and x.device.type == "cpu"
            and x.is_contiguous()):
        t = x
    else:
        t = torch.as_tensor(x).to(device="cpu", dtype=torch.int32).contiguous()
    return t, ctypes.cast(t.data_ptr(), L._pi32)


class DecodePlan:
    """Owns a ``pka_plan*``; freed with ``paged_decode_plan_destroy``."""

    def __init__(self, handle, desc, workspace_bytes):
        self.handle = handle
        self.desc = desc
        self.workspace_bytes = workspace_bytes

    @property
    def info(self):
        inf = L.PlanInfo()
        L.check(L.lib().paged_decode_plan_info(self.handle, ctypes.byref(inf)), "plan_info")
        return {f: getattr(inf, f) for f, _ in L.PlanInfo._fields_}

    def export(self):
        """Host arrays of the plan: items (n, 5), n_chunks, part_base, page_lo, page_hi, order."""
        n = self.info["num_items"]
        B = self.desc.batch_size
        items = torch.zeros(max(n, 1) * 5, dtype=torch.int32)
        arrs = [torch.zeros(B, dtype=torch.int32) for _ in range(5)]
        ptrs = [ctypes.cast(a.data_ptr(), L._pi32) for a in [items] + arrs]
        L.check(L.lib().paged_decode_plan_export(self.handle, *ptrs), "plan_export")
        keys = ["n_chunks", "part_base", "page_lo", "page_hi", "order"]
        out = {k: a.tolist() for k, a in zip(keys, arrs)}
        out["items"] = [tuple(r) for r in items[: n * 5].view(n, 5).tolist()]
        return out

    def update(self, seq_lens_kv, qo_indptr=None, stream=None):
        """Re-plan in place for a new batch (``paged_decode_plan_update``): new host
        lengths (and packed offsets), same heads, masks and options."""
        seq_t, seq_p = _host_i32(seq_lens_kv)
        ind_t, ind_p = _host_i32(qo_indptr)
        ws = ctypes.c_size_t()
        host_only = bool(self.desc.flags & L.PKA_PLAN_HOST_ONLY)
        rc = L.lib().paged_decode_plan_update(self.handle, seq_t.numel(), seq_p, ind_p,
                                              ctypes.byref(ws),
                                              None if host_only else _stream(stream))
        L.check(rc, "paged_decode_plan_update")
        self.desc.batch_size = seq_t.numel()
        self.workspace_bytes = ws.value
        return self

    def check(self, stream=None):
        """Synchronise and read the device status word (raises on a kernel timeout, or
        on a bad block-table entry found by ``check_tables``)."""
        L.check(L.lib().paged_decode_plan_check(self.handle, _stream(stream)), "plan_check")

    def check_tables(self, block_tables, seq_lens_kv=None, stream=None):
        """Validate on the device the block-table entries a run of this plan reads
        (``paged_decode_check_tables``); ``check()`` then raises on a bad one."""
        if block_tables.stride(-1) != 1:
            raise ValueError("block_tables rows must be dense")
        rc = L.lib().paged_decode_check_tables(self.handle, _ptr(block_tables),
                                               block_tables.stride(0), _ptr(seq_lens_kv),
                                               _stream(stream))
        L.check(rc, "paged_decode_check_tables")

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            L.lib().paged_decode_plan_destroy(h)


def paged_decode_plan(seq_lens_kv, *, num_qo_heads, num_kv_heads, page_size, max_pages_per_seq,
                      num_pages, qo_indptr=None, q_len=1, max_q_len=0, causal=False,
                      window_left=-1, scale=None, bmm2_scale=1.0, return_lse=False,
                      freeze_seq_lens=True, num_sms=0, split_waves=0, min_chunk_tokens=0,
                      mma_min_rows=0, host_only=False, head_dim=128, dtype=torch.bfloat16,
                      out_dtype=None, stream=None):
    """Plan a batched paged decode from host copies of the lengths (see pka.h).
    ``dtype``: q and the K/V pools (bfloat16 or float16); ``out_dtype``: O (bfloat16,
    float16 or float32; default ``dtype``)."""
    in_code, out_code = _dtype_codes(dtype, out_dtype)
    seq_t, seq_p = _host_i32(seq_lens_kv)
    ind_t, ind_p = _host_i32(qo_indptr)
    d = L.DecodeDesc(
        batch_size=seq_t.numel(), num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, page_size=page_size, max_pages_per_seq=max_pages_per_seq,
        num_pages=num_pages, dtype=in_code, out_dtype=out_code, q_len=q_len, max_q_len=max_q_len,
        mask=L.PKA_MASK_CAUSAL if causal else L.PKA_MASK_DENSE, window_left=window_left,
        scale=float("nan") if scale is None else scale, bmm2_scale=bmm2_scale,
        return_lse=int(bool(return_lse)), freeze_seq_lens=int(bool(freeze_seq_lens)),
        num_sms=num_sms, split_waves=split_waves, min_chunk_tokens=min_chunk_tokens,
        mma_min_rows=mma_min_rows, flags=L.PKA_PLAN_HOST_ONLY if host_only else 0)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    rc = L.lib().paged_decode_plan(ctypes.byref(h), ctypes.byref(d), seq_p, ind_p,
                                   ctypes.byref(ws), _stream(stream) if not host_only else None)
    L.check(rc, "paged_decode_plan")
    return DecodePlan(h, d, ws.value)


def paged_decode_run(plan, q, k_pages, v_pages, block_tables, seq_lens_kv=None, sinks=None,
                     out=None, lse=None, workspace=None, stream=None):
    """Run a planned decode; returns ``out`` (and ``lse`` when the plan returns it)."""
    _check_inputs(plan, q, k_pages, v_pages)
    _check_layout(q, k_pages, v_pages, out, lse, paged=True)
    if block_tables.stride(-1) != 1:
        raise ValueError("block_tables rows must be dense")
    if out is not None and out.dtype != _TORCH[plan.desc.out_dtype]:
        raise ValueError(f"out must be {_TORCH[plan.desc.out_dtype]} (the plan's out_dtype)")
    total_q, Hq, D = q.shape
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=_TORCH[plan.desc.out_dtype], device=q.device)
    if plan.desc.return_lse and lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if workspace is None and plan.workspace_bytes > 0:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = L.lib().paged_decode_run(
        plan.handle, _ptr(q), q.stride(0), q.stride(1), _ptr(k_pages), _ptr(v_pages),
        k_pages.stride(0), k_pages.stride(1), _ptr(block_tables), block_tables.stride(0),
        _ptr(seq_lens_kv), _ptr(sinks), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        _stream(stream))
    L.check(rc, "paged_decode_run")
    return (out, lse) if plan.desc.return_lse else out


class DecodeHostIO:
    """Host and device buffers of ``paged_decode_step_host`` (``pka_decode_host_io``).

    Host tensors (CPU, pinned for asynchronous copies) hold each step's q, block
    table rows and key lengths and receive O (and the LSE); device tensors of the
    same shapes are the staging copies the run reads and writes.  A device slot may
    be given its host tensor itself when that is pinned: the run then reads or
    writes the host memory in place and the step copies nothing for it.  The
    buffers are sized for the largest batch; a step uses their leading rows.  The
    object keeps every tensor alive and a workspace that grows when a re-plan
    needs more."""

    def __init__(self, q_host, block_tables_host, seq_lens_kv_host, out_host, q_dev,
                 block_tables_dev, out_dev, lse_host=None, lse_dev=None, seq_lens_kv_dev=None,
                 qo_indptr_host=None):
        host = dict(q_host=q_host, block_tables_host=block_tables_host,
                    seq_lens_kv_host=seq_lens_kv_host, out_host=out_host, lse_host=lse_host,
                    qo_indptr_host=qo_indptr_host)
        dev = dict(q_dev=q_dev, block_tables_dev=block_tables_dev, out_dev=out_dev,
                   lse_dev=lse_dev, seq_lens_kv_dev=seq_lens_kv_dev)
        for name, t in host.items():
            if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CPU tensor")
        for name in ("block_tables_host", "seq_lens_kv_host", "qo_indptr_host",
                     "block_tables_dev", "seq_lens_kv_dev"):
            t = host.get(name, dev.get(name))
            if t is not None and t.dtype != torch.int32:
                raise ValueError(f"{name} must be int32")
        for name, t in dev.items():
            h = host.get(name[:-4] + "_host")
            if t is not None and h is not None and t is h:   # in place: pinned host memory
                if not h.is_pinned():
                    raise ValueError(f"{name} may be {name[:-4]}_host itself only when that "
                                     "tensor is pinned")
                continue
            if t is not None and (t.device.type != "cuda" or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
        pairs = (("q", q_host, q_dev), ("block_tables", block_tables_host, block_tables_dev),
                 ("out", out_host, out_dev), ("lse", lse_host, lse_dev))
        for name, h, d in pairs:
            if h is not None and d is not None and (h.shape != d.shape or h.dtype != d.dtype):
                raise ValueError(f"{name}_host and {name}_dev must have one shape and dtype")
        if q_host.shape != out_host.shape:
            raise ValueError("out must have the shape of q")
        self.tensors = dict(host, **dev)
        self.workspace = None
        self.c = L.DecodeHostIO(bt_row_stride=block_tables_host.stride(0),
                                **{k: _ptr(v) for k, v in self.tensors.items()})


def paged_decode_step_host(plan, io, k_pages, v_pages, sinks=None, batch_size=None,
                           synchronize=True, stream=None):
    """One decode step from host buffers (``paged_decode_step_host``): copy q / tables
    (/ lengths) in, re-plan on the lengths in ``io``, run, copy O (/ LSE) out; arrays
    the io gives in place are read or written where they are.  With ``synchronize``
    the host outputs are ready on return."""
    t = io.tensors
    _check_inputs(plan, t["q_host"], k_pages, v_pages)
    _check_layout(t["q_dev"], k_pages, v_pages, t["out_dev"], t["lse_dev"], paged=True)
    if t["out_dev"].dtype != _TORCH[plan.desc.out_dtype]:
        raise ValueError(f"out must be {_TORCH[plan.desc.out_dtype]} (the plan's out_dtype)")
    B = t["seq_lens_kv_host"].numel() if batch_size is None else int(batch_size)
    if B > t["block_tables_host"].shape[0] or B > t["seq_lens_kv_host"].numel():
        raise ValueError("batch_size exceeds the io's table rows or lengths")
    ind = t["qo_indptr_host"]
    total_q = int(ind[B]) if ind is not None else B * plan.desc.q_len
    if total_q > t["q_host"].shape[0]:
        raise ValueError(f"the batch has {total_q} query rows, the io holds {t['q_host'].shape[0]}")
    lib = L.lib()
    ws_need = ctypes.c_size_t()
    for attempt in range(2):
        ws = io.workspace
        ws_bytes = 0 if ws is None else ws.numel()
        rc = lib.paged_decode_step_host(
            plan.handle, B, ctypes.byref(io.c), _ptr(k_pages), _ptr(v_pages), k_pages.stride(0),
            k_pages.stride(1), _ptr(sinks), _ptr(ws), ws_bytes, ctypes.byref(ws_need),
            int(bool(synchronize)), _stream(stream))
        if rc in (L.PKA_OK, L.PKA_ERR_WORKSPACE_TOO_SMALL):   # the plan was re-planned
            plan.desc.batch_size = B
            plan.workspace_bytes = ws_need.value
        if rc != L.PKA_ERR_WORKSPACE_TOO_SMALL or attempt == 1:
            break
        io.workspace = torch.empty(ws_need.value + ws_need.value // 4 + 256, dtype=torch.uint8,
                                   device=k_pages.device)
    L.check(rc, "paged_decode_step_host")
    return (t["out_host"], t["lse_host"]) if plan.desc.return_lse else t["out_host"]


class DecodeStep:
    """``paged_decode_step_host`` prepared for a serving loop that repeats it on one
    plan, io, pair of pools and stream: the binding's checks of the tensors run once
    here, and each call is a single C-ABI call with its arguments already marshalled
    (the library still checks them all on every call).  A call runs one step on the
    current contents of the io's host arrays (lengths, offsets, q, tables) and returns
    what ``paged_decode_step_host`` returns.  The batch size is fixed here (a batch of
    another size needs another DecodeStep); the lengths and the io's packed offsets may
    change between calls, and the offsets' row count is checked against the io's q rows
    each time."""

    def __init__(self, plan, io, k_pages, v_pages, sinks=None, batch_size=None,
                 synchronize=True, stream=None):
        t = io.tensors
        _check_inputs(plan, t["q_host"], k_pages, v_pages)
        _check_layout(t["q_dev"], k_pages, v_pages, t["out_dev"], t["lse_dev"], paged=True)
        if t["out_dev"].dtype != _TORCH[plan.desc.out_dtype]:
            raise ValueError(f"out must be {_TORCH[plan.desc.out_dtype]} (the plan's out_dtype)")
        B = t["seq_lens_kv_host"].numel() if batch_size is None else int(batch_size)
        if B < 1 or B > t["block_tables_host"].shape[0] or B > t["seq_lens_kv_host"].numel():
            raise ValueError("batch_size must be >= 1 and within the io's table rows and lengths")
        ind = t["qo_indptr_host"]
        if ind is not None and ind.numel() < B + 1:
            raise ValueError("qo_indptr_host holds fewer than batch_size + 1 offsets")
        self.plan, self.io, self.batch_size = plan, io, B
        self._keep = (k_pages, v_pages, sinks)
        self._rows = t["q_host"].shape[0]
        self._ind = None if ind is None else ctypes.cast(ind.data_ptr(), L._pi32)
        if self._ind is None and B * plan.desc.q_len > self._rows:
            raise ValueError(f"the batch has {B * plan.desc.q_len} query rows, the io holds "
                             f"{self._rows}")
        self._fn = L.lib().paged_decode_step_host
        self._need = ctypes.c_size_t()
        self._head = (plan.handle, B, ctypes.byref(io.c), _ptr(k_pages), _ptr(v_pages),
                      k_pages.stride(0), k_pages.stride(1), _ptr(sinks))
        self._tail = (ctypes.byref(self._need), int(bool(synchronize)), _stream(stream))
        self._result = (t["out_host"], t["lse_host"]) if plan.desc.return_lse else t["out_host"]
        self._bind_workspace()

    def _bind_workspace(self):
        ws = self.io.workspace
        self._args = self._head + (_ptr(ws), 0 if ws is None else ws.numel()) + self._tail

    def __call__(self):
        if self._ind is not None and self._ind[self.batch_size] > self._rows:
            raise ValueError(f"the batch has {self._ind[self.batch_size]} query rows, the io "
                             f"holds {self._rows}")
        rc = self._fn(*self._args)
        if rc == L.PKA_ERR_WORKSPACE_TOO_SMALL:   # re-planned, not run: grow and step again
            need = self._need.value
            self.io.workspace = torch.empty(need + need // 4 + 256, dtype=torch.uint8,
                                            device=self._keep[0].device)
            self._bind_workspace()
            rc = self._fn(*self._args)
        if rc in (L.PKA_OK, L.PKA_ERR_WORKSPACE_TOO_SMALL):   # the plan was re-planned
            self.plan.desc.batch_size = self.batch_size
            self.plan.workspace_bytes = self._need.value
        L.check(rc, "paged_decode_step_host")
        return self._result


def attn_merge_lse(v_states, s_states, out_dtype=torch.bfloat16, v_out=None, s_out=None,
                   stream=None):
    """Merge ``[N, S, H, D]`` fp32 states by their ``[N, S, H]`` base-2 LSEs."""
    N, S, H, D = v_states.shape
    if v_out is None:
        v_out = torch.empty((S, H, D), dtype=out_dtype, device=v_states.device)
    if s_out is None:
        s_out = torch.empty((S, H), dtype=torch.float32, device=v_states.device)
    code = _DTYPES[v_out.dtype]
    rc = L.lib().attn_merge_lse(_ptr(v_states), _ptr(s_states), N, S, H, D, _ptr(v_out), code,
                                _ptr(s_out), _stream(stream))
    L.check(rc, "attn_merge_lse")
    return v_out, s_out


class PrefillPlan:
    """Owns a ``pka_prefill_plan*``."""

    def __init__(self, handle, desc, num_tiles):
        self.handle = handle
        self.desc = desc
        self.num_tiles = num_tiles

    def check(self, stream=None):
        L.check(L.lib().batch_prefill_plan_check(self.handle, _stream(stream)), "prefill_check")

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            L.lib().batch_prefill_plan_destroy(h)


def batch_prefill_plan(qo_indptr, kv_indptr, *, num_qo_heads, num_kv_heads, causal=True,
                       sm_scale=None, output_scale=1.0, return_lse=False, head_dim=128,
                       window_left=-1, host_only=False, dtype=torch.bfloat16, out_dtype=None,
                       stream=None):
    """Plan a packed ragged prefill from host copies of the indptr arrays (``dtype`` /
    ``out_dtype`` as for ``paged_decode_plan``)."""
    in_code, out_code = _dtype_codes(dtype, out_dtype)
    qo_t, qo_p = _host_i32(qo_indptr)
    kv_t, kv_p = _host_i32(kv_indptr)
    d = L.PrefillDesc(
        batch_size=qo_t.numel() - 1, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, dtype=in_code, out_dtype=out_code,
        mask=L.PKA_MASK_CAUSAL if causal else L.PKA_MASK_DENSE, window_left=window_left,
        sm_scale=float("nan") if sm_scale is None else sm_scale, output_scale=output_scale,
        return_lse=int(bool(return_lse)), num_sms=0,
        flags=L.PKA_PLAN_HOST_ONLY if host_only else 0)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    nt = ctypes.c_int32()
    rc = L.lib().batch_prefill_plan(ctypes.byref(h), ctypes.byref(d), qo_p, kv_p,
                                    ctypes.byref(ws), ctypes.byref(nt),
                                    _stream(stream) if not host_only else None)
    L.check(rc, "batch_prefill_plan")
    return PrefillPlan(h, d, nt.value)


def batch_prefill_plan_fixed(batch_size, seq_len_q, seq_len_kv, *, num_qo_heads, num_kv_heads,
                             mask_type="causal", window_left=-1,
                             variable_window_token_starts=None, variable_window_token_ends=None,
                             sm_scale=None, output_scale=1.0, return_lse=False, head_dim=128,
                             host_only=False, dtype=torch.bfloat16, out_dtype=None, stream=None):
    """Plan a fixed-shape prefill: q ``[B, Sq, Hq, D]``, k/v ``[B, Sk, Hkv, D]`` (run it with
    ``batch_prefill_run`` on the tensors viewed as ``[B*S, H, D]``).  ``mask_type``:
    ``'causal'``, ``'dense'`` or ``'variable_window'`` (inclusive per-query key bounds
    ``[B, Sq]``; host copies are taken here for planning)."""
    masks = {"dense": L.PKA_MASK_DENSE, "causal": L.PKA_MASK_CAUSAL,
             "variable_window": L.PKA_MASK_VARIABLE_WINDOW}
    in_code, out_code = _dtype_codes(dtype, out_dtype)
    st_t, st_p = _host_i32(variable_window_token_starts)
    en_t, en_p = _host_i32(variable_window_token_ends)
    d = L.PrefillDesc(
        batch_size=batch_size, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, dtype=in_code, out_dtype=out_code, mask=masks[mask_type],
        window_left=window_left,
        sm_scale=float("nan") if sm_scale is None else sm_scale, output_scale=output_scale,
        return_lse=int(bool(return_lse)), num_sms=0,
        flags=L.PKA_PLAN_HOST_ONLY if host_only else 0)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    nt = ctypes.c_int32()
    rc = L.lib().batch_prefill_plan_fixed(ctypes.byref(h), ctypes.byref(d), seq_len_q, seq_len_kv,
                                          st_p, en_p, ctypes.byref(ws), ctypes.byref(nt),
                                          _stream(stream) if not host_only else None)
    L.check(rc, "batch_prefill_plan_fixed")
    return PrefillPlan(h, d, nt.value)


def batch_prefill_run(plan, q, k, v, out=None, lse=None, stream=None):
    """Run a planned prefill; returns ``out`` (and ``lse`` when the plan returns it).
    Packed ``[total, H, D]`` tensors, or fixed-shape ``[B, S, H, D]`` ones (viewed as
    ``[B*S, H, D]``; ``out``/``lse`` then come back as ``[B, Sq, Hq, D]``/``[B, Sq, Hq]``)."""
    fixed = q.dim() == 4
    if fixed:
        B, Sq = q.shape[0], q.shape[1]
        q, k, v = q.flatten(0, 1), k.flatten(0, 1), v.flatten(0, 1)
        if out is not None:
            out = out.view(B * Sq, *out.shape[2:])
        if lse is not None:
            lse = lse.view(B * Sq, lse.shape[2])
        res = batch_prefill_run(plan, q, k, v, out=out, lse=lse, stream=stream)
        if plan.desc.return_lse:
            return res[0].view(B, Sq, *res[0].shape[1:]), res[1].view(B, Sq, res[1].shape[1])
        return res.view(B, Sq, *res.shape[1:])
    _check_inputs(plan, q, k, v)
    _check_layout(q, k, v, out, lse)
    if out is not None and out.dtype != _TORCH[plan.desc.out_dtype]:
        raise ValueError(f"out must be {_TORCH[plan.desc.out_dtype]} (the plan's out_dtype)")
    total_q, Hq, D = q.shape
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=_TORCH[plan.desc.out_dtype], device=q.device)
    if plan.desc.return_lse and lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    rc = L.lib().batch_prefill_run(plan.handle, _ptr(q), q.stride(0), q.stride(1), _ptr(k),
                                   _ptr(v), k.stride(0), k.stride(1), _ptr(out), _ptr(lse),
                                   None, 0, _stream(stream))
    L.check(rc, "batch_prefill_run")
    return (out, lse) if plan.desc.return_lse else out


def paged_kv_gather(pages, block_tables, request, kv_head, tok_begin, tok_end, out=None,
                    stream=None):
    """Dense copy of paged rows ``[tok_begin, tok_end)`` through the decode addressing."""
    P, Hkv, ps, D = pages.shape
    if out is None:
        out = torch.empty((tok_end - tok_begin, D), dtype=pages.dtype, device=pages.device)
    rc = L.lib().paged_kv_gather(_ptr(pages), P, pages.stride(0), pages.stride(1), Hkv, ps, D,
                                 _ptr(block_tables), block_tables.stride(0), request, kv_head,
                                 tok_begin, tok_end, _ptr(out), _stream(stream))
    L.check(rc, "paged_kv_gather")
    return out


def default_scale(head_dim=128):
    return 1.0 / math.sqrt(head_dim)


def wait_timeout_probe(limit_ns=10_000_000, plan=None, status=None, stream=None):
    """Run the kernels' bounded wait on a barrier nothing completes until it gives
    up after ``limit_ns``.  The timeout bit (1) goes into ``plan``'s status word
    (its ``check()`` then raises) or, without a plan, into ``status`` (a device
    int32 tensor, made when not given), which is returned."""
    if plan is None and status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.lib().pka_wait_timeout_probe(plan.handle if plan is not None else None,
                                        _ptr(status), int(limit_ns), _stream(stream))
    L.check(rc, "pka_wait_timeout_probe")
    return status
