"""fp64 reference arithmetic for paged decode, LSE merge and ragged prefill.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Sources (FlashInfer API documentation pages):

* ``flashinfer.attention.prims_ts.batch_decode_with_paged_kv_cache`` --
  parameters ``block_tables``, ``seq_lens_kv``, ``qo_indptr``,
  ``mask_type``, ``window_left``, ``bmm1_scale``/``bmm2_scale``.
* ``flashinfer.cudnn.cudnn_batch_decode_with_kv_cache`` -- parameters
  ``k_cache``/``v_cache`` (HND page pools), ``scale``, ``q_len_per_req``
  (bottom-right causal rows), ``window_left``, ``sinks``, and the Note's
  "LSE convention" (base-2 log-sum-exp over the valid KV positions, GQA
  head map ``h // (num_heads_qo // num_heads_kv)``).
* ``flashinfer.attention.prims_ts.batch_prefill`` -- packed ``qo_indptr`` /
  ``kv_indptr``, bottom-right causal mask, ``sm_scale`` default
  ``1/sqrt(head_dim)``, ``output_scale``.

Everything here is the plain definition: gather the keys a row may see,
score them, take the softmax, weight the values.  No blocking, no online
softmax, no splitting.  All arithmetic is float64.
"""

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


# ---------------------------------------------------------------------------
# bf16 storage <-> float64
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits):
    """Widen bf16 values, given as their uint16 bit patterns, to float64.

    A bf16 number is the upper 16 bits of an IEEE float32, so placing the
    pattern in the upper half of a 32-bit word gives the float32 with the same
    value, and float32 -> float64 is exact.
    """
    b = np.asarray(bits).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # NaN payloads widen to NaN
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits):
    """Widen IEEE binary16 values, given as uint16 bit patterns, to float64.

    ``cudnn_batch_decode_with_kv_cache`` takes ``torch.float16`` as well as
    ``torch.bfloat16`` inputs.  Written from the format's definition: sign bit
    15, exponent bits 10-14 (bias 15), fraction bits 0-9; exponent 0 is
    subnormal ``f / 2^10 * 2^-14``, exponent 31 is infinity (f = 0) or NaN.
    """
    b = np.asarray(bits).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    sub = np.ldexp(f / 1024.0, -14)
    out = np.where(e == 0, sub, normal)
    out = np.where(e == 31, np.where(f == 0, np.inf, np.nan), out)
    return sign * out


def bits_to_f64(bits, dtype="bf16"):
    """Input values of dtype ``'bf16'`` or ``'f16'`` (uint16 bit patterns) as float64."""
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    raise ValueError(f"unknown input dtype {dtype!r}")


# ---------------------------------------------------------------------------
# Paged K/V addressing
# ---------------------------------------------------------------------------

def gather_kv(pages_bits, block_table_row, page_size, kv_head, start, stop, dtype="bf16"):
    """Rows ``start .. stop-1`` of one request's K (or V) for one KV head, float64.

    ``pages_bits`` is the HND page pool ``[num_pages, num_kv_heads, page_size,
    head_dim]`` as bf16 bit patterns (``cudnn_batch_decode_with_kv_cache``,
    parameters ``k_cache``/``v_cache``).  Token ``t`` of the request lives in
    page ``block_table_row[t // page_size]`` at slot ``t % page_size``
    (``batch_decode_with_paged_kv_cache``, parameter ``block_tables``).
    """
    t = np.arange(start, stop, dtype=np.int64)
    page = np.asarray(block_table_row, dtype=np.int64)[t // page_size]
    return bits_to_f64(pages_bits[page, kv_head, t % page_size, :], dtype)


def decode_row_key_range(kv_len, q_len, i, causal, window_left):
    """Keys ``[lo, hi)`` that query row ``i`` of a request may attend to.

    * Bottom-right causal diagonal: row ``i`` of a request with ``q_len`` rows
      and ``kv_len`` keys sees keys ``0 .. kv_len - q_len + i``
      (``cudnn_batch_decode_with_kv_cache``, parameter ``q_len_per_req``).
    * Left window: the row keeps the ``window_left`` keys before its diagonal
      position plus that position itself; ``-1`` disables the window
      (same page, parameter ``window_left``).
    * Dense mask (no causal cut): keys up to ``kv_len - 1``.  With a window the
      window is anchored at the same diagonal position (the pages do not
      define a window without a causal diagonal; this is the plain reading).
    """
    d = kv_len - q_len + i
    hi = d + 1 if causal else kv_len
    lo = max(0, d - window_left) if window_left >= 0 else 0
    return lo, hi


# ---------------------------------------------------------------------------
# Softmax attention of a set of query rows over one key set
# ---------------------------------------------------------------------------

def attention_rows(q_rows, keys, values, allowed, scale, sink=None, out_scale=1.0):
    """Plain softmax attention for query rows ``q_rows`` ``[R, D]``.

    ``allowed[r, j]`` says whether row ``r`` may see key ``j``.  For each row:

    * ``s_j = scale * q . k_j`` over the allowed keys;
    * the optional ``sink`` logit joins the softmax denominator as one more
      term with a zero value row (``cudnn_batch_decode_with_kv_cache``,
      parameter ``sinks``);
    * ``o = out_scale * sum_j softmax_j * v_j``;
    * ``lse = log2(sum_j exp(s_j))`` over the allowed keys only -- the sink
      is not a KV position (same page, Note "LSE convention").

    Returns ``(o [R, D], lse [R])``.  A row with no allowed key gives
    ``o = 0`` when there is no sink (and ``lse = -inf``).
    """
    R = q_rows.shape[0]
    D = values.shape[1]
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    if keys.shape[0] == 0:
        return o, lse
    scores = scale * (q_rows @ keys.T)                      # [R, n]
    for r in range(R):
        sel = allowed[r]
        s = scores[r, sel]
        v = values[sel]
        if s.size == 0:
            continue
        m_keys = s.max()
        lse[r] = LOG2E * (m_keys + math.log(np.exp(s - m_keys).sum()))
        m = m_keys if sink is None else max(m_keys, sink)
        w = np.exp(s - m)
        z = w.sum() + (0.0 if sink is None else math.exp(sink - m))
        o[r] = out_scale * (w @ v) / z
    return o, lse


# ---------------------------------------------------------------------------
# Paged decode
# ---------------------------------------------------------------------------

def paged_decode_request(b, q_bits, k_pages_bits, v_pages_bits, block_tables, seq_lens_kv,
                         q_start, q_len, num_kv_heads, page_size, causal=False,
                         window_left=-1, scale=None, bmm2_scale=1.0, sinks=None, dtype="bf16"):
    """Decode output of request ``b``: ``(O [q_len, Hq, D], LSE [q_len, Hq])``.

    ``q_bits`` is the packed query ``[total_q, Hq, D]`` (bit patterns of
    ``dtype``, ``'bf16'`` or ``'f16'``, like the K/V pools); the
    request's rows are ``q_start .. q_start + q_len - 1``
    (``batch_decode_with_paged_kv_cache``, parameter ``qo_indptr``).  Query
    head ``h`` reads KV head ``h // (Hq // Hkv)`` (GQA,
    ``cudnn_batch_decode_with_kv_cache`` Note).  ``scale`` defaults to
    ``1/sqrt(D)``; ``bmm2_scale`` multiplies the output only.
    """
    Hq, D = q_bits.shape[1], q_bits.shape[2]
    if Hq % num_kv_heads != 0:
        raise ValueError("num_heads_qo must be a multiple of num_heads_kv")
    group = Hq // num_kv_heads
    kv_len = int(seq_lens_kv[b])
    if kv_len < q_len:
        raise ValueError("every request needs kv_len >= q_len")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q = bits_to_f64(q_bits[q_start:q_start + q_len], dtype)        # [L, Hq, D]
    O = np.zeros((q_len, Hq, D), dtype=np.float64)
    LSE = np.zeros((q_len, Hq), dtype=np.float64)
    ranges = [decode_row_key_range(kv_len, q_len, i, causal, window_left) for i in range(q_len)]
    first = min(lo for lo, _ in ranges)
    last = max(hi for _, hi in ranges)
    for hk in range(num_kv_heads):
        K = gather_kv(k_pages_bits, block_tables[b], page_size, hk, first, last, dtype)
        V = gather_kv(v_pages_bits, block_tables[b], page_size, hk, first, last, dtype)
        keys = np.arange(first, last)
        allowed = np.stack([(keys >= lo) & (keys < hi) for lo, hi in ranges])   # [L, n]
        for g in range(group):
            h = hk * group + g
            sink = None if sinks is None else float(sinks[h])
            o, lse = attention_rows(q[:, h, :], K, V, allowed, scale, sink, bmm2_scale)
            O[:, h, :] = o
            LSE[:, h] = lse
    return O, LSE


def paged_decode(q_bits, k_pages_bits, v_pages_bits, block_tables, seq_lens_kv, num_kv_heads,
                 page_size, qo_indptr=None, q_len=1, causal=False, window_left=-1, scale=None,
                 bmm2_scale=1.0, sinks=None, requests=None, dtype="bf16"):
    """Paged decode over a batch: ``(O [total_q, Hq, D], LSE [total_q, Hq])``.

    Without ``qo_indptr`` every request has ``q_len`` consecutive rows
    (fixed multi-token query, ``batch_decode_with_paged_kv_cache``, parameter
    ``seq_len_q``); with it, request ``b`` owns rows
    ``qo_indptr[b] .. qo_indptr[b+1]-1`` (packed query).  ``requests`` limits
    the work to a subset of requests; rows of other requests are NaN.
    """
    B = len(seq_lens_kv)
    total_q, Hq, D = q_bits.shape
    if qo_indptr is None:
        qo_indptr = [b * q_len for b in range(B + 1)]
    O = np.full((total_q, Hq, D), np.nan)
    LSE = np.full((total_q, Hq), np.nan)
    for b in (range(B) if requests is None else requests):
        s0, s1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        o, lse = paged_decode_request(b, q_bits, k_pages_bits, v_pages_bits, block_tables,
                                      seq_lens_kv, s0, s1 - s0, num_kv_heads, page_size,
                                      causal, window_left, scale, bmm2_scale, sinks, dtype)
        O[s0:s1] = o
        LSE[s0:s1] = lse
    return O, LSE


# ---------------------------------------------------------------------------
# Merge of partial attention states by their base-2 LSE
# ---------------------------------------------------------------------------

def merge_states(v_states, s_states):
    """Merge ``N`` partial attention results of the same rows.

    ``v_states [N, S, H, D]`` are normalised partial outputs, each over a
    disjoint key subset, and ``s_states [N, S, H]`` their base-2 LSEs.  The
    softmax over the union of the subsets weights state ``i`` by
    ``2**s_i / sum_k 2**s_k``, and the union's LSE is ``log2(sum_i 2**s_i)``
    (``cudnn_batch_decode_with_kv_cache``, Note "LSE convention": the base-2
    LSE is what the cascade-merge kernels take).  Rows whose states are all
    ``-inf`` give ``v = 0`` and ``s = -inf``.
    """
    v = np.asarray(v_states, dtype=np.float64)
    s = np.asarray(s_states, dtype=np.float64)
    N, S, H, D = v.shape
    v_out = np.zeros((S, H, D))
    s_out = np.full((S, H), -np.inf)
    for si in range(S):
        for h in range(H):
            ls = s[:, si, h]
            m = ls.max()
            if m == -np.inf:
                continue
            w = np.power(2.0, ls - m)
            v_out[si, h] = (w[:, None] * v[:, si, h, :]).sum(axis=0) / w.sum()
            s_out[si, h] = m + math.log2(w.sum())
    return v_out, s_out


# ---------------------------------------------------------------------------
# Ragged causal prefill
# ---------------------------------------------------------------------------

def prefill_request(b, q_bits, k_bits, v_bits, qo_indptr, kv_indptr, num_kv_heads, causal=True,
                    sm_scale=None, output_scale=1.0, heads=None, rows=None, window_left=-1,
                    window_bounds=None, dtype="bf16"):
    """Prefill output of request ``b``: ``(O [Lq, Hq, D], LSE [Lq, Hq])``.

    Packed storage: request ``b`` owns query rows ``qo_indptr[b] ..
    qo_indptr[b+1]-1`` and K/V rows ``kv_indptr[b] .. kv_indptr[b+1]-1``
    (``batch_prefill``, parameters ``qo_indptr``/``kv_indptr``).  Causal
    masking is bottom-right aligned, so query row ``i`` sees keys
    ``0 .. Lk - Lq + i``.  ``sm_scale`` defaults to ``1/sqrt(D)`` and
    ``output_scale`` multiplies the output.  ``heads``/``rows`` restrict the
    computation to a subset (others are NaN).  ``window_left`` (``batch_prefill``
    lists it; the page's head-paired policy for it is undefined, so this is the
    plain sliding window of the decode pages): row ``i`` keeps the keys from
    ``Lk - Lq + i - window_left`` on, as ``decode_row_key_range`` states.
    ``window_bounds = (starts, ends)`` selects ``mask_type='variable_window'``
    instead: row ``i`` sees exactly keys ``starts[i] .. ends[i]`` (inclusive
    per-query bounds, ``variable_window_token_starts`` / ``_ends``).
    """
    Hq, D = q_bits.shape[1], q_bits.shape[2]
    group = Hq // num_kv_heads
    q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
    k0, k1 = int(kv_indptr[b]), int(kv_indptr[b + 1])
    Lq, Lk = q1 - q0, k1 - k0
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    heads = range(Hq) if heads is None else heads
    rows = np.arange(Lq) if rows is None else np.asarray(rows)
    O = np.full((Lq, Hq, D), np.nan)
    LSE = np.full((Lq, Hq), np.nan)
    keys = np.arange(Lk)
    allowed = np.zeros((len(rows), Lk), dtype=bool)
    for r, i in enumerate(rows):
        if window_bounds is not None:
            lo, hi = int(window_bounds[0][i]), int(window_bounds[1][i]) + 1
        else:
            lo, hi = decode_row_key_range(Lk, Lq, int(i), causal, window_left)
        allowed[r] = (keys >= lo) & (keys < hi)
    for h in heads:
        hk = h // group
        Q = bits_to_f64(q_bits[q0 + rows, h, :], dtype)
        K = bits_to_f64(k_bits[k0:k1, hk, :], dtype)
        V = bits_to_f64(v_bits[k0:k1, hk, :], dtype)
        o, lse = attention_rows(Q, K, V, allowed, sm_scale, None, output_scale)
        O[rows, h, :] = o
        LSE[rows, h] = lse
    return O, LSE


def batch_prefill(q_bits, k_bits, v_bits, qo_indptr, kv_indptr, num_kv_heads, causal=True,
                  sm_scale=None, output_scale=1.0, window_left=-1, window_starts=None,
                  window_ends=None, dtype="bf16"):
    """Ragged prefill over the whole batch: ``(O [total_q, Hq, D], LSE [total_q, Hq])``.

    ``window_starts`` / ``window_ends`` (``[B, Sq]``, fixed-shape batches only,
    as ``batch_prefill`` restricts ``variable_window``) give each query row its
    inclusive key bounds; ``causal`` and ``window_left`` are then unused.
    """
    total_q, Hq, D = q_bits.shape
    O = np.zeros((total_q, Hq, D))
    LSE = np.zeros((total_q, Hq))
    for b in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        bounds = None
        if window_starts is not None:
            bounds = (np.asarray(window_starts)[b], np.asarray(window_ends)[b])
        o, lse = prefill_request(b, q_bits, k_bits, v_bits, qo_indptr, kv_indptr, num_kv_heads,
                                 causal, sm_scale, output_scale, window_left=window_left,
                                 window_bounds=bounds, dtype=dtype)
        O[q0:q1] = o
        LSE[q0:q1] = lse
    return O, LSE
