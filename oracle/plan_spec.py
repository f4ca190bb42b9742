"""Written specification of the split-KV decode plan, restated in plain Python.

TEST INFRASTRUCTURE ONLY: the C++ planner of the product library must produce
exactly these arrays; this file shares no code with it.

The pages fix only what the plan is for: the one-shot planner reads
``seq_lens_kv`` on the host to derive exact bounds, and a plan made before CUDA
graph capture keeps the run path capturable (``batch_decode_with_paged_kv_cache``,
description paragraph on the planner).  How the key range is cut into chunks is
a design choice of this library, stated here:

1. Request ``b`` has ``n = kv_len_b`` keys and ``L = q_len_b`` query rows.  Its
   first visited key is ``kv_lo = max(0, n - L - window_left)`` when the window
   is on and the plan freezes the lengths, else 0 (the window's left edge of
   row 0 -- rows below see later keys only).  Pages visited:
   ``[kv_lo // ps, ceil(n / ps))``, ``np_b`` of them.
2. CTAs per work item: ``t_b = ceil(group * L_b / 16)`` when the tensor-core
   kernel runs (one CTA per 16-row tile of the group's query rows; it runs when
   ``group * max L >= mma_min_rows`` or ``> 8``), else 1.  Target CTA count
   ``T = waves * num_sms``.  If ``Hkv * sum_b t_b >= T`` no request is split:
   the chunk is ``max_b np_b`` pages.  Otherwise the chunk ``c`` is the smallest
   integer in ``[min(c_min, max np), max np]`` with
   ``Hkv * sum_b t_b * ceil(np_b / c) <= T``, where ``c_min = ceil(min_chunk_tokens / ps)``.
3. ``n_chunks_b = ceil(np_b / c)``, except for the tail of a launch that does
   not split (``Hkv * sum_b t_b >= T``): with ``S = r * num_sms`` resident CTAs
   (``r`` = 3 for the tensor-core kernel, 2 for the CUDA-core kernel), walk the
   requests longest first and let the prefix whose CTAs ``Hkv * t_b`` sum to at
   most ``S`` be the first wave; the remaining requests (``R`` CTAs) start only
   as the first wave ends, so each is cut into ``k = S // R`` chunks of
   ``c_b = max(ceil(np_b / k), min(c_min, np_b))`` pages (``n_chunks_b =
   ceil(np_b / c_b)``) when ``k > 1``, so that they run as one short round on
   all SMs.  With the tensor-core kernel and one 16-row tile per request
   (``group * max L <= 16``), every request longer than 3/5 of the average
   load of a resident slot, ``A = Hkv * sum_b np_b / S`` pages (in integers:
   ``np_b * 5S > 3 Hkv sum np``), is also cut into ``p_b = ceil(5 S np_b /
   (3 Hkv sum np))`` parts: ``c_b = min(c_b, max(ceil(np_b / p_b), min(c_min,
   np_b)))``.  Requests are visited longest first
   (``np_b`` descending, ties by ``b`` ascending); for each, chunks in order,
   and for each chunk every KV head: one work item
   ``(b, kv_head, chunk, page_lo, page_hi)``.
4. Requests with ``n_chunks_b > 1`` are "split": in ``b`` order each gets a base
   row ``part_base_b`` in the fp32 partial buffers, holding
   ``n_chunks_b * L * Hq`` partial rows (index ``(chunk * L + i) * Hq + h``).
   Unsplit requests write the final output directly (``part_base_b = -1``).
5. Workspace: the partial outputs ``[rows, D]`` fp32 at offset 0, padded to a
   256-byte multiple, then the partial base-2 LSEs ``[rows]`` fp32.
"""


def _ceil_div(a, b):
    return -(-a // b)


def plan_spec(seq_lens_kv, q_lens, num_qo_heads, num_kv_heads, head_dim, page_size,
              window_left, num_sms, waves, min_chunk_tokens, freeze_seq_lens=True,
              mma_min_rows=1):
    """Return the plan as a dict of plain Python lists and ints (see module docstring)."""
    B = len(seq_lens_kv)
    page_lo, page_hi, npages = [], [], []
    for b in range(B):
        n, L = int(seq_lens_kv[b]), int(q_lens[b])
        kv_lo = max(0, n - L - window_left) if (window_left >= 0 and freeze_seq_lens) else 0
        lo = kv_lo // page_size
        hi = _ceil_div(n, page_size)
        page_lo.append(lo)
        page_hi.append(hi)
        npages.append(hi - lo)
    group = num_qo_heads // num_kv_heads
    rows = group * max(int(x) for x in q_lens)
    mma = rows >= mma_min_rows or rows > 8
    tiles = [_ceil_div(group * int(q_lens[b]), 16) if mma else 1 for b in range(B)]
    max_np = max(npages)
    target = waves * num_sms
    if num_kv_heads * sum(tiles) >= target:
        chunk = max_np
    else:
        c_min = _ceil_div(min_chunk_tokens, page_size)
        chunk = max_np
        for c in range(min(c_min, max_np), max_np + 1):
            if num_kv_heads * sum(t * _ceil_div(x, c) for t, x in zip(tiles, npages)) <= target:
                chunk = c
                break
    order = sorted(range(B), key=lambda b: (-npages[b], b))
    cb = [chunk] * B
    if num_kv_heads * sum(tiles) >= target:
        slots = (3 if mma else 2) * num_sms
        acc, tail = 0, []
        for b in order:
            if not tail and acc + num_kv_heads * tiles[b] <= slots:
                acc += num_kv_heads * tiles[b]
            else:
                tail.append(b)
        rest = num_kv_heads * sum(tiles[b] for b in tail)
        k = slots // rest if rest else 1
        c_min = _ceil_div(min_chunk_tokens, page_size)
        if k > 1:
            for b in tail:
                cb[b] = max(_ceil_div(npages[b], k), min(c_min, npages[b]))
        if mma and rows <= 16:   # one tile per request: cut past 3/5 of a slot's load
            load = num_kv_heads * sum(npages)
            for b in range(B):
                num, den = npages[b] * 5 * slots, 3 * load
                if num > den:
                    parts = _ceil_div(num, den)
                    cb[b] = min(cb[b], max(_ceil_div(npages[b], parts), min(c_min, npages[b])))
    n_chunks = [_ceil_div(x, c) for x, c in zip(npages, cb)]
    items = []
    for b in order:
        for ci in range(n_chunks[b]):
            lo = page_lo[b] + ci * cb[b]
            hi = min(page_lo[b] + (ci + 1) * cb[b], page_hi[b])
            for hk in range(num_kv_heads):
                items.append((b, hk, ci, lo, hi))
    part_base, rows = [], 0
    for b in range(B):
        if n_chunks[b] > 1:
            part_base.append(rows)
            rows += n_chunks[b] * int(q_lens[b]) * num_qo_heads
        else:
            part_base.append(-1)
    o_bytes = rows * head_dim * 4
    o_bytes_padded = _ceil_div(o_bytes, 256) * 256
    workspace = o_bytes_padded + rows * 4 if rows else 0
    return {
        "chunk_pages": chunk,
        "page_lo": page_lo,
        "page_hi": page_hi,
        "n_chunks": n_chunks,
        "order": order,
        "items": items,
        "part_base": part_base,
        "partial_rows": rows,
        "workspace_bytes": workspace,
    }
