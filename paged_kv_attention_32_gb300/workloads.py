"""Seeded synthetic inputs for paged decode and ragged prefill.

This module holds no attention arithmetic: it only draws lengths, page tables
and N(0, 1) bf16 tensors.  It is the one module that both the CUDA path's
callers (tests, bench) and the fp64 oracle's callers use, so both sides see
the same inputs.

Recipe (all seeds explicit):

* lengths, query lengths and the page permutation come from a CPU
  ``torch.Generator`` seeded with ``seed``;
* q, K/V pools, sinks come from a ``torch.Generator`` on the target device
  seeded with ``seed + 1`` (bf16 ``N(0, 1)``; sinks fp32 ``N(0, 1)``).  The
  values therefore depend on the device the inputs are drawn on; every test
  draws once and hands the same tensors to both sides.
* the K/V pool holds ``pool_pages`` pages; every request draws the pages it
  needs, without replacement, from one random permutation of the pool;
  unused ``block_tables`` slots hold -1 and are never read.
* "climbing" inputs (``climbing_keys``, ``aligned_queries``) replace the
  N(0, 1) keys and queries with keys whose component along one random unit
  direction grows linearly with the key's position, and queries close to that
  direction: every row's scores then rise towards its last keys.  Values and
  lengths are drawn as above; the extra draws use a CPU generator seeded
  with ``seed + 2``.
"""

from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_len_range: tuple            # inclusive uniform range for every request
    q_len_range: tuple = (1, 1)    # inclusive uniform range of query rows per request
    packed_q: bool = False         # qo_indptr given (packed query)
    causal: bool = False
    window_left: int = -1
    sinks: bool = False
    return_lse: bool = True
    fixed_first_kv_len: Optional[int] = None   # request 0's length, if pinned
    pool_pages: Optional[int] = None           # None: pages needed * (1 + pool_slack)
    pool_slack: float = 0.10
    table_width: Optional[int] = None          # C; None: enough for the longest request
    bmm2_scale: float = 1.0


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    len_range: tuple
    causal: bool = True
    output_scale: float = 1.0


# The five synthetic workloads: four decode shapes and one ragged prefill.
TINY_DECODE = DecodeWorkload(
    name="tiny paged decode B=4 Hq=8 Hkv=2 D=128 ps=16 kv_len U[1,300]",
    batch=4, num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
    kv_len_range=(1, 300), pool_pages=96, table_width=19)

LLAMA3_8B_DECODE = DecodeWorkload(
    name="Llama-3-8B-shaped paged decode B=64 Hq=32 Hkv=8 D=128 ps=16 kv_len U[512,8192]",
    batch=64, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
    kv_len_range=(512, 8192), pool_pages=40000, table_width=512, return_lse=False)

SKEWED_DECODE = DecodeWorkload(
    name="skewed long-context paged decode B=16 (one kv_len=131072, others U[1024,4096]) "
         "Hq=64 Hkv=8 D=128 ps=32",
    batch=16, num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=32,
    kv_len_range=(1024, 4096), fixed_first_kv_len=131072, table_width=4096)

SPEC_DECODE = DecodeWorkload(
    name="speculative packed-Q paged decode B=32 q_len U[1,6] causal window_left=4095 sinks "
         "Hq=64 Hkv=8 D=128 ps=16 kv_len U[2048,16384]",
    batch=32, num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=16,
    kv_len_range=(2048, 16384), q_len_range=(1, 6), packed_q=True, causal=True,
    window_left=4095, sinks=True, table_width=1024)

RAGGED_PREFILL = PrefillWorkload(
    name="ragged causal batch_prefill B=8 len U[512,8192] Hq=32 Hkv=8 D=128",
    batch=8, num_qo_heads=32, num_kv_heads=8, head_dim=128, len_range=(512, 8192))

DECODE_WORKLOADS = {
    "tiny": TINY_DECODE,
    "llama3_8b": LLAMA3_8B_DECODE,
    "skewed": SKEWED_DECODE,
    "spec": SPEC_DECODE,
}


def shrink(w, **kw):
    """A smaller copy of a workload with the same structure (for oracle-sized tests)."""
    return replace(w, **kw)


def _randint(gen, lo, hi, n):
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, device="cpu", dtype=torch.bfloat16):
    """Draw one batch of decode inputs for workload ``w``.

    Returns a dict of tensors (q, k_pages, v_pages, block_tables, seq_lens_kv,
    qo_indptr or None, q_lens, sinks or None) plus the scalar parameters.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B = w.batch
    kv = _randint(g, w.kv_len_range[0], w.kv_len_range[1], B)
    if w.fixed_first_kv_len is not None:
        kv[0] = w.fixed_first_kv_len
    ql = _randint(g, w.q_len_range[0], w.q_len_range[1], B)
    kv = torch.maximum(kv, ql)            # every request needs kv_len >= q_len
    ps = w.page_size
    need = (kv + ps - 1) // ps
    total_need = int(need.sum())
    pool = w.pool_pages if w.pool_pages is not None else int(total_need * (1.0 + w.pool_slack)) + 1
    if pool < total_need:
        raise ValueError(f"pool of {pool} pages cannot hold {total_need} pages")
    C = w.table_width if w.table_width is not None else int(need.max())
    if int(need.max()) > C:
        raise ValueError("block table too narrow for the longest request")
    perm = torch.randperm(pool, generator=g, dtype=torch.int64)
    tables = torch.full((B, C), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(need[b])
        tables[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    if w.packed_q:
        qo_indptr = torch.zeros(B + 1, dtype=torch.int32)
        qo_indptr[1:] = torch.cumsum(ql, 0).to(torch.int32)
        total_q = int(qo_indptr[-1])
    else:
        ql = torch.full((B,), int(w.q_len_range[0]), dtype=torch.int64)
        kv = torch.maximum(kv, ql)
        qo_indptr = None
        total_q = B * int(w.q_len_range[0])

    gd = torch.Generator(device=device)
    gd.manual_seed(seed + 1)
    shape_pool = (pool, w.num_kv_heads, ps, w.head_dim)
    k_pages = torch.randn(shape_pool, generator=gd, device=device, dtype=dtype)
    v_pages = torch.randn(shape_pool, generator=gd, device=device, dtype=dtype)
    q = torch.randn((total_q, w.num_qo_heads, w.head_dim), generator=gd, device=device,
                    dtype=dtype)
    sinks = (torch.randn((w.num_qo_heads,), generator=gd, device=device, dtype=torch.float32)
             if w.sinks else None)
    return {
        "q": q,
        "k_pages": k_pages,
        "v_pages": v_pages,
        "block_tables": tables.to(device),
        "seq_lens_kv": kv.to(torch.int32).to(device),
        "q_lens": ql.to(torch.int32),
        "qo_indptr": qo_indptr.to(device) if qo_indptr is not None else None,
        "sinks": sinks,
        "num_kv_heads": w.num_kv_heads,
        "page_size": ps,
        "q_len": int(w.q_len_range[0]) if not w.packed_q else None,
        "causal": w.causal,
        "window_left": w.window_left,
        "return_lse": w.return_lse,
        "bmm2_scale": w.bmm2_scale,
    }


def make_prefill_inputs(w: PrefillWorkload, seed: int = 0, device="cpu"):
    """Draw one batch of packed ragged prefill inputs (qo_indptr == kv_indptr)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    lens = _randint(g, w.len_range[0], w.len_range[1], w.batch)
    indptr = torch.zeros(w.batch + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(lens, 0).to(torch.int32)
    total = int(indptr[-1])
    gd = torch.Generator(device=device)
    gd.manual_seed(seed + 1)
    q = torch.randn((total, w.num_qo_heads, w.head_dim), generator=gd, device=device,
                    dtype=torch.bfloat16)
    k = torch.randn((total, w.num_kv_heads, w.head_dim), generator=gd, device=device,
                    dtype=torch.bfloat16)
    v = torch.randn((total, w.num_kv_heads, w.head_dim), generator=gd, device=device,
                    dtype=torch.bfloat16)
    return {
        "q": q, "k": k, "v": v,
        "qo_indptr": indptr.to(device), "kv_indptr": indptr.to(device),
        "lens": lens.to(torch.int32),
        "num_kv_heads": w.num_kv_heads,
        "causal": w.causal,
        "output_scale": w.output_scale,
    }


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a 16-bit (bf16 or f16) tensor, as a numpy array (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def climbing_keys(positions, num_heads, u, slope, gen, noise=0.25):
    """Key rows whose component along the unit direction ``u`` grows with the key's
    position: row p is ``(slope * p) * u + noise * N(0, 1)`` for every head
    (float32 on the CPU, ``[len(positions), num_heads, D]``).  With queries close to
    ``u``, each query row's largest scores sit at its last keys, so the running row
    maximum climbs from one key tile to the next."""
    pos = torch.as_tensor(positions, dtype=torch.float32)
    D = u.numel()
    rows = torch.randn((pos.numel(), num_heads, D), generator=gen, dtype=torch.float32) * noise
    return rows + (slope * pos)[:, None, None] * u.to(torch.float32)[None, None, :]


def aligned_queries(num_rows, num_heads, u, gen, noise=0.05):
    """Query rows ``a_h * u + noise * N(0, 1)``, one factor ``a_h`` in [1, 1.25] per
    head (float32 on the CPU, ``[num_rows, num_heads, D]``)."""
    a = 1.0 + 0.25 * torch.rand((num_heads,), generator=gen, dtype=torch.float32)
    D = u.numel()
    rows = torch.randn((num_rows, num_heads, D), generator=gen, dtype=torch.float32) * noise
    return rows + a[None, :, None] * u.to(torch.float32)[None, None, :]


def unit_direction(head_dim, gen):
    """A random unit vector of ``head_dim`` components (float32 on the CPU)."""
    u = torch.randn((head_dim,), generator=gen, dtype=torch.float64)
    return (u / u.norm()).to(torch.float32)


def make_climbing_decode_inputs(w: DecodeWorkload, seed: int = 0, device="cpu",
                                dtype=torch.bfloat16, slope=1.5):
    """Decode inputs of workload ``w`` (lengths, tables, V, sinks as ``make_decode_inputs``
    draws them) whose keys climb along one direction with the token index and whose
    queries point along it (``climbing_keys``, ``aligned_queries``): the scores of every
    row rise towards its last keys, so the chunks of a split request end with partial
    LSEs far apart."""
    inp = make_decode_inputs(w, seed=seed, device=device, dtype=dtype)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 2)
    u = unit_direction(w.head_dim, g)
    ps = w.page_size
    tables = inp["block_tables"].cpu().to(torch.int64)
    seq = inp["seq_lens_kv"].cpu().to(torch.int64)
    kp = inp["k_pages"].cpu().to(torch.float32)
    for b in range(w.batch):
        t = torch.arange(int(seq[b]), dtype=torch.int64)
        pages = tables[b, t // ps]
        kp[pages, :, t % ps, :] = climbing_keys(t, w.num_kv_heads, u, slope, g)
    inp["k_pages"] = kp.to(dtype).to(device)
    q = inp["q"]
    inp["q"] = aligned_queries(q.shape[0], q.shape[1], u, g).to(dtype).to(device)
    return inp
