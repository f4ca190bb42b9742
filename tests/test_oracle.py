"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test ties one part of the oracle to a closed form, an invariant of the
definition, or an independent library routine (torch's fp64
``scaled_dot_product_attention``, ``logsumexp``, ``tril``/``triu`` masks),
so that a dropped term, a wrong sign or index, or a transposed operand in
the oracle fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import LOG2E, bf16_bits_to_f64
from paged_kv_attention_32_gb300 import workloads as wl


def _bits(t):
    return wl.bf16_bits(t)


def _rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _pool_from_dense(dense_list, page_size, pool_pages, seed):
    """Scatter per-request dense K ``[n_b, H, D]`` into a shuffled HND page pool.

    Built page-block by page-block with reshape/permute, not token by token,
    so it does not restate the oracle's per-token address formula.
    """
    H, D = dense_list[0].shape[1], dense_list[0].shape[2]
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(pool_pages, generator=g)
    pool = _rand_bf16((pool_pages, H, page_size, D), seed + 7)
    width = max((x.shape[0] + page_size - 1) // page_size for x in dense_list)
    table = torch.full((len(dense_list), width), -1, dtype=torch.int32)
    off = 0
    for b, x in enumerate(dense_list):
        n = x.shape[0]
        npg = (n + page_size - 1) // page_size
        padded = torch.zeros((npg * page_size, H, D), dtype=torch.bfloat16)
        padded[:n] = x
        blocks = padded.reshape(npg, page_size, H, D).permute(0, 2, 1, 3)   # [npg, H, ps, D]
        ids = perm[off:off + npg]
        off += npg
        pool[ids] = blocks
        table[b, :npg] = ids.to(torch.int32)
    return pool, table


def _sdpa_reference(q, k, v, scale, mask):
    """torch fp64 SDPA for one head: q [L, D], k/v [n, D], mask [L, n] bool."""
    out = F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None],
                                         attn_mask=mask[None, None], scale=scale)
    return out[0, 0]


def _bottom_right_mask(L, n, causal, window_left):
    """Mask from torch's tril/triu: causal keeps j <= n-L+i, window keeps j >= n-L+i-W."""
    m = torch.ones((L, n), dtype=torch.bool)
    if causal:
        m = torch.tril(m, diagonal=n - L)
    if window_left >= 0:
        m = m & torch.triu(torch.ones((L, n), dtype=torch.bool), diagonal=n - L - window_left)
    return m


# ---------------------------------------------------------------------------
# bf16 widening
# ---------------------------------------------------------------------------

def test_bf16_widening_matches_torch():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (50000,), generator=g, dtype=torch.int32).to(torch.int16)
    as_bf16 = bits.view(torch.bfloat16)
    finite = torch.isfinite(as_bf16.float())
    ref = as_bf16.to(torch.float64)[finite].numpy()
    got = bf16_bits_to_f64(bits.numpy().view(np.uint16))[finite.numpy()]
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Closed forms and special cases of the decode definition
# ---------------------------------------------------------------------------

def _one_request(n, H_q, H_kv, D, ps, seed, L=1):
    k = _rand_bf16((n, H_kv, D), seed)
    v = _rand_bf16((n, H_kv, D), seed + 1)
    q = _rand_bf16((L, H_q, D), seed + 2)
    pool_pages = (n + ps - 1) // ps + 5
    kp, table = _pool_from_dense([k], ps, pool_pages, seed + 3)
    vp, table_v = _pool_from_dense([v], ps, pool_pages, seed + 3)
    assert torch.equal(table, table_v)
    return q, k, v, kp, vp, table


def test_single_key_returns_that_value_row():
    q, k, v, kp, vp, table = _one_request(1, 4, 2, 128, 16, 10)
    O, lse = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(),
                                 np.array([1]), 2, 16)
    kf, vf, qf = k.double(), v.double(), q.double()
    for h in range(4):
        assert np.allclose(O[0, h], vf[0, h // 2].numpy(), rtol=0, atol=1e-15)
        s = (qf[0, h] @ kf[0, h // 2]).item() / math.sqrt(128)
        assert lse[0, h] == pytest.approx(s * LOG2E, abs=1e-12)


def test_zero_query_gives_mean_of_values_and_log2_count():
    n = 37
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, 16, 20)
    qz = torch.zeros_like(q)
    O, lse = oracle.paged_decode(_bits(qz), _bits(kp), _bits(vp), table.numpy(),
                                 np.array([n]), 1, 16)
    mean = v.double()[:, 0].mean(0).numpy()
    for h in range(2):
        assert np.allclose(O[0, h], mean, atol=1e-13)
        assert lse[0, h] == pytest.approx(math.log2(n), abs=1e-12)


def test_identical_keys_give_uniform_weights():
    n = 23
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, 16, 30)
    k_same = k[:1].expand(n, -1, -1).contiguous()
    kp2, table2 = _pool_from_dense([k_same], 16, (n + 15) // 16 + 5, 33)
    vp2, _ = _pool_from_dense([v], 16, (n + 15) // 16 + 5, 33)
    O, _ = oracle.paged_decode(_bits(q), _bits(kp2), _bits(vp2), table2.numpy(),
                               np.array([n]), 1, 16)
    assert np.allclose(O[0, 0], v.double()[:, 0].mean(0).numpy(), atol=1e-13)


def test_lse_is_log2e_times_torch_logsumexp():
    n = 201
    q, k, v, kp, vp, table = _one_request(n, 8, 2, 128, 16, 40)
    O, lse = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(),
                                 np.array([n]), 2, 16)
    for h in range(8):
        s = (k.double()[:, h // 4] @ q.double()[0, h]) / math.sqrt(128)
        assert lse[0, h] == pytest.approx(torch.logsumexp(s, 0).item() * LOG2E, abs=1e-11)


def test_permuted_page_table_equals_identity_layout():
    n, ps = 150, 16
    q, k, v, kp, vp, table = _one_request(n, 4, 2, 128, ps, 50)
    npg = (n + ps - 1) // ps
    # identity layout: request pages stored in order 0..npg-1
    pad = torch.zeros((npg * ps, 2, 128), dtype=torch.bfloat16)
    pad[:n] = k
    kid = pad.reshape(npg, ps, 2, 128).permute(0, 2, 1, 3).contiguous()
    pad[:n] = v
    vid = pad.reshape(npg, ps, 2, 128).permute(0, 2, 1, 3).contiguous()
    ident = np.arange(npg, dtype=np.int32)[None]
    O1, l1 = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 2, ps)
    O2, l2 = oracle.paged_decode(_bits(q), _bits(kid), _bits(vid), ident, [n], 2, ps)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_page_size_repacking_is_invariant():
    n = 100
    q = _rand_bf16((1, 4, 128), 60)
    k = _rand_bf16((n, 1, 128), 61)
    v = _rand_bf16((n, 1, 128), 62)
    outs = []
    for ps in (16, 32):
        kp, t = _pool_from_dense([k], ps, (n + ps - 1) // ps + 3, 63 + ps)
        vp, _ = _pool_from_dense([v], ps, (n + ps - 1) // ps + 3, 63 + ps)
        outs.append(oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), t.numpy(), [n], 1, ps))
    assert np.allclose(outs[0][0], outs[1][0], atol=1e-14)
    assert np.allclose(outs[0][1], outs[1][1], atol=1e-12)


@pytest.mark.parametrize("causal,window_left,L", [
    (False, -1, 1), (True, -1, 1), (True, -1, 5), (True, 7, 4), (False, 9, 3), (True, 0, 3),
])
def test_matches_torch_sdpa_on_dense_gather(causal, window_left, L):
    """Brute force: gather densely (by page blocks), mask with tril/triu, torch fp64 SDPA."""
    lens = [40, 17, 64]
    Hq, Hkv, D, ps = 6, 2, 128, 16
    ks = [_rand_bf16((n, Hkv, D), 70 + i) for i, n in enumerate(lens)]
    vs = [_rand_bf16((n, Hkv, D), 80 + i) for i, n in enumerate(lens)]
    npool = sum((n + ps - 1) // ps for n in lens) + 4
    kp, table = _pool_from_dense(ks, ps, npool, 90)
    vp, _ = _pool_from_dense(vs, ps, npool, 90)
    q = _rand_bf16((L * len(lens), Hq, D), 91)
    scale = 0.37
    O, lse = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), lens, Hkv, ps,
                                 q_len=L, causal=causal, window_left=window_left, scale=scale)
    for b, n in enumerate(lens):
        mask = _bottom_right_mask(L, n, causal, window_left)
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            qq = q.double()[b * L:(b + 1) * L, h]
            ref = _sdpa_reference(qq, ks[b].double()[:, hk], vs[b].double()[:, hk], scale, mask)
            assert np.allclose(O[b * L:(b + 1) * L, h], ref.numpy(), atol=1e-12)
            s = scale * (qq @ ks[b].double()[:, hk].T)
            ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), 1) * LOG2E
            assert np.allclose(lse[b * L:(b + 1) * L, h], ref_lse.numpy(), atol=1e-11)


def test_gqa_equals_mha_with_repeated_kv_heads():
    n, ps = 50, 16
    q = _rand_bf16((1, 8, 128), 100)
    k = _rand_bf16((n, 2, 128), 101)
    v = _rand_bf16((n, 2, 128), 102)
    kp, t = _pool_from_dense([k], ps, 8, 103)
    vp, _ = _pool_from_dense([v], ps, 8, 103)
    krep = k.repeat_interleave(4, dim=1)
    vrep = v.repeat_interleave(4, dim=1)
    kp8, t8 = _pool_from_dense([krep], ps, 8, 104)
    vp8, _ = _pool_from_dense([vrep], ps, 8, 104)
    O1, l1 = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), t.numpy(), [n], 2, ps)
    O2, l2 = oracle.paged_decode(_bits(q), _bits(kp8), _bits(vp8), t8.numpy(), [n], 8, ps)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_causal_row_sees_exactly_its_keys():
    """Perturbing V rows past row i's diagonal leaves row i unchanged; the diagonal itself does not."""
    n, L, ps = 45, 4, 16
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, ps, 110, L=L)
    base, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, ps,
                                  q_len=L, causal=True)
    for i in range(L):
        d = n - L + i
        v2 = v.clone()
        v2[d + 1:] += 3.0
        vp2, _ = _pool_from_dense([v2], ps, (n + ps - 1) // ps + 5, 113)
        o2, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp2), table.numpy(), [n], 1,
                                    ps, q_len=L, causal=True)
        assert np.array_equal(o2[i], base[i])
        v3 = v.clone()
        v3[d] += 3.0
        vp3, _ = _pool_from_dense([v3], ps, (n + ps - 1) // ps + 5, 113)
        o3, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp3), table.numpy(), [n], 1,
                                    ps, q_len=L, causal=True)
        assert not np.allclose(o3[i], base[i])


def test_window_keeps_window_left_plus_one_keys():
    n, ps, W = 60, 16, 10
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, ps, 120)
    base, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, ps,
                                  window_left=W)
    first = n - 1 - W
    v2 = v.clone()
    v2[:first] += 5.0
    vp2, _ = _pool_from_dense([v2], ps, (n + ps - 1) // ps + 5, 123)
    o2, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp2), table.numpy(), [n], 1, ps,
                                window_left=W)
    assert np.array_equal(o2, base)
    v3 = v.clone()
    v3[first] += 5.0
    vp3, _ = _pool_from_dense([v3], ps, (n + ps - 1) // ps + 5, 123)
    o3, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp3), table.numpy(), [n], 1, ps,
                                window_left=W)
    assert not np.allclose(o3, base)


def test_window_at_least_kv_len_is_no_window():
    n = 33
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, 16, 130, L=3)
    a = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, 16,
                            q_len=3, causal=True)
    b = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, 16,
                            q_len=3, causal=True, window_left=n)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_sink_minus_inf_is_no_sink():
    n = 70
    q, k, v, kp, vp, table = _one_request(n, 4, 2, 128, 16, 140)
    a = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 2, 16)
    b = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 2, 16,
                            sinks=np.full(4, -np.inf))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_sink_single_key_closed_form():
    q, k, v, kp, vp, table = _one_request(1, 2, 1, 128, 16, 150)
    sinks = np.array([0.3, -1.7])
    O, lse = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [1], 1, 16,
                                 sinks=sinks)
    for h in range(2):
        s = (q.double()[0, h] @ k.double()[0, 0]).item() / math.sqrt(128)
        w = math.exp(s) / (math.exp(s) + math.exp(sinks[h]))
        assert np.allclose(O[0, h], w * v.double()[0, 0].numpy(), atol=1e-14)
        assert lse[0, h] == pytest.approx(s * LOG2E, abs=1e-12)   # sink not in the LSE


def test_sink_scales_output_by_logistic_of_lse():
    """With a sink, O = O_nosink / (1 + exp(sink - ln-LSE)) where ln-LSE is torch's logsumexp."""
    n = 90
    q, k, v, kp, vp, table = _one_request(n, 4, 1, 128, 16, 160)
    sinks = np.array([2.5, -0.5, 0.0, 7.0])
    Os, _ = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, 16,
                                sinks=sinks)
    for h in range(4):
        qq = q.double()[0, h]
        s = (k.double()[:, 0] @ qq) / math.sqrt(128)
        ref = _sdpa_reference(qq[None], k.double()[:, 0], v.double()[:, 0], 1 / math.sqrt(128),
                              torch.ones((1, n), dtype=torch.bool))[0]
        factor = 1.0 / (1.0 + math.exp(sinks[h] - torch.logsumexp(s, 0).item()))
        assert np.allclose(Os[0, h], (factor * ref).numpy(), atol=1e-13)


def test_bmm2_scale_is_linear_and_leaves_lse():
    n = 30
    q, k, v, kp, vp, table = _one_request(n, 2, 1, 128, 16, 170)
    a = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, 16)
    b = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [n], 1, 16,
                            bmm2_scale=-2.5)
    assert np.allclose(b[0], -2.5 * a[0], atol=1e-14)
    assert np.array_equal(a[1], b[1])


def test_packed_q_equals_per_request_fixed_calls():
    lens, qls, ps = [40, 55, 20], [3, 1, 2], 16
    ks = [_rand_bf16((n, 2, 128), 180 + i) for i, n in enumerate(lens)]
    vs = [_rand_bf16((n, 2, 128), 185 + i) for i, n in enumerate(lens)]
    kp, table = _pool_from_dense(ks, ps, 20, 190)
    vp, _ = _pool_from_dense(vs, ps, 20, 190)
    q = _rand_bf16((sum(qls), 4, 128), 191)
    indptr = np.concatenate([[0], np.cumsum(qls)])
    O, lse = oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), lens, 2, ps,
                                 qo_indptr=indptr, causal=True)
    for b in range(3):
        s0, s1 = indptr[b], indptr[b + 1]
        o1, l1 = oracle.paged_decode(_bits(q[s0:s1]), _bits(kp), _bits(vp), table.numpy()[b:b + 1],
                                     [lens[b]], 2, ps, q_len=qls[b], causal=True)
        assert np.array_equal(O[s0:s1], o1) and np.array_equal(lse[s0:s1], l1)


def test_decode_rejects_kv_shorter_than_q():
    q, k, v, kp, vp, table = _one_request(3, 2, 1, 128, 16, 200, L=4)
    with pytest.raises(ValueError):
        oracle.paged_decode(_bits(q), _bits(kp), _bits(vp), table.numpy(), [3], 1, 16, q_len=4)


# ---------------------------------------------------------------------------
# Merge
# ---------------------------------------------------------------------------

def test_merge_of_key_splits_equals_unsplit():
    n = 120
    rng = np.random.default_rng(5)
    qr = rng.standard_normal((3, 64))
    K = rng.standard_normal((n, 64))
    V = rng.standard_normal((n, 64))
    full_o, full_l = oracle.attention_rows(qr, K, V, np.ones((3, n), bool), 0.2)
    cuts = [0, 17, 18, 70, n]
    vs, ss = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.attention_rows(qr, K[a:b], V[a:b], np.ones((3, b - a), bool), 0.2)
        vs.append(o[:, None, :])
        ss.append(l[:, None])
    vo, so = oracle.merge_states(np.stack(vs), np.stack(ss))
    assert np.allclose(vo[:, 0], full_o, atol=1e-13)
    assert np.allclose(so[:, 0], full_l, atol=1e-12)


def test_merge_against_torch_logsumexp_and_empty_states():
    rng = np.random.default_rng(6)
    N, S, H, D = 5, 4, 3, 16
    v = rng.standard_normal((N, S, H, D))
    s = rng.standard_normal((N, S, H)) * 4
    s[:, 0, 0] = -np.inf                 # an all-empty row
    s[1, 1, 1] = -np.inf                 # one empty state among others
    vo, so = oracle.merge_states(v, s)
    assert np.all(vo[0, 0] == 0) and so[0, 0] == -np.inf
    st = torch.tensor(s)
    ref_s = torch.logsumexp(st * math.log(2.0), 0) / math.log(2.0)
    mask = ~torch.isinf(ref_s)
    assert np.allclose(so[mask.numpy()], ref_s[mask].numpy(), atol=1e-12)
    w = torch.softmax(st * math.log(2.0), 0)                      # [N, S, H]
    ref_v = (w[..., None] * torch.tensor(v)).sum(0)
    m = mask.numpy()
    assert np.allclose(vo[m], ref_v.numpy()[m], atol=1e-12)


# ---------------------------------------------------------------------------
# Prefill
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_prefill_matches_torch_sdpa(causal):
    lens = [33, 1, 70]
    Hq, Hkv, D = 4, 2, 128
    indptr = np.concatenate([[0], np.cumsum(lens)])
    T = int(indptr[-1])
    q = _rand_bf16((T, Hq, D), 210)
    k = _rand_bf16((T, Hkv, D), 211)
    v = _rand_bf16((T, Hkv, D), 212)
    O, lse = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), indptr, indptr, Hkv,
                                  causal=causal, output_scale=1.5)
    for b in range(3):
        a, e = indptr[b], indptr[b + 1]
        for h in range(Hq):
            hk = h // 2
            ref = F.scaled_dot_product_attention(
                q.double()[a:e, h][None, None], k.double()[a:e, hk][None, None],
                v.double()[a:e, hk][None, None], is_causal=causal)[0, 0]
            assert np.allclose(O[a:e, h], 1.5 * ref.numpy(), atol=1e-12)
            s = (q.double()[a:e, h] @ k.double()[a:e, hk].T) / math.sqrt(D)
            if causal:
                s = s.masked_fill(~torch.ones_like(s, dtype=torch.bool).tril(), -math.inf)
            assert np.allclose(lse[a:e, h], (torch.logsumexp(s, 1) * LOG2E).numpy(), atol=1e-11)


def test_prefill_row_and_head_subsets_agree_with_full():
    lens = [20, 45]
    indptr = np.concatenate([[0], np.cumsum(lens)])
    q = _rand_bf16((65, 4, 128), 220)
    k = _rand_bf16((65, 1, 128), 221)
    v = _rand_bf16((65, 1, 128), 222)
    O, lse = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), indptr, indptr, 1)
    o, l = oracle.prefill_request(1, _bits(q), _bits(k), _bits(v), indptr, indptr, 1,
                                  heads=[2], rows=[0, 44, 7])
    for r in (0, 44, 7):
        assert np.array_equal(o[r, 2], O[20 + r, 2]) and l[r, 2] == lse[20 + r, 2]


@pytest.mark.parametrize("causal,W", [(True, 0), (True, 5), (True, 40), (False, 7)])
def test_prefill_window_matches_torch_sdpa_band(causal, W):
    """Prefill window_left: torch SDPA with a band mask built by tril/triu."""
    lens_q, lens_k = [33, 1, 70], [40, 1, 70]
    Hq, Hkv, D = 4, 2, 128
    qi = np.concatenate([[0], np.cumsum(lens_q)])
    ki = np.concatenate([[0], np.cumsum(lens_k)])
    q = _rand_bf16((int(qi[-1]), Hq, D), 230)
    k = _rand_bf16((int(ki[-1]), Hkv, D), 231)
    v = _rand_bf16((int(ki[-1]), Hkv, D), 232)
    O, lse = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), qi, ki, Hkv, causal=causal,
                                  window_left=W)
    for b in range(3):
        a, e, ka, kb = qi[b], qi[b + 1], ki[b], ki[b + 1]
        L, n = e - a, kb - ka
        mask = _bottom_right_mask(L, n, causal, W)
        for h in range(Hq):
            hk = h // 2
            ref = F.scaled_dot_product_attention(
                q.double()[a:e, h][None, None], k.double()[ka:kb, hk][None, None],
                v.double()[ka:kb, hk][None, None], attn_mask=mask[None, None])[0, 0]
            assert np.allclose(O[a:e, h], ref.numpy(), atol=1e-12)


def test_prefill_window_zero_returns_diagonal_value_row():
    """window_left = 0 with the causal mask: row i sees only key Lk - Lq + i."""
    lq, lk = [5], [9]
    q = _rand_bf16((5, 2, 128), 240)
    k = _rand_bf16((9, 1, 128), 241)
    v = _rand_bf16((9, 1, 128), 242)
    O, lse = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), np.array([0, 5]),
                                  np.array([0, 9]), 1, causal=True, window_left=0)
    for i in range(5):
        assert np.array_equal(O[i, 0], v.double()[4 + i, 0].numpy())
        s = float((q.double()[i, 1] @ k.double()[4 + i, 0])) / math.sqrt(128)
        assert abs(lse[i, 1] - s * LOG2E) < 1e-12


def test_prefill_window_at_least_kv_len_is_no_window():
    lens = [20, 45]
    ind = np.concatenate([[0], np.cumsum(lens)])
    q = _rand_bf16((65, 2, 128), 250)
    k = _rand_bf16((65, 1, 128), 251)
    v = _rand_bf16((65, 1, 128), 252)
    a = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), ind, ind, 1, window_left=45)
    b = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), ind, ind, 1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _variable_bounds(B, Sq, Sk, seed):
    g = np.random.default_rng(seed)
    a = g.integers(0, Sk, size=(B, Sq))
    b = g.integers(0, Sk, size=(B, Sq))
    return np.minimum(a, b), np.maximum(a, b)


def test_prefill_variable_window_matches_torch_sdpa():
    """variable_window: torch SDPA with a mask from comparisons against the bounds."""
    B, Sq, Sk, Hq, Hkv = 2, 9, 14, 4, 2
    q = _rand_bf16((B * Sq, Hq, 128), 260)
    k = _rand_bf16((B * Sk, Hkv, 128), 261)
    v = _rand_bf16((B * Sk, Hkv, 128), 262)
    st, en = _variable_bounds(B, Sq, Sk, 263)
    qi, ki = np.arange(B + 1) * Sq, np.arange(B + 1) * Sk
    O, lse = oracle.batch_prefill(_bits(q), _bits(k), _bits(v), qi, ki, Hkv,
                                  window_starts=st, window_ends=en)
    j = torch.arange(Sk)
    for b in range(B):
        mask = (j[None, :] >= torch.tensor(st[b])[:, None]) & (j[None, :] <= torch.tensor(en[b])[:, None])
        for h in range(Hq):
            hk = h // 2
            qq = q.double()[b * Sq:(b + 1) * Sq, h]
            kk = k.double()[b * Sk:(b + 1) * Sk, hk]
            ref = F.scaled_dot_product_attention(qq[None, None], kk[None, None],
                                                 v.double()[b * Sk:(b + 1) * Sk, hk][None, None],
                                                 attn_mask=mask[None, None])[0, 0]
            assert np.allclose(O[b * Sq:(b + 1) * Sq, h], ref.numpy(), atol=1e-12)
            s = (qq @ kk.T / math.sqrt(128)).masked_fill(~mask, -math.inf)
            assert np.allclose(lse[b * Sq:(b + 1) * Sq, h], (torch.logsumexp(s, 1) * LOG2E).numpy(),
                               atol=1e-11)


def test_prefill_variable_window_special_cases():
    """Full bounds reduce to the dense mask; bounds [0, Sk - Sq + i] to the causal one;
    a single key start = end returns that value row."""
    B, Sq, Sk = 2, 6, 10
    q = _rand_bf16((B * Sq, 2, 128), 270)
    k = _rand_bf16((B * Sk, 1, 128), 271)
    v = _rand_bf16((B * Sk, 1, 128), 272)
    qi, ki = np.arange(B + 1) * Sq, np.arange(B + 1) * Sk
    args = (_bits(q), _bits(k), _bits(v), qi, ki, 1)
    zeros, full = np.zeros((B, Sq), int), np.full((B, Sq), Sk - 1)
    diag = np.tile(Sk - Sq + np.arange(Sq), (B, 1))
    a = oracle.batch_prefill(*args, window_starts=zeros, window_ends=full)
    d = oracle.batch_prefill(*args, causal=False)
    assert np.array_equal(a[0], d[0]) and np.array_equal(a[1], d[1])
    a = oracle.batch_prefill(*args, window_starts=zeros, window_ends=diag)
    c = oracle.batch_prefill(*args, causal=True)
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])
    one = np.tile(np.arange(Sq) + 2, (B, 1))
    a = oracle.batch_prefill(*args, window_starts=one, window_ends=one)
    for b in range(B):
        for i in range(Sq):
            assert np.array_equal(a[0][b * Sq + i, 0], v.double()[b * Sk + i + 2, 0].numpy())


def test_f16_widening_matches_numpy_on_every_pattern():
    """The binary16 definition written out in the oracle against numpy's float16."""
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_and_bf16_inputs_agree_on_shared_values():
    """Values both formats hold exactly (small integers / 8) give one result either way."""
    g = np.random.default_rng(5)
    B, Hq, Hkv, ps, D = 2, 4, 2, 16, 128
    vals = g.integers(-16, 17, size=(6, Hq, D)) / 8.0
    kv = g.integers(-16, 17, size=(8, Hkv, ps, D)) / 8.0
    vv = g.integers(-16, 17, size=(8, Hkv, ps, D)) / 8.0
    as_f16 = lambda x: np.asarray(x, np.float16).view(np.uint16)
    as_bf16 = lambda x: (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bt = np.array([[3, 1, 5, 7], [0, 2, 4, 6]])
    seq = np.array([50, 33])
    kw = dict(qo_indptr=[0, 3, 6], causal=True, window_left=20)
    a = oracle.paged_decode(as_f16(vals), as_f16(kv), as_f16(vv), bt, seq, Hkv, ps, dtype="f16", **kw)
    b = oracle.paged_decode(as_bf16(vals), as_bf16(kv), as_bf16(vv), bt, seq, Hkv, ps, **kw)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    qp = g.integers(-16, 17, size=(40, Hq, D)) / 8.0
    kp = g.integers(-16, 17, size=(40, Hkv, D)) / 8.0
    ind = np.array([0, 15, 40])
    a = oracle.batch_prefill(as_f16(qp), as_f16(kp), as_f16(kp), ind, ind, Hkv, dtype="f16")
    b = oracle.batch_prefill(as_bf16(qp), as_bf16(kp), as_bf16(kp), ind, ind, Hkv)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
