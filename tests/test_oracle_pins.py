"""Pins for the CPU oracle: each check fixes the oracle to something other than
itself (a hand-worked example, brute force over tiny inputs written another
way, a closed form, a reduction to a library routine, or an equivalence the
pages assert), chosen so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _one_seq_meta(kv_len, q_len=1, ps=4, npages=None):
    npg = -(-kv_len // ps)
    npages = npages or npg
    return dict(
        seq_lens=np.array([kv_len], np.int32),
        cu_q_lens=np.array([0, q_len], np.int32),
        cu_kv_lens=np.array([0, npg * ps], np.int32),
        page_indices=np.arange(npg, dtype=np.int32),
    )


def _cache_from_logical(keys, ps, page_indices, P):
    """Place logical key rows into a paged pool according to the page table."""
    keys = np.asarray(keys, np.float32)
    D = keys.shape[1]
    cache = np.full((P, ps, D), np.nan, np.float32)
    for j in range(keys.shape[0]):
        cache[page_indices[j // ps], j % ps] = keys[j]
    return cache


# ---------------------------------------------------------------- a1 / a2 / a3
def test_hand_worked_indexer_examples():
    with open(os.path.join(GOLDEN, "indexer_hand_example.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        q = np.array(case["q"], np.float32)[None]  # [T=1, H, D]
        w = np.array(case["w"], np.float32)[None]
        keys = np.array(case["keys"], np.float32)
        n = keys.shape[0]
        for ps in (1, 2, 4):
            meta = _one_seq_meta(n, ps=ps)
            cache = _cache_from_logical(keys, ps, meta["page_indices"], len(meta["page_indices"]))
            rows = O.indexer_scores(q, w, cache, **meta)
            np.testing.assert_array_equal(rows[0], np.array(case["scores"], np.float32))
        for tk in case["topk"]:
            s = np.array(case["scores"], np.float32)[: tk["kv_len"]]
            assert O.topk_of_row(s, tk["k"]).tolist() == tk["sel"], (case["name"], tk)
        for pk in case["page_topk"]:
            s = np.array(case["scores"], np.float32)[: pk["kv_len"]]
            assert O.page_topk_of_row(s, pk["ps"], pk["k_pages"]).tolist() == pk["sel"], pk


def _bf16_grid(rng, shape, scale=1.0):
    # values exactly representable in bf16 (few mantissa bits)
    return (np.round(rng.standard_normal(shape) * 8) / 8 * scale).astype(np.float32)


def test_scores_brute_force_multihead_ragged():
    """Python-loop brute force (math.fsum dots, explicit relu and head weights)
    over a ragged batch with a shuffled page table."""
    rng = np.random.default_rng(1)
    H, D, ps = 3, 5, 4
    q_lens, kv_lens = [2, 1, 3], [7, 5, 9]
    S = 3
    npg = [-(-k // ps) for k in kv_lens]
    cu_kv = np.concatenate([[0], np.cumsum(np.array(npg) * ps)]).astype(np.int32)
    P = sum(npg) + 2
    perm = rng.permutation(P).astype(np.int32)
    page_indices = perm[: sum(npg)]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = cu_q[-1]
    logical = [_bf16_grid(rng, (kv_lens[s], D)) for s in range(S)]
    cache = np.zeros((P, ps, D), np.float32)
    for s in range(S):
        for j in range(kv_lens[s]):
            pg = page_indices[cu_kv[s] // ps + j // ps]
            cache[pg, j % ps] = logical[s][j]
    q = _bf16_grid(rng, (T, H, D))
    w = np.abs(_bf16_grid(rng, (T, H))) + 0.125
    w[0, 1] = 0.0
    rows = O.indexer_scores(q, w, cache, np.array(kv_lens, np.int32), cu_q, cu_kv, page_indices)
    t = 0
    for s in range(S):
        for i in range(q_lens[s]):
            pos = kv_lens[s] - q_lens[s] + i
            nvis = min(kv_lens[s], pos + 1)
            assert len(rows[t]) == nvis
            for j in range(nvis):
                tot = 0.0
                for h in range(H):
                    d = math.fsum(float(q[t, h, e]) * float(logical[s][j][e]) for e in range(D))
                    tot += max(d, 0.0) * float(w[t, h])
                assert rows[t][j] == np.float32(tot), (t, j)
            t += 1


def test_score_single_head_reduces_to_dot():
    """With one head, w=1 and positive dots the score is the plain dot product."""
    rng = np.random.default_rng(2)
    D, n = 128, 64
    q = np.abs(_bf16_grid(rng, (1, 1, D))) + 0.125
    keys = np.abs(_bf16_grid(rng, (n, D)))
    meta = _one_seq_meta(n, ps=64)
    rows = O.indexer_scores(q, np.ones((1, 1), np.float32), keys.reshape(1, 64, D), **meta)
    ref = np.array([np.dot(q[0, 0].astype(np.float64), keys[j].astype(np.float64)) for j in range(n)])
    np.testing.assert_array_equal(rows[0], ref.astype(np.float32))
    assert np.all(rows[0] >= 0)


def test_causal_and_kvlen_visibility_closed_form():
    # one request, kv_len 10, 4 new tokens -> positions 6..9 see 7..10 keys
    pos = O.token_pos(np.array([10]), np.array([0, 4]))
    assert pos.tolist() == [6, 7, 8, 9]
    assert O.visible_len(np.array([10]), np.array([0, 4])).tolist() == [7, 8, 9, 10]
    # decode: the single query sits at kv_len - 1, so the causal bound is kv_len
    assert O.visible_len(np.array([5, 9]), np.array([0, 1, 2])).tolist() == [5, 9]
    # an empty request in the middle of the batch
    assert O.token_seq(np.array([0, 2, 2, 5])).tolist() == [0, 0, 2, 2, 2]
    # physical rows follow the packed table
    rows = O.physical_rows(np.array([0, 128, 320]), np.array([7, 3, 9, 1, 4]), 64, 1, np.array([0, 63, 64, 130]))
    assert rows.tolist() == [9 * 64, 9 * 64 + 63, 64 + 0, 4 * 64 + 2]


def test_scores_invariant_under_page_permutation():
    rng = np.random.default_rng(3)
    D, ps, n = 8, 4, 13
    keys = _bf16_grid(rng, (n, D))
    q = _bf16_grid(rng, (1, 2, D))
    w = np.abs(_bf16_grid(rng, (1, 2))) + 0.5
    out = []
    for seed in range(3):
        perm = np.random.default_rng(seed).permutation(6).astype(np.int32)[:4]
        meta = dict(seq_lens=np.array([n], np.int32), cu_q_lens=np.array([0, 1], np.int32),
                    cu_kv_lens=np.array([0, 16], np.int32), page_indices=perm)
        cache = _cache_from_logical(keys, ps, perm, 6)
        out.append(O.indexer_scores(q, w, cache, **meta)[0])
    np.testing.assert_array_equal(out[0], out[1])
    np.testing.assert_array_equal(out[0], out[2])


def _brute_topk(s, k):
    order = sorted(range(len(s)), key=lambda j: (-float(s[j]), j))[:k]
    sel = sorted(order)
    return sel + [-1] * (k - len(sel))


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 60))
    s = (rng.integers(-3, 4, n) / 2).astype(np.float32)  # many exact ties
    for k in (1, 3, n - 1 if n > 1 else 1, n, n + 5):
        got = O.topk_of_row(s, k)
        assert got.tolist() == _brute_topk(s, k)
        sel = got[got >= 0]
        assert len(sel) == min(k, n) and len(set(sel.tolist())) == len(sel)
        rest = np.setdiff1d(np.arange(n), sel)
        if len(rest) and len(sel):
            assert s[sel].min() >= s[rest].max()


def test_page_topk_reduces_to_token_topk_at_page_size_one():
    rng = np.random.default_rng(7)
    s = rng.standard_normal(40).astype(np.float32)
    for k in (1, 5, 40, 45):
        assert O.page_topk_of_row(s, 1, k).tolist() == O.topk_of_row(s, k).tolist()


@pytest.mark.parametrize("seed", range(4))
def test_page_topk_brute_force(seed):
    rng = np.random.default_rng(10 + seed)
    n, ps = int(rng.integers(1, 50)), 4
    s = (rng.integers(-4, 5, n) / 4).astype(np.float32)
    npg = -(-n // ps)
    pmax = [max(float(x) for x in s[p * ps: min(n, (p + 1) * ps)]) for p in range(npg)]
    for kp in (1, 2, npg, npg + 2):
        assert O.page_topk_of_row(s, ps, kp).tolist() == _brute_topk(pmax, kp)


# ----------------------------------------------------------------------- a4
def _brute_union(g, QB, u_max):
    T = len(g)
    nqb = -(-T // QB)
    res = []
    for b in range(nqb):
        blk = g[b * QB:(b + 1) * QB]
        uniq = sorted({x for row in blk for x in row if x >= 0})
        kept = uniq[:u_max]
        units = kept + [-1] * (u_max - len(kept))
        mem = [[1 if (u >= 0 and u in set(row)) else 0 for u in units] for row in blk]
        mem += [[0] * u_max] * (QB - len(blk))
        res.append((units, mem, len(uniq)))
    return res


@pytest.mark.parametrize("seed", range(5))
def test_block_union_brute_force(seed):
    rng = np.random.default_rng(20 + seed)
    T, K, QB = int(rng.integers(1, 23)), 3, 4
    g = rng.integers(-1, 12, (T, K)).astype(np.int64)
    for u_max in (1, 3, 12, QB * K):
        units, member, counts = O.block_union(g, QB, u_max)
        for b, (bu, bm, bc) in enumerate(_brute_union(g.tolist(), QB, u_max)):
            assert units[b].tolist() == bu
            assert member[b].tolist() == bm
            assert counts[b] == bc


def test_lift_units_closed_form():
    tk = np.array([[0, 1, -1], [1, -1, -1], [0, 2, 3]])
    g = O.lift_units(tk, np.array([0, 1, 3]), np.array([0, 128, 448]), 64)
    assert g.tolist() == [[0, 1, -1], [3, -1, -1], [2, 4, 5]]


# ------------------------------------------------------------------- a5 / a6
def _mla_setup(rng, q_lens, kv_lens, H=3, Dk=12, Dv=8, ps=4, spare=2):
    npg = [-(-k // ps) for k in kv_lens]
    cu_kv = np.concatenate([[0], np.cumsum(np.array(npg) * ps)]).astype(np.int32)
    P = sum(npg) + spare
    perm = rng.permutation(P).astype(np.int32)[: sum(npg)]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu_q[-1])
    q = _bf16_grid(rng, (T, H, Dk), 0.5)
    kv = _bf16_grid(rng, (P, ps, Dk))
    meta = dict(seq_lens=np.array(kv_lens, np.int32), cu_q_lens=cu_q, cu_kv_lens=cu_kv, page_indices=perm)
    return q, kv, meta, Dv, ps


def test_attend_single_key_and_uniform_closed_forms():
    rng = np.random.default_rng(30)
    q, kv, meta, Dv, ps = _mla_setup(rng, [1], [9])
    sel = np.array([[5, -1, -1]])
    o, lse = O.sparse_mla(q, kv, **meta, sel=sel, unit=1, sm_scale=0.7, Dv=Dv)
    row = kv[meta["page_indices"][5 // ps], 5 % ps].astype(np.float64)
    np.testing.assert_allclose(o[0], np.broadcast_to(row[:Dv], o[0].shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], 0.7 * q[0].astype(np.float64) @ row[:12], rtol=1e-12)
    # q = 0: every logit is 0 -> plain mean of the values, lse = log(n)
    qz = np.zeros_like(q)
    sel = np.array([[0, 3, 8]])
    o, lse = O.sparse_mla(qz, kv, **meta, sel=sel, unit=1, sm_scale=1.0, Dv=Dv)
    rows = np.stack([kv[meta["page_indices"][j // ps], j % ps] for j in (0, 3, 8)]).astype(np.float64)
    np.testing.assert_allclose(o[0], np.broadcast_to(rows[:, :Dv].mean(0), o[0].shape), atol=1e-12)
    np.testing.assert_allclose(lse[0], math.log(3.0), atol=1e-12)
    # nothing visible: -1 entries and positions past kv_len -> 0 and -inf
    o, lse = O.sparse_mla(q, kv, **meta, sel=np.array([[-1, 9, 12]]), unit=1, sm_scale=1.0, Dv=Dv)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_attend_two_key_closed_form():
    # logits 0 and 1 exactly -> weights 1/(1+e), e/(1+e)
    ps, D = 2, 4
    kv = np.zeros((1, ps, D), np.float32)
    kv[0, 0] = [0.0, 0.0, 1.0, -2.0]
    kv[0, 1] = [1.0, 0.0, 3.0, 5.0]
    q = np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32)
    meta = dict(seq_lens=np.array([2], np.int32), cu_q_lens=np.array([0, 1], np.int32),
                cu_kv_lens=np.array([0, 2], np.int32), page_indices=np.array([0], np.int32))
    o, lse = O.sparse_mla(q, kv, **meta, sel=np.array([[0, 1]]), unit=1, sm_scale=1.0, Dv=2)
    e = math.e
    np.testing.assert_allclose(o[0, 0], [e / (1 + e), 0.0], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(1 + e), atol=1e-14)


def test_attend_causal_mask_and_order_invariance():
    rng = np.random.default_rng(31)
    q, kv, meta, Dv, ps = _mla_setup(rng, [3], [10])
    # token 0 sits at position 7: positions 8, 9 are masked even when selected
    sel = np.array([[9, 2, 8, 7, 0]] * 3)
    o1, _ = O.sparse_mla(q, kv, **meta, sel=sel, unit=1, sm_scale=0.5, Dv=Dv)
    o2, _ = O.sparse_mla(q, kv, **meta, sel=np.array([[0, 2, 7, -1, -1]] * 3), unit=1, sm_scale=0.5, Dv=Dv)
    np.testing.assert_allclose(o1[0], o2[0], atol=1e-13)
    perm = sel[:, ::-1].copy()
    o3, _ = O.sparse_mla(q, kv, **meta, sel=perm, unit=1, sm_scale=0.5, Dv=Dv)
    np.testing.assert_allclose(o1, o3, atol=1e-13)


@pytest.mark.parametrize("seed", range(3))
def test_sparse_with_everything_selected_equals_dense(seed):
    """The spec property: top-k with k >= kv_len is dense causal MLA."""
    rng = np.random.default_rng(40 + seed)
    q_lens, kv_lens = [1, 4, 2], [6, 11, 3]
    q, kv, meta, Dv, ps = _mla_setup(rng, q_lens, kv_lens)
    kmax = max(kv_lens)
    sel = np.tile(np.arange(kmax), (sum(q_lens), 1))
    o_s, _ = O.sparse_mla(q, kv, **meta, sel=sel, unit=1, sm_scale=0.3, Dv=Dv)
    o_d = O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv)
    np.testing.assert_allclose(o_s, o_d, rtol=1e-12, atol=1e-13)
    # the same through page units
    pages = np.tile(np.arange(-(-kmax // ps)), (sum(q_lens), 1))
    o_p, _ = O.sparse_mla(q, kv, **meta, sel=pages, unit=ps, sm_scale=0.3, Dv=Dv)
    np.testing.assert_allclose(o_p, o_d, rtol=1e-12, atol=1e-13)


def test_page_units_equal_expanded_token_units():
    rng = np.random.default_rng(50)
    q, kv, meta, Dv, ps = _mla_setup(rng, [2, 1], [9, 14])
    pages = np.array([[0, 2, -1], [3, 1, 0], [1, -1, -1]])
    toks = np.full((3, 12), -1)
    for t in range(3):
        lst = [p * ps + r for p in pages[t] if p >= 0 for r in range(ps)]
        toks[t, : len(lst)] = lst
    o_p, l_p = O.sparse_mla(q, kv, **meta, sel=pages, unit=ps, sm_scale=0.4, Dv=Dv)
    o_t, l_t = O.sparse_mla(q, kv, **meta, sel=toks, unit=1, sm_scale=0.4, Dv=Dv)
    np.testing.assert_allclose(o_p, o_t, atol=1e-13)
    np.testing.assert_allclose(l_p, l_t, atol=1e-13)


@pytest.mark.parametrize("seed", range(3))
def test_qblock_equals_per_query_sparse_mla(seed):
    """The pages' parity claim: the blocked kernel computes the same
    masked-softmax math as the per-query kernel (blocks straddle requests)."""
    rng = np.random.default_rng(60 + seed)
    q_lens, kv_lens = [1, 5, 1, 6], [7, 13, 4, 10]
    q, kv, meta, Dv, ps = _mla_setup(rng, q_lens, kv_lens)
    T, K, QB = sum(q_lens), 3, 4
    seq = O.token_seq(meta["cu_q_lens"])
    nvis = O.visible_len(meta["seq_lens"], meta["cu_q_lens"])
    sel = np.full((T, K), -1, np.int64)
    for t in range(T):
        npg = -(-int(nvis[t]) // ps)
        ch = rng.permutation(npg)[: rng.integers(0, K + 1)]
        sel[t, : len(ch)] = np.sort(ch)
    g = O.lift_units(sel, meta["cu_q_lens"], meta["cu_kv_lens"], ps)
    u_max = min(QB * K, len(meta["page_indices"]))
    units, member, counts = O.block_union(g, QB, u_max)
    o_b, l_b = O.qblock_attend(q, kv, **meta, units=units, member=member, counts=counts, QB=QB,
                               sm_scale=0.6, Dv=Dv)
    o_q, l_q = O.sparse_mla(q, kv, **meta, sel=sel, unit=ps, sm_scale=0.6, Dv=Dv)
    np.testing.assert_allclose(o_b, o_q, atol=1e-13)
    np.testing.assert_allclose(l_b, l_q, atol=1e-13)
    assert seq[-1] == 3


def test_qblock_truncated_union_drops_the_tail():
    rng = np.random.default_rng(70)
    q, kv, meta, Dv, ps = _mla_setup(rng, [4], [16])
    sel = np.array([[0, 3, -1], [1, 2, -1], [0, 1, 2], [3, -1, -1]])
    g = O.lift_units(sel, meta["cu_q_lens"], meta["cu_kv_lens"], ps)
    units, member, counts = O.block_union(g, 4, 2)  # keeps pages 0, 1 only
    assert counts.tolist() == [4] and units.tolist() == [[0, 1]]
    o_b, _ = O.qblock_attend(q, kv, **meta, units=units, member=member, counts=counts, QB=4,
                             sm_scale=0.5, Dv=Dv)
    kept = np.where(np.isin(sel, [0, 1]), sel, -1)
    o_q, _ = O.sparse_mla(q, kv, **meta, sel=kept, unit=ps, sm_scale=0.5, Dv=Dv)
    np.testing.assert_allclose(o_b, o_q, atol=1e-13)


# ----------------------------------------------------------------------- a7
def test_share_map_closed_form_and_errors():
    full, src, n = O.build_index_share_map(["full", "shared", "shared", "full"], 0, 4)
    assert full == {0: 0, 3: 1} and src == {0: 0, 1: 0, 2: 0, 3: 1} and n == 2
    full, src, n = O.build_index_share_map(None, 5, 3)
    assert full == {0: 0, 1: 1, 2: 2} and src == full and n == 3
    with pytest.raises(O.ShareMapError):
        O.build_index_share_map(["shared", "full"], 0, 2)
    with pytest.raises(O.ShareMapError):
        O.build_index_share_map(["full", "dense"], 0, 2)
    with pytest.raises(O.ShareMapError):
        O.build_index_share_map(["full"], 0, 2)


def test_widen_bf16_bits_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F80], np.uint16)
    vals = O.widen(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0 and np.isinf(vals[5])
    assert vals[2] == 3.140625


# ------------------------------------------------ paged write-back (before a1)
def test_write_back_hand_example():
    # one request, page size 4, pages [2, 0, 1]: kv_len 6 with 2 new tokens at
    # positions 4 and 5 -> logical page 1 -> physical page 0, rows 0 and 1
    cache = np.zeros((3, 4, 2), np.float32)
    rows = np.array([[1.0, 2.0], [3.0, 4.0]])
    out = O.paged_write_back(cache, rows, seq_lens=[6], cu_q_lens=[0, 2], cu_kv_lens=[0, 12],
                             page_indices=[2, 0, 1])
    expect = np.zeros_like(cache)
    expect[0, 0] = [1.0, 2.0]
    expect[0, 1] = [3.0, 4.0]
    np.testing.assert_array_equal(out, expect)
    assert cache.sum() == 0  # the input is not modified


@pytest.mark.parametrize("seed", [0, 1])
def test_write_back_round_trip_and_untouched_rows(seed):
    # ragged batch (decode, extend, empty request, prefill): reading the written
    # cache back through the independent position -> row map returns each
    # token's row, at exactly its position, and leaves every other row as is
    rng = np.random.default_rng(seed)
    ps = 8
    q_lens = np.array([1, 5, 0, 12])
    kv_lens = np.array([19, 30, 3, 12])
    npages = -(-kv_lens // ps)
    cu_kv = np.concatenate([[0], np.cumsum(npages * ps)])
    P = int(npages.sum()) + 2
    page_indices = rng.permutation(P)[: int(npages.sum())]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)])
    T, W, D = int(cu_q[-1]), 10, 7
    cache = rng.standard_normal((P, ps, W))
    rows = rng.standard_normal((T, D))
    out = O.paged_write_back(cache, rows, kv_lens, cu_q, cu_kv, page_indices)
    written = np.zeros((P * ps,), bool)
    t = 0
    for s in range(len(q_lens)):
        for j in range(q_lens[s]):
            pos = kv_lens[s] - q_lens[s] + j
            r = int(O.physical_rows(cu_kv, page_indices, ps, s, [pos])[0])
            np.testing.assert_array_equal(out.reshape(-1, W)[r, :D], rows[t])
            np.testing.assert_array_equal(out.reshape(-1, W)[r, D:], cache.reshape(-1, W)[r, D:])
            assert not written[r]
            written[r] = True
            t += 1
    np.testing.assert_array_equal(out.reshape(-1, W)[~written], cache.reshape(-1, W)[~written])


# ---------------------------------------- token top-k -> page list (NEXT-2)
def test_topk_pages_of_tokens_closed_forms():
    pages, n = O.topk_pages_of_tokens([130, 5, -1, 64, 127, 0, 63], 64, 4)
    assert pages.tolist() == [0, 1, 2, -1] and n == 3
    pages, n = O.topk_pages_of_tokens([-1, -1], 64, 2)
    assert pages.tolist() == [-1, -1] and n == 0
    # truncation keeps the lowest pages; page size 1 turns it into a sort
    pages, n = O.topk_pages_of_tokens([9, 3, 7, 3, 1], 1, 3)
    assert pages.tolist() == [1, 3, 7] and n == 4


def test_topk_pages_cover_exactly_the_selected_tokens():
    rng = np.random.default_rng(5)
    row = rng.choice(5000, size=700, replace=False)
    pages, n = O.topk_pages_of_tokens(row, 64, 200)
    got = set(pages[pages >= 0].tolist())
    assert got == {int(j) // 64 for j in row} and n == len(got)
    assert all(a < b for a, b in zip(pages[:n], pages[1:n]))


# ------------------------------------- dense MLA fallback: window and cap (NEXT-4)
def test_dense_window_and_soft_cap_limits():
    rng = np.random.default_rng(77)
    q_lens, kv_lens = [1, 4, 2], [6, 11, 3]
    q, kv, meta, Dv, ps = _mla_setup(rng, q_lens, kv_lens)
    base = O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv)
    # a window at least as long as every context changes nothing
    np.testing.assert_allclose(O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv, sliding_window=64), base,
                               rtol=1e-12, atol=1e-13)
    # a huge cap is the identity on the logits
    np.testing.assert_allclose(O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv, soft_cap=1e9), base,
                               rtol=1e-9, atol=1e-9)
    seq = O.token_seq(meta["cu_q_lens"])
    pos = O.token_pos(meta["seq_lens"], meta["cu_q_lens"])
    kvf = O.widen(kv)
    w1 = O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv, sliding_window=1)
    tiny = O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv, soft_cap=1e-12)
    w3 = O.dense_mla(q, kv, **meta, sm_scale=0.3, Dv=Dv, sliding_window=3, soft_cap=1e-12)
    for t in range(sum(q_lens)):
        s, p = int(seq[t]), int(pos[t])
        rows = O.physical_rows(meta["cu_kv_lens"], meta["page_indices"], ps, s, np.arange(p + 1))
        vals = kvf.reshape(-1, kvf.shape[-1])[rows, :Dv]
        # window 1: only the query's own position -> its value, for every head
        np.testing.assert_allclose(w1[t], np.tile(vals[-1], (w1.shape[1], 1)), rtol=1e-12, atol=1e-13)
        # a vanishing cap flattens every logit -> the plain mean of the visible values
        np.testing.assert_allclose(tiny[t], np.tile(vals.mean(axis=0), (tiny.shape[1], 1)), rtol=1e-9, atol=1e-9)
        # both: the mean of the last three positions
        np.testing.assert_allclose(w3[t], np.tile(vals[-3:].mean(axis=0), (w3.shape[1], 1)), rtol=1e-9,
                                   atol=1e-9)


# --------------------------------------------- approximate top-k (NEXT-3)
def test_approx_topk_hand_example_and_exact_limit():
    s = np.array([5, 1, 9, 3, 2, 8, 7, 0], np.float32)
    # k=2, over=2 -> 4 bins {0,4} {1,5} {2,6} {3,7}: maxima 5@0, 8@5, 9@2, 3@3
    # -> best two bins hold 9@2 and 8@5
    assert O.approx_topk_of_row(s, 2, 2).tolist() == [2, 5]
    # k=3, over=1 -> 3 bins {0,3,6} {1,4,7} {2,5}: maxima 7@6, 2@4, 9@2 -> all three bins
    assert O.approx_topk_of_row(s, 3, 1).tolist() == [2, 4, 6]
    rng = np.random.default_rng(9)
    for n in (1, 17, 300):
        x = rng.standard_normal(n).astype(np.float32)
        for k in (1, 5, 64):
            # enough bins for every position: the exact top-k
            assert O.approx_topk_of_row(x, k, max(1, -(-n // k))).tolist() == O.topk_of_row(x, k).tolist()


def test_approx_topk_selects_bin_maxima_and_count():
    rng = np.random.default_rng(12)
    x = rng.standard_normal(5000).astype(np.float32)
    k, over = 64, 4
    sel = O.approx_topk_of_row(x, k, over)
    assert (sel >= 0).sum() == k and np.all(np.diff(sel) > 0)
    B = over * k
    exact = set(O.topk_of_row(x, k).tolist())
    for j in sel:
        bin_idx = np.arange(j % B, 5000, B)
        assert x[j] == x[bin_idx].max()
    # every exact winner that is the maximum of its bin is found
    for j in exact:
        bin_idx = np.arange(j % B, 5000, B)
        if x[j] == x[bin_idx].max():
            assert j in set(sel.tolist())


# ------------------------------------------- composed entries, small helpers
def test_hand_worked_selections_through_the_indexer_entries():
    """The composed oracle entries (score the paged cache, then select) give
    the hand-worked selections, with kv_len cutting the row; the cache holds
    NaN past kv_len, so a read of a masked position would show."""
    with open(os.path.join(GOLDEN, "indexer_hand_example.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        q = np.array(case["q"], np.float32)[None]
        w = np.array(case["w"], np.float32)[None]
        keys = np.array(case["keys"], np.float32)
        for tk in case["topk"]:
            kv = tk["kv_len"]
            meta = _one_seq_meta(kv, ps=2)
            cache = _cache_from_logical(keys[:kv], 2, meta["page_indices"], len(meta["page_indices"]))
            sel, rows = O.indexer_topk(q, w, cache, k=tk["k"], **meta)
            assert sel[0].tolist() == tk["sel"], (case["name"], tk)
            np.testing.assert_array_equal(rows[0], np.array(case["scores"][:kv], np.float32))
        for pk in case["page_topk"]:
            kv, ps = pk["kv_len"], pk["ps"]
            meta = _one_seq_meta(kv, ps=ps)
            cache = _cache_from_logical(keys[:kv], ps, meta["page_indices"], len(meta["page_indices"]))
            sel, _ = O.indexer_page_topk(q, w, cache, k_pages=pk["k_pages"], **meta)
            assert sel[0].tolist() == pk["sel"], (case["name"], pk)


def test_score_row_worked_by_hand():
    # two heads, three keys: dots h0 = (1, -1, 3), h1 = (2, 4, -5); relu, then
    # weights (2, 3): 2*(1, 0, 3) + 3*(2, 4, 0) = (8, 12, 6)
    q = np.array([[1.0, 0.0], [0.0, 1.0]], np.float32)
    w = np.array([2.0, 3.0], np.float32)
    keys = np.array([[1.0, 2.0], [-1.0, 4.0], [3.0, -5.0]], np.float32)
    np.testing.assert_array_equal(O.indexer_score_row(q, w, keys), np.array([8.0, 12.0, 6.0], np.float32))


def test_page_scores_of_row_worked_by_hand():
    row = np.array([1.0, 5.0, 2.0, -3.0, 0.5], np.float32)
    # pages of two: max(1, 5), max(2, -3), and the partial last page 0.5
    np.testing.assert_array_equal(O.page_scores_of_row(row, 2), np.array([5.0, 2.0, 0.5], np.float32))
    np.testing.assert_array_equal(O.page_scores_of_row(row, 1), row)  # page size 1: the row itself
    np.testing.assert_array_equal(O.page_scores_of_row(row, 8), np.array([5.0], np.float32))


def test_selected_positions_worked_by_hand():
    assert O.selected_positions([5, -1, 2, 5], 1, 4).tolist() == [5, 2, 5]  # tokens: -1 dropped, as given
    assert O.selected_positions([2, -1, 0], 4, 4).tolist() == [8, 9, 10, 11, 0, 1, 2, 3]  # pages of 4
    assert O.selected_positions([-1, -1], 4, 4).tolist() == []
