"""GPU parity of every hot-path step against the CPU oracle, through the C ABI,
on seeded ragged batches that span several tiles and a ragged tail."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import (check_attention, check_scores, check_topk_rows, f32, member_bits_to_int8, meta_np,
                      meta_to)

pytestmark = pytest.mark.gpu

CASES = {
    "decode": ([1, 1, 1, 1, 1], [300, 1000, 64, 2500, 7]),
    "prefill": ([200], [200]),
    "extend": ([37], [500]),
    "mixed": ([1, 50, 0, 1, 9, 3], [700, 300, 40, 65, 1000, 4]),
    "tails": ([8, 17, 2], [8, 130, 129]),
    # as many tokens as requests although two requests have several: the
    # indexer plans every token as a one-token tile
    "one_token": ([2, 0, 1, 3, 0, 0], [300, 40, 900, 129, 10, 64]),
}


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _wl(case, seed, ps=64, k=64, k_pages=3, H=16):
    q_lens, kv_lens = CASES[case]
    return DI.random_small(seed, q_lens, kv_lens, H=H, page_size=ps, k=k, k_pages=k_pages)


def _oracle_scores(wl):
    rg = wl.rg
    return O.indexer_scores(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg))


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("ps", [64, 32, 128])
def test_indexer_token_topk(dsa, case, ps):
    dev = torch.device("cuda")
    wl = _wl(case, 100 + len(case) + ps, ps=ps, k=64)
    rg = wl.rg
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    topk, vals = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta, k=wl.k,
                                      max_kv=rg.max_kv, want_scores=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = _oracle_scores(wl)
    ref = np.stack([O.topk_of_row(r, wl.k) for r in rows])
    check_topk_rows(topk.cpu().numpy(), ref, wl.k, rows)
    check_scores(vals.cpu().numpy(), topk.cpu().numpy(), rows)


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("ps", [64, 32, 128])
def test_indexer_page_topk(dsa, case, ps):
    dev = torch.device("cuda")
    wl = _wl(case, 200 + len(case) + ps, ps=ps, k=48, k_pages=3)
    rg = wl.rg
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pages, topk = dsa.dsa_indexer_page_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta,
                                            k_pages=wl.k_pages, max_kv=rg.max_kv, k=wl.k, with_tokens=True,
                                            dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = _oracle_scores(wl)
    prow = [O.page_scores_of_row(r, ps) for r in rows]
    ref_p = np.stack([O.topk_of_row(p, wl.k_pages) for p in prow])
    check_topk_rows(pages.cpu().numpy(), ref_p, wl.k_pages, prow, "page top-k")
    ref_t = np.stack([O.topk_of_row(r, wl.k) for r in rows])
    check_topk_rows(topk.cpu().numpy(), ref_t, wl.k, rows, "token top-k")


def _rand_sel(rng, rg, K, unit, dense=False):
    nvis = O.visible_len(rg.seq_lens, rg.cu_q_lens)
    sel = np.full((rg.T, K), -1, np.int32)
    for t in range(rg.T):
        n = int(nvis[t]) if unit == 1 else -(-int(nvis[t]) // unit)
        if n == 0:
            continue
        m = min(K, n) if dense else int(rng.integers(0, min(K, n) + 1))
        ch = np.sort(rng.choice(n, size=m, replace=False))
        sel[t, :m] = ch
    return sel


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("unit_kind", ["token", "page"])
@pytest.mark.parametrize("H", [16, 128])
def test_sparse_mla_decode(dsa, case, unit_kind, H):
    dev = torch.device("cuda")
    ps = 64
    wl = _wl(case, 300 + len(case) + H, ps=ps, H=H)
    rg = wl.rg
    rng = np.random.default_rng(7)
    unit = 1 if unit_kind == "token" else ps
    K = 96 if unit == 1 else 4
    sel = _rand_sel(rng, rg, K, unit, dense=True)
    sel[0, ::3] = -1  # holes inside a row
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = dsa.dsa_sparse_mla_decode(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, torch.from_numpy(sel).to(dev),
                                       unit=unit, sm_scale=wl.sm_scale, want_lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_o, ref_l = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=unit,
                                sm_scale=wl.sm_scale, Dv=512)
    check_attention(o, ref_o)
    l = lse.cpu().numpy()
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    np.testing.assert_allclose(l[fin], ref_l[fin], rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("unit_kind", ["token", "page"])
@pytest.mark.parametrize("H", [128, 40])
def test_sparse_mla_decode_most_splits(dsa, unit_kind, H):
    """One decode token with a long selection: the key list is split over the
    most CTAs the kernel allows (8), and with H = 40 some head rows of the
    merge are missing."""
    dev = torch.device("cuda")
    ps = 64
    wl = DI.random_small(411 + H, [1], [4000], H=H, page_size=ps, k=64, k_pages=3)
    rg = wl.rg
    rng = np.random.default_rng(11)
    unit = 1 if unit_kind == "token" else ps
    K = 512 if unit == 1 else 16
    sel = _rand_sel(rng, rg, K, unit, dense=True)
    sel[0, 5:K:7] = -1  # holes inside the row
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = dsa.dsa_sparse_mla_decode(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, torch.from_numpy(sel).to(dev),
                                       unit=unit, sm_scale=wl.sm_scale, want_lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_o, ref_l = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=unit,
                                sm_scale=wl.sm_scale, Dv=512)
    check_attention(o, ref_o)
    l = lse.cpu().numpy()
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    np.testing.assert_allclose(l[fin], ref_l[fin], rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("unit,K", [(1, 1024), (64, 40)])
def test_sparse_mla_decode_splits_reproducible(dsa, unit, K):
    """Decode rows split over several CTAs (token and page units) merge their
    splits in a fixed order: repeated calls give the same output bits,
    whichever CTA of a row finishes last."""
    dev = torch.device("cuda")
    wl = DI.random_small(419, [1, 1, 1], [4000, 3000, 2500], H=128, k=64)
    rg = wl.rg
    sel = _rand_sel(np.random.default_rng(12), rg, K, unit, dense=True)
    meta = meta_to(rg, dev)
    q, kv, s = wl.q[0].to(dev), wl.kv[0].to(dev), torch.from_numpy(sel).to(dev)
    assert dsa.dsa_sparse_mla_decode_workspace_size(rg.T, 128) > 0, "the rows must be split"
    outs = []
    for _ in range(6):
        o = dsa.dsa_sparse_mla_decode(q, kv, *meta, s, unit=unit, sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        outs.append(o.view(torch.int16).cpu().numpy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "split decode output changed between identical calls"
    ref_o, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=unit, sm_scale=wl.sm_scale,
                            Dv=512)
    check_attention(torch.from_numpy(outs[0]).view(torch.bfloat16), ref_o)


@pytest.mark.parametrize("case", ["prefill", "mixed", "tails", "extend"])
@pytest.mark.parametrize("QB", [32, 64])
def test_block_union_and_qblock(dsa, case, QB):
    dev = torch.device("cuda")
    ps = 64
    wl = _wl(case, 400 + len(case) + QB, ps=ps, H=128)
    rg = wl.rg
    rng = np.random.default_rng(11)
    K = 3
    sel = _rand_sel(rng, rg, K, ps)
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sel_d = torch.from_numpy(sel).to(dev)
    u_max = min(QB * K, rg.PTW)
    units, member, counts = dsa.dsa_build_block_union(sel_d, QB=QB, u_max=u_max, cu_q_lens=meta[1],
                                                      cu_kv_lens=meta[2], ps=ps, PTW=rg.PTW, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    g = O.lift_units(sel, rg.cu_q_lens, rg.cu_kv_lens, ps)
    ru, rm, rc = O.block_union(g, QB, u_max)
    assert np.array_equal(units.cpu().numpy(), ru)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(member_bits_to_int8(member.cpu().numpy().view(np.uint32), QB), rm)
    o = dsa.dsa_sparse_mla_prefill_qblock(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, units, member, counts, QB=QB,
                                          sm_scale=wl.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_o, _ = O.qblock_attend(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), units=ru, member=rm, counts=rc, QB=QB,
                               sm_scale=wl.sm_scale, Dv=512)
    check_attention(o, ref_o, "qblock")


def test_block_union_truncation_flag(dsa):
    dev = torch.device("cuda")
    T, K, QB, PTW = 64, 4, 32, 100
    rng = np.random.default_rng(5)
    sel = rng.integers(-1, PTW, (T, K)).astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    units, member, counts = dsa.dsa_build_block_union(torch.from_numpy(sel).to(dev), QB=QB, u_max=16, PTW=PTW,
                                                      dev_status=st)
    torch.cuda.synchronize()
    ru, rm, rc = O.block_union(sel.astype(np.int64), QB, 16)
    assert np.array_equal(units.cpu().numpy(), ru)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(member_bits_to_int8(member.cpu().numpy().view(np.uint32), QB), rm)
    assert st.item() & 0x1


def test_tiny_decode_end_to_end(dsa):
    """The tiny-decode workload through indexer -> top-k -> sparse MLA."""
    dev = torch.device("cuda")
    wl = DI.tiny_decode()
    rg = wl.rg
    meta = meta_to(rg, dev)
    topk = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta, k=wl.k,
                                max_kv=rg.max_kv)
    rows = _oracle_scores(wl)
    ref = np.stack([O.topk_of_row(r, wl.k) for r in rows])
    check_topk_rows(topk.cpu().numpy(), ref, wl.k, rows)
    o = dsa.dsa_sparse_mla_decode(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, torch.from_numpy(ref).to(dev), unit=1,
                                  sm_scale=wl.sm_scale)
    ref_o, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=ref, unit=1, sm_scale=wl.sm_scale,
                            Dv=512)
    check_attention(o, ref_o)


@pytest.mark.parametrize("ps", [32, 64])
def test_page_units_odd_step_count_reads_no_stray_rows(dsa, ps):
    """A selection with an odd number of 32-key steps is completed by an empty
    step; its boxes must be zero-filled, not read from the start of the cache
    (here physical page 0 holds NaN and is selected by nobody)."""
    dev = torch.device("cuda")
    wl = DI.random_small(431 + ps, [1, 1], [700, 900], H=16, page_size=ps)
    rg = wl.rg
    kv = wl.kv[0].clone()
    kv.view(torch.int16)[0] = 0x7FC0  # bf16 NaN in every row of physical page 0
    owner = np.nonzero(rg.page_indices == 0)[0]
    pages = [np.arange(-(-int(n) // ps)) for n in rg.seq_lens]
    sel = np.full((rg.T, 3), -1, np.int32)
    for t in range(rg.T):
        base = rg.cu_kv_lens[t] // ps
        ok = [p for p in pages[t] if base + p not in owner]  # pages that are not physical page 0
        sel[t] = ok[:3]
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o = dsa.dsa_sparse_mla_decode(wl.q[0].to(dev), kv.to(dev), *meta, torch.from_numpy(sel).to(dev), unit=ps,
                                  sm_scale=wl.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.isfinite(o.float()).all(), "a stray row of page 0 reached the output"
    ref_o, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=ps, sm_scale=wl.sm_scale,
                            Dv=512)
    check_attention(o, ref_o, "odd page steps")
