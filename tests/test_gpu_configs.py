"""Full-size workloads through the same layer runner the bench times, checked
against the CPU oracle on sampled rows (request edges, block boundaries,
decode rows): indexer scores and token top-k (near-tie rule), page top-k,
block union tables (bit-exact), and the attention fed the oracle's
selections (decode) or tables (query-block prefill), including IndexShare."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from config_util import CompactPool, rows_of, sel_entries, seq_entries
from gpu_util import check_attention, check_scores, check_topk_rows, member_bits_to_int8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _meta(rg):
    return dict(seq_lens=rg.seq_lens, cu_q_lens=rg.cu_q_lens, cu_kv_lens=rg.cu_kv_lens)


def _oracle_scores(wl, slot, tokens):
    rg = wl.rg
    tseq = O.token_seq(rg.cu_q_lens)
    pool = CompactPool([wl.kcache[slot]], rg.page_indices, seq_entries(rg, sorted({int(tseq[t]) for t in tokens})))
    rows = O.indexer_scores(rows_of(wl.q_idx, tokens), rows_of(wl.w, tokens), pool.caches[0],
                            page_indices=pool.page_indices, tokens=tokens, **_meta(rg))
    return dict(zip(tokens, rows))


def _check_indexer_rows(rn, slot, scores, tokens, token_topk=True, page_topk=True):
    rg = rn.rg
    ps = rg.page_size
    if token_topk:
        got = rn.topk[slot][tokens].cpu().numpy()
        ref = np.stack([O.topk_of_row(scores[t], rn.k) for t in tokens])
        check_topk_rows(got, ref, rn.k, [scores[t] for t in tokens], "token top-k")
    if page_topk:
        got = rn.topk_pages[slot][tokens].cpu().numpy()
        prow = [O.page_scores_of_row(scores[t], ps) for t in tokens]
        ref = np.stack([O.topk_of_row(p, rn.k_pages) for p in prow])
        check_topk_rows(got, ref, rn.k_pages, prow, "page top-k")


def _check_decode_attend(dsa, wl, rn, layer, slot, tokens, scores, unit):
    """Attention on the oracle's selections for the sampled rows."""
    rg = wl.rg
    ps = rg.page_size
    if unit == 1:
        ref_sel = {t: O.topk_of_row(scores[t], rn.k) for t in tokens}
        sel = rn.topk[slot].clone()
    else:
        ref_sel = {t: O.topk_of_row(O.page_scores_of_row(scores[t], ps), rn.k_pages) for t in tokens}
        sel = rn.topk_pages[slot].clone()
    for t in tokens:
        sel[t] = torch.from_numpy(ref_sel[t]).to(sel.device)
    o = dsa.dsa_sparse_mla_decode(rn.q[layer], rn.kv[layer], *rn.meta, sel, unit=unit, sm_scale=wl.sm_scale,
                                  ws=rn.ws_att, dev_status=rn.status)
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    tseq = O.token_seq(rg.cu_q_lens)
    pool = CompactPool([wl.kv[layer]], rg.page_indices, sel_entries(rg, tseq, tokens, ref_sel, unit))
    ref_o, _ = O.sparse_mla(rows_of(wl.q[layer], tokens), pool.caches[0], page_indices=pool.page_indices, sel=ref_sel,
                            unit=unit, sm_scale=wl.sm_scale, Dv=512, tokens=tokens, **_meta(rg))
    check_attention(o[tokens], ref_o, f"decode attention (layer {layer})")


def _oracle_tables(rn, slot, blocks):
    """Oracle union tables of the sampled blocks, from the GPU page top-k
    (whose sampled rows are checked against the oracle separately)."""
    rg = rn.rg
    QB, u_max = rn.QB, rn.u_max
    tp = rn.topk_pages[slot].cpu().numpy()
    g = O.lift_units(tp, rg.cu_q_lens, rg.cu_kv_lens, rg.page_size)
    nqb = rn.units[slot].shape[0]
    units = np.full((nqb, u_max), -1, np.int32)
    member = np.zeros((nqb, QB, u_max), np.int8)
    counts = np.zeros(nqb, np.int32)
    for b in blocks:
        u, m, c = O.block_union(g[b * QB:(b + 1) * QB], QB, u_max)
        units[b], member[b], counts[b] = u[0], m[0], c[0]
    return units, member, counts


def _check_union_and_qblock(dsa, wl, rn, layer, slot, tokens):
    rg = wl.rg
    QB = rn.QB
    blocks = sorted({t // QB for t in tokens})
    units, member, counts = _oracle_tables(rn, slot, blocks)
    gu = rn.units[slot].cpu().numpy()
    gm = member_bits_to_int8(rn.member[slot].cpu().numpy().view(np.uint32), QB)
    gc = rn.counts[slot].cpu().numpy()
    for b in blocks:
        assert np.array_equal(gu[b], units[b]), f"union units, block {b}"
        assert np.array_equal(gc[b], counts[b]), f"union count, block {b}"
        assert np.array_equal(gm[b], member[b]), f"membership, block {b}"
    # the GPU tables equal the oracle's on these blocks: the qblock kernel is fed them
    o = dsa.dsa_sparse_mla_prefill_qblock(rn.q[layer], rn.kv[layer], *rn.meta, rn.units[slot], rn.member[slot],
                                          rn.counts[slot], QB=QB, sm_scale=wl.sm_scale, dev_status=rn.status)
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    entries = []
    for t in tokens:
        b, q = divmod(t, QB)
        n = min(int(counts[b]), rn.u_max)
        entries.extend(units[b, :n][member[b, q, :n] > 0].tolist())
    pool = CompactPool([wl.kv[layer]], rg.page_indices, entries or [0])
    ref_o, _ = O.qblock_attend(rows_of(wl.q[layer], tokens), pool.caches[0], page_indices=pool.page_indices,
                               units=units, member=member, counts=counts, QB=QB, sm_scale=wl.sm_scale, Dv=512,
                               tokens=tokens, **_meta(rg))
    check_attention(o[tokens], ref_o, f"qblock attention (layer {layer})")


@pytest.mark.parametrize("name,tokens", [("batched_decode", [0, 17, 31]), ("long_decode", [0, 63])])
def test_decode_workload_token_topk(dsa, name, tokens):
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.WORKLOADS[name](device="cuda")
    rn = LayerRunner(wl, "cuda")
    rn.index(0)
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    scores = _oracle_scores(wl, 0, tokens)
    _check_indexer_rows(rn, 0, scores, tokens, token_topk=True, page_topk=False)
    _check_decode_attend(dsa, wl, rn, 0, 0, tokens, scores, unit=1)


def test_long_decode_page_budget(dsa):
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.long_decode(device="cuda")
    rn = LayerRunner(wl, "cuda", page_budget=32)
    rn.index(0)
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    tokens = [5, 40]
    scores = _oracle_scores(wl, 0, tokens)
    _check_indexer_rows(rn, 0, scores, tokens, token_topk=False, page_topk=True)
    _check_decode_attend(dsa, wl, rn, 0, 0, tokens, scores, unit=wl.rg.page_size)


def test_single_prefill(dsa):
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.single_prefill(device="cuda")
    rn = LayerRunner(wl, "cuda")
    assert rn.prefill and rn.u_max == 128
    rn.index(0)
    rn.union(0)
    torch.cuda.synchronize()
    assert rn.status.item() == 0  # also: no block union exceeded u_max
    tokens = [0, 100, 255, 256, 2047, 2048, 5000, 8191]
    scores = _oracle_scores(wl, 0, tokens)
    _check_indexer_rows(rn, 0, scores, tokens)
    _check_union_and_qblock(dsa, wl, rn, 0, 0, tokens)


def test_ragged_mixed_with_indexshare(dsa):
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.ragged_mixed(device="cuda")
    rn = LayerRunner(wl, "cuda")
    assert rn.src_slot == [0, 0, 0, 1] and rn.num_full == 2
    rg = wl.rg
    ends = [int(x) for x in rg.cu_q_lens]
    # decode rows, the first and last token of every extend, a block boundary
    tokens = sorted({0, 47, 255, 256} | {ends[s] for s in range(48, rg.S)} | {ends[s + 1] - 1 for s in range(48, rg.S)})
    for layer in range(4):
        rn.layer_step(layer)
        torch.cuda.synchronize()
        assert rn.status.item() == 0, f"layer {layer}"
        slot = rn.src_slot[layer]
        if rn.full_slot[layer] >= 0:
            scores = _oracle_scores(wl, slot, tokens)
            _check_indexer_rows(rn, slot, scores, tokens)
        if layer in (0, 1, 3):  # full slot 0, a shared layer reusing it, full slot 1
            _check_union_and_qblock(dsa, wl, rn, layer, slot, tokens)
