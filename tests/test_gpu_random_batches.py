"""Seeded random ragged batches through the whole path (indexer with both
top-k outputs, block union, query-block and token decode attention) against
the oracle: request mixes with empty, single-token and multi-token requests,
page sizes 32/64/128, k from 16 to 2048, block sizes 32..256."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import check_attention, check_topk_rows, f32, member_bits_to_int8, meta_np, meta_to

pytestmark = pytest.mark.gpu

N_CASES = 30


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _config(case):
    rng = np.random.default_rng(9000 + case)
    S = int(rng.integers(1, 7))
    ps = int(rng.choice([32, 64, 128]))
    q_lens, kv_lens = [], []
    for _ in range(S):
        kind = rng.integers(0, 4)
        kv = int(rng.integers(1, 6000))
        ql = 1 if kind == 0 else (0 if kind == 1 and S > 1 else int(rng.integers(1, min(kv, 64) + 1)))
        q_lens.append(min(ql, kv))
        kv_lens.append(kv)
    if sum(q_lens) == 0:
        q_lens[0] = 1
    k = int(rng.choice([16, 64, 257, 2048]))
    k_pages = int(rng.integers(1, 9))
    H = 128 if rng.random() < 0.2 else 16
    QB = int(rng.choice([32, 64, 256]))
    return q_lens, kv_lens, ps, k, k_pages, H, QB


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_batch(dsa, case):
    q_lens, kv_lens, ps, k, k_pages, H, QB = _config(case)
    dev = torch.device("cuda")
    wl = DI.random_small(1000 + case, q_lens, kv_lens, H=H, page_size=ps, k=k, k_pages=k_pages)
    rg = wl.rg
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pages, topk = dsa.dsa_indexer_page_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta,
                                            k_pages=k_pages, max_kv=rg.max_kv, k=k, with_tokens=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = O.indexer_scores(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg))
    check_topk_rows(topk.cpu().numpy(), O.topk_rows_of(rows, k), k, rows)
    prow = [O.page_scores_of_row(r, ps) for r in rows]
    check_topk_rows(pages.cpu().numpy(), O.topk_rows_of(prow, k_pages), k_pages, prow, what="page top-k")
    # the block tables and both attention forms over the library's own
    # selections (the oracle attends exactly the same keys)
    sel = pages.cpu().numpy()
    u_max = min(QB * k_pages, rg.PTW)
    units, member, counts = dsa.dsa_build_block_union(pages, QB=QB, u_max=u_max, cu_q_lens=meta[1],
                                                      cu_kv_lens=meta[2], ps=ps, PTW=rg.PTW, dev_status=st)
    torch.cuda.synchronize()
    ru, rm, rc = O.block_union(O.lift_units(sel, rg.cu_q_lens, rg.cu_kv_lens, ps), QB, u_max)
    assert np.array_equal(units.cpu().numpy(), ru)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(member_bits_to_int8(member.cpu().numpy().view(np.uint32), QB), rm)
    o = dsa.dsa_sparse_mla_prefill_qblock(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, units, member, counts, QB=QB,
                                          sm_scale=wl.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    ref_o, _ = O.qblock_attend(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), units=ru, member=rm, counts=rc, QB=QB,
                               sm_scale=wl.sm_scale, Dv=512)
    check_attention(o, ref_o, "qblock")
    o2 = dsa.dsa_sparse_mla_decode(wl.q[0].to(dev), wl.kv[0].to(dev), *meta, topk, unit=1, sm_scale=wl.sm_scale,
                                   dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref2, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=topk.cpu().numpy(), unit=1,
                           sm_scale=wl.sm_scale, Dv=512)
    check_attention(o2, ref2, "decode")
