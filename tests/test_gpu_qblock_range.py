"""The token-range form of the query-block prefill attention
(dsa_sparse_mla_prefill_qblock_range): computing a layer's output in a few
token ranges gives, row for row and bit for bit, the output of the single
call, and a range writes no row outside itself."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import check_attention, f32, meta_np, meta_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def test_token_ranges_match_the_full_call(dsa):
    dev = torch.device("cuda")
    ps, QB, K = 64, 32, 3
    wl = DI.random_small(523, [1, 70, 1, 45], [900, 1300, 700, 600], H=128, page_size=ps, k=64, k_pages=K)
    rg = wl.rg
    meta = meta_to(rg, dev)
    rng = np.random.default_rng(5)
    nvis = O.visible_len(rg.seq_lens, rg.cu_q_lens)
    sel = np.full((rg.T, K), -1, np.int32)
    for t in range(rg.T):
        npg = -(-int(nvis[t]) // ps)
        ch = rng.choice(npg, size=min(K, npg), replace=False)
        sel[t, : len(ch)] = np.sort(ch)
    units, member, counts = dsa.dsa_build_block_union(torch.from_numpy(sel).to(dev), QB=QB, cu_q_lens=meta[1],
                                                      cu_kv_lens=meta[2], ps=ps, PTW=rg.PTW)
    q, kv = wl.q[0].to(dev), wl.kv[0].to(dev)
    full = dsa.dsa_sparse_mla_prefill_qblock(q, kv, *meta, units, member, counts, QB=QB, sm_scale=wl.sm_scale)
    sentinel = torch.full_like(full, 7.0)
    pieces = sentinel.clone()
    bounds = [0, 1, 40, 77, 77, rg.T]  # ragged ranges, one empty
    for b, e in zip(bounds[:-1], bounds[1:]):
        dsa.dsa_sparse_mla_prefill_qblock(q, kv, *meta, units, member, counts, QB=QB, sm_scale=wl.sm_scale,
                                          o=pieces, t_range=(b, e))
    torch.cuda.synchronize()
    assert torch.equal(pieces.view(torch.int16), full.view(torch.int16))
    # one range alone leaves every other row untouched
    part = sentinel.clone()
    dsa.dsa_sparse_mla_prefill_qblock(q, kv, *meta, units, member, counts, QB=QB, sm_scale=wl.sm_scale, o=part,
                                      t_range=(40, 77))
    torch.cuda.synchronize()
    assert torch.equal(part[40:77].view(torch.int16), full[40:77].view(torch.int16))
    assert torch.equal(part[:40], sentinel[:40]) and torch.equal(part[77:], sentinel[77:])
    ref, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=ps, sm_scale=wl.sm_scale,
                          Dv=512)
    check_attention(pieces, ref)
