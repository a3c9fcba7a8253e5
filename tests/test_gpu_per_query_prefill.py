"""The per-query prefill shape (the pages' baseline that the query-block
kernel replaces): prefill and extend queries through dsa_sparse_mla_decode
with page units give the same attention as dsa_sparse_mla_prefill_qblock on
the block unions of the same page selections, and both match the oracle.
The pages state this parity ("same masked-softmax math")."""
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


@pytest.mark.parametrize("q_lens,kv_lens", [([300], [300]), ([1, 120, 2, 70], [900, 500, 65, 70])])
def test_per_query_equals_qblock(dsa, q_lens, kv_lens):
    dev = torch.device("cuda")
    ps, K, QB = 64, 4, 64
    wl = DI.random_small(31 + len(q_lens), q_lens, kv_lens, H=128, page_size=ps, k=64, k_pages=K)
    rg = wl.rg
    rng = np.random.default_rng(3)
    nvis = O.visible_len(rg.seq_lens, rg.cu_q_lens)
    sel = np.full((rg.T, K), -1, np.int32)
    for t in range(rg.T):
        n = -(-int(nvis[t]) // ps)
        if n:
            m = min(K, n)
            sel[t, :m] = np.sort(rng.choice(n, size=m, replace=False))
    meta = meta_to(rg, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    q, kv = wl.q[0].to(dev), wl.kv[0].to(dev)
    sel_d = torch.from_numpy(sel).to(dev)
    o_pq = dsa.dsa_sparse_mla_decode(q, kv, *meta, sel_d, unit=ps, sm_scale=wl.sm_scale, dev_status=st)
    units, member, counts = dsa.dsa_build_block_union(sel_d, QB=QB, u_max=min(QB * K, rg.PTW), cu_q_lens=meta[1],
                                                      cu_kv_lens=meta[2], ps=ps, PTW=rg.PTW, dev_status=st)
    o_qb = dsa.dsa_sparse_mla_prefill_qblock(q, kv, *meta, units, member, counts, QB=QB, sm_scale=wl.sm_scale,
                                             dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, _ = O.sparse_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sel=sel, unit=ps, sm_scale=wl.sm_scale, Dv=512)
    check_attention(o_pq, ref, "per-query prefill")
    check_attention(o_qb, ref, "query-block prefill")
    a, b = o_pq.float().cpu().numpy(), o_qb.float().cpu().numpy()
    assert np.linalg.norm(a - b) <= 1e-2 * max(np.linalg.norm(b), 1e-30)
