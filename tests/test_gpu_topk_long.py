"""Top-k on rows longer than the shared-memory staging capacity (the path that
streams the row from L2 and collects winners unordered), including rows with
massive exact ties (tie list sorted in shared memory, and the ordered
fallback when the ties overflow it)."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import check_scores, check_topk_rows, f32, meta_np, meta_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _long_workload():
    kv_lens = [40000, 33000, 40000, 36001]
    wl = DI.random_small(77, [1] * len(kv_lens), kv_lens, H=16, k=2048)
    rg = wl.rg
    ps = rg.page_size
    kc = wl.kcache[0].view(-1, 128)
    # request 1: keys drawn from 4 distinct vectors -> 4 distinct scores, ~8K-way ties
    base = int(rg.cu_kv_lens[1]) // ps
    rows = (rg.page_indices[base + np.arange(33000) // ps].astype(np.int64) * ps + np.arange(33000) % ps)
    protos = torch.randn((4, 128), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    kc[torch.from_numpy(rows)] = protos[torch.from_numpy(np.arange(33000) % 4)]
    # request 2: a zero query -> every score is 0 (40000-way tie)
    wl.q_idx[2] = 0
    return wl


def test_long_rows_token_topk(dsa):
    dev = torch.device("cuda")
    wl = _long_workload()
    rg = wl.rg
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    topk, vals = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta_to(rg, dev),
                                      k=wl.k, max_kv=rg.max_kv, want_scores=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = O.indexer_scores(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg))
    ref = np.stack([O.topk_of_row(r, wl.k) for r in rows])
    got = topk.cpu().numpy()
    check_topk_rows(got, ref, wl.k, rows)
    check_scores(vals.cpu().numpy(), got, rows)
    # the all-tie row must take exactly the lowest k positions
    assert np.array_equal(got[2], np.arange(wl.k))
    # the 4-value row: the winners are exact (no near-tie freedom between distinct values)
    assert np.array_equal(got[1], ref[1])


def test_long_rows_k_above_the_winner_lists(dsa):
    """k larger than the shared-memory candidate and winner lists (half the
    staging area each): the winners are emitted in position order straight
    from the score row."""
    dev = torch.device("cuda")
    wl = _long_workload()
    rg = wl.rg
    k = 20000
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    topk = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta_to(rg, dev), k=k,
                                max_kv=rg.max_kv, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = O.indexer_scores(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg))
    ref = O.topk_rows_of(rows, k)
    got = topk.cpu().numpy()
    check_topk_rows(got, ref, k, rows)
    assert np.array_equal(got[2], np.arange(k))  # the all-tie row: the lowest k positions
