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


def test_many_long_rows_token_topk(dsa):
    """More long rows than twice the SM count (the launch shape of a long
    prefill): random rows, rows of four distinct score values (tie lists
    longer than the winner lists) and all-zero rows, checked on a sample of
    rows against the oracle."""
    dev = torch.device("cuda")
    n_per = dsa.dsa_device_sm_count() + 8
    kv_lens = [36000, 33000]
    wl = DI.random_small(79, [n_per, n_per], kv_lens, H=16, k=2048)
    rg = wl.rg
    ps = rg.page_size
    kc = wl.kcache[0].view(-1, 128)
    base = int(rg.cu_kv_lens[1]) // ps
    n1 = kv_lens[1]
    rows = rg.page_indices[base + np.arange(n1) // ps].astype(np.int64) * ps + np.arange(n1) % ps
    protos = torch.randn((4, 128), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    kc[torch.from_numpy(rows)] = protos[torch.from_numpy(np.arange(n1) % 4)]
    zero_tok = [3, 40, n_per - 1]
    wl.q_idx[zero_tok] = 0
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    topk = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta_to(rg, dev),
                                k=wl.k, max_kv=rg.max_kv, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    T = rg.T
    sample = sorted(set(zero_tok) | {0, 1, n_per // 2, n_per - 2, n_per, n_per + 1, T // 2 + 7, T - 1}
                    | set(np.random.default_rng(3).choice(T, 8, replace=False).tolist()))
    ref, srows = O.indexer_topk(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg), k=wl.k,
                                tokens=np.asarray(sample))
    got = topk.cpu().numpy()[sample]
    check_topk_rows(got, ref, wl.k, srows)
    for i, t in enumerate(sample):
        if t in zero_tok:
            assert np.array_equal(got[i], np.arange(wl.k))  # all-tie rows: the lowest k positions
        if t >= n_per:
            assert np.array_equal(got[i], ref[i])  # four distinct values: no near-tie freedom


def test_long_rows_sample_misleads(dsa):
    """A row whose evenly spaced positions (the ones a strided sample of the
    row sees) hold its largest scores: a threshold taken from such a sample
    admits fewer than k keys, and the selection must still be exact."""
    dev = torch.device("cuda")
    n = 40960
    wl = DI.random_small(81, [1, 1], [n, 37000], H=16, k=2048)
    rg = wl.rg
    ps = rg.page_size
    kc = wl.kcache[0].view(-1, 128)
    qsum = wl.q_idx[0].float().sum(0)
    v = (qsum / qsum.norm() * 16).to(torch.bfloat16)
    planted = np.arange(0, n, n // 1024)
    base = int(rg.cu_kv_lens[0]) // ps
    rows = rg.page_indices[base + planted // ps].astype(np.int64) * ps + planted % ps
    kc[torch.from_numpy(rows)] = v
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    topk = dsa.dsa_indexer_topk(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta_to(rg, dev),
                                k=wl.k, max_kv=rg.max_kv, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, srows = O.indexer_topk(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg), k=wl.k)
    # the planted positions are the row's 1024 largest scores
    assert set(np.argsort(-srows[0].astype(np.float64), kind="stable")[:1024].tolist()) == set(planted.tolist())
    got = topk.cpu().numpy()
    check_topk_rows(got, ref, wl.k, srows)


@pytest.mark.parametrize("ps,full_pages", [(64, 600), (64, 34380), (128, 600)])
def test_page_topk_folds_visible_granules(dsa, ps, full_pages):
    """Page scores are folded from 32-key granule maxima. A page whose tail is
    not visible must ignore the granules past the visible length even when
    the workspace still holds larger values there from an earlier call with a
    longer row. With 34 380 full pages the rows exceed every shared-memory
    stage (a folding pass runs first); with 600 they are folded while staged.
    Keys are zero except planted copies of two vectors A and B = A / 2, so
    the expected selection follows from the oracle's scores of A and B."""
    dev = torch.device("cuda")
    k_pages, seed = 16, 83
    n_long, n_short = full_pages * ps + 60, full_pages * ps + 20  # same page count
    q_lens = [1, 1, 1, 1]
    rgs = [DI.make_ragged(q_lens, [n, 1000, 1500, 700], ps, master_seed=seed, spare_pages=2)
           for n in (n_long, n_short)]
    assert np.array_equal(rgs[0].page_indices, rgs[1].page_indices)
    T, P = 4, rgs[0].num_pages
    q_idx = DI.randn((T, DI.INDEX_HEADS, DI.INDEX_DIM), seed, "q_idx").to(torch.bfloat16)
    w = DI.rand((T, DI.INDEX_HEADS), seed, "w") / np.sqrt(DI.INDEX_HEADS)
    qs = q_idx[0].float().sum(0)
    A = (qs / qs.norm() * 16).to(torch.bfloat16)
    B = (A.float() * 0.5).to(torch.bfloat16)
    sA, sB = O.indexer_score_row(f32(q_idx[0]), f32(w[0]), f32(torch.stack([A, B])))
    assert sA > sB > 0
    # request 0: zero keys with planted A / B keys; the other requests' keys N(0,1)
    pi = rgs[0].page_indices
    last = full_pages  # index of request 0's partly visible page
    kc = torch.zeros((P, ps, DI.INDEX_DIM), dtype=torch.bfloat16)
    rest = torch.from_numpy(pi[last + 1:].astype(np.int64))
    kc[rest] = DI.randn((len(rest), ps, DI.INDEX_DIM), seed, "kcache").to(torch.bfloat16)
    pa = [5, full_pages // 2, full_pages - 1]
    pb = sorted(set(np.linspace(1, full_pages - 2, 40).astype(int).tolist()) - set(pa))
    for p in pa:
        kc[int(pi[p]), 7] = A
    for p in pb:
        kc[int(pi[p]), 33] = B
    kc[int(pi[last]), 45] = A  # visible at n_long (offset 45 < 60), past n_short (45 >= 20)
    kcd = kc.to(dev)
    ws = torch.empty(dsa.dsa_indexer_workspace_size(T, 4, n_long, ps), dtype=torch.uint8, device=dev)
    got = []
    for rg in rgs:
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        pages = dsa.dsa_indexer_page_topk(q_idx.to(dev), w.to(dev), kcd, *meta_to(rg, dev), k_pages=k_pages,
                                          max_kv=n_long, ws=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        got.append(pages.cpu().numpy())
    # request 0: the A pages, then the lowest-index B pages (ties to the lower index)
    want_long = sorted(pa + [last] + pb[: k_pages - len(pa) - 1])
    want_short = sorted(pa + pb[: k_pages - len(pa)])
    assert got[0][0].tolist() == want_long
    assert got[1][0].tolist() == want_short
    # requests 1..3 against the oracle's page top-k
    ref, srows = O.indexer_page_topk(f32(q_idx), f32(w), kc.view(torch.int16).numpy(), **meta_np(rgs[1]),
                                     k_pages=k_pages, tokens=np.arange(1, T))
    prow = [O.page_scores_of_row(r, ps) for r in srows]
    check_topk_rows(got[1][1:], ref, k_pages, prow, what="page top-k")


def test_long_context_chunked_prefill_rows(dsa):
    """A chunk of new tokens at the end of a 600 K-token context: more rows
    than twice the SM count, token rows of 600 K scores (read once with a
    sampled threshold) and page rows of 9 K pages (longer than the short
    blocks' stage: the wide blocks fold granules while staging). Sampled rows
    are checked against the oracle."""
    dev = torch.device("cuda")
    n_new = 2 * dsa.dsa_device_sm_count() + 16
    ctx = 600_000
    ps, k, k_pages, seed = 64, 2048, 32, 85
    rg = DI.make_ragged([n_new], [ctx], ps, master_seed=seed, spare_pages=1)
    T = rg.T
    q_idx = DI.randn((T, DI.INDEX_HEADS, DI.INDEX_DIM), seed, "q_idx").to(torch.bfloat16)
    w = DI.rand((T, DI.INDEX_HEADS), seed, "w") / np.sqrt(DI.INDEX_HEADS)
    kc = DI.randn((rg.num_pages, ps, DI.INDEX_DIM), seed, "kcache").to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pages, topk = dsa.dsa_indexer_page_topk(q_idx.to(dev), w.to(dev), kc.to(dev), *meta_to(rg, dev),
                                            k_pages=k_pages, max_kv=ctx, k=k, with_tokens=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    sample = np.array(sorted({0, 1, T // 3, T // 2, T - 2, T - 1}
                             | set(np.random.default_rng(5).choice(T, 6, replace=False).tolist())))
    kb = kc.view(torch.int16).numpy()
    ref, srows = O.indexer_topk(f32(q_idx), f32(w), kb, **meta_np(rg), k=k, tokens=sample)
    check_topk_rows(topk.cpu().numpy()[sample], ref, k, srows)
    pref = O.topk_rows_of([O.page_scores_of_row(r, ps) for r in srows], k_pages)
    prow = [O.page_scores_of_row(r, ps) for r in srows]
    check_topk_rows(pages.cpu().numpy()[sample], pref, k_pages, prow, what="page top-k")
