"""Paged write-back (dsa_paged_write_back) against the oracle's
paged_write_back, bit for bit: ragged batches with decode rows, extends, an
empty request and a prefill, page sizes 32/64/128, the latent cache (576
columns of a 576- or 640-wide row) and the indexer key cache (128 columns);
plus a bad page table, which is reported in the status word."""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _batch(seed, ps, q_lens, kv_lens, spare=3):
    rng = np.random.default_rng(seed)
    q_lens, kv_lens = np.asarray(q_lens), np.asarray(kv_lens)
    npages = -(-kv_lens // ps)
    cu_kv = np.concatenate([[0], np.cumsum(npages * ps)]).astype(np.int32)
    P = int(npages.sum()) + spare
    page_indices = rng.permutation(P)[: int(npages.sum())].astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return rng, kv_lens.astype(np.int32), cu_q, cu_kv, page_indices, P


def _bits(rng, shape):
    return (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("ps,width,D", [(64, 576, 576), (32, 640, 576), (128, 128, 128), (64, 640, 128)])
def test_write_back_matches_oracle(dsa, ps, width, D):
    dev = torch.device("cuda")
    rng, kv, cu_q, cu_kv, pi, P = _batch(7 + ps + width, ps, [1, 37, 0, 300, 1], [5000, 700, 64, 300, 1])
    T = int(cu_q[-1])
    cache = _bits(rng, (P, ps, width))
    rows = _bits(rng, (T, D))
    ref = O.paged_write_back(cache, rows, kv, cu_q, cu_kv, pi)
    g_cache = torch.from_numpy(cache.view(np.int16)).to(dev).view(torch.bfloat16)
    g_rows = torch.from_numpy(rows.view(np.int16)).to(dev).view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    meta = [torch.from_numpy(a).to(dev) for a in (kv, cu_q, cu_kv, pi)]
    dsa.dsa_paged_write_back(g_rows, g_cache, *meta, D=D, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = g_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("ps", [32, 64, 128])
def test_write_back_pair_matches_oracle(dsa, ps):
    """Both caches of a full layer (latent rows, 576 of 640 columns; indexer
    keys, 128) written by one launch: each equals the oracle's single-cache
    write-back, bit for bit."""
    dev = torch.device("cuda")
    rng, kv, cu_q, cu_kv, pi, P = _batch(11 + ps, ps, [1, 37, 0, 300, 1], [5000, 700, 64, 300, 1])
    T = int(cu_q[-1])
    c0, c1 = _bits(rng, (P, ps, 640)), _bits(rng, (P, ps, 128))
    r0, r1 = _bits(rng, (T, 576)), _bits(rng, (T, 128))
    ref0 = O.paged_write_back(c0, r0, kv, cu_q, cu_kv, pi)  # the first 576 columns
    ref1 = O.paged_write_back(c1, r1, kv, cu_q, cu_kv, pi)
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    g0, g1, gr0, gr1 = to(c0), to(c1), to(r0), to(r1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    meta = [torch.from_numpy(a).to(dev) for a in (kv, cu_q, cu_kv, pi)]
    dsa.dsa_paged_write_back_pair(gr0, g0, gr1, g1, *meta, D0=576, D1=128, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(g0.view(torch.int16).cpu().numpy().view(np.uint16), ref0)
    assert np.array_equal(g1.view(torch.int16).cpu().numpy().view(np.uint16), ref1)


def test_write_back_reports_bad_page_table(dsa):
    dev = torch.device("cuda")
    rng, kv, cu_q, cu_kv, pi, P = _batch(3, 64, [2, 3], [130, 70])
    T = int(cu_q[-1])
    bad = pi.copy()
    bad[-1] = P + 5  # the last request's last page points outside the pool
    cache = _bits(rng, (P, 64, 576))
    rows = _bits(rng, (T, 576))
    g_cache = torch.from_numpy(cache.view(np.int16)).to(dev).view(torch.bfloat16)
    g_rows = torch.from_numpy(rows.view(np.int16)).to(dev).view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    meta = [torch.from_numpy(a).to(dev) for a in (kv, cu_q, cu_kv, bad)]
    dsa.dsa_paged_write_back(g_rows, g_cache, *meta, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 2  # DSA_STATUS_BAD_METADATA
    # tokens whose pages are valid were still written
    ok_ref = O.paged_write_back(cache, rows[:2], kv[:1], cu_q[:2], cu_kv[:2], pi)
    got = g_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    r = O.physical_rows(cu_kv, pi, 64, 0, [128, 129])
    assert np.array_equal(got.reshape(-1, 576)[r], ok_ref.reshape(-1, 576)[r])
