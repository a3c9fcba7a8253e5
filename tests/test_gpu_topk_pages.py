"""Token top-k -> page list (dsa_topk_pages_from_tokens) against the
oracle's topk_pages_of_tokens, bit for bit, including truncation at the cap,
empty rows, rows in any order and an out-of-range position (status)."""
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


@pytest.mark.parametrize("ps,cap,max_pages", [(64, 512, 2048), (32, 40, 4096), (128, 512, 1 << 14)])
def test_topk_pages_match_oracle(dsa, ps, cap, max_pages):
    rng = np.random.default_rng(ps + cap)
    T, K = 37, 2048
    topk = np.full((T, K), -1, np.int32)
    for t in range(T):
        n = int(rng.integers(0, K + 1)) if t % 5 else (0 if t == 0 else K)
        span = max_pages * ps
        row = rng.choice(span, size=n, replace=False) if t % 3 else np.sort(rng.choice(span, size=n, replace=False))
        topk[t, :n] = row
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pages, counts = dsa.dsa_topk_pages_from_tokens(torch.from_numpy(topk).cuda(), ps=ps, max_pages=max_pages,
                                                   cap=cap, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    pages, counts = pages.cpu().numpy(), counts.cpu().numpy()
    for t in range(T):
        ref, n = O.topk_pages_of_tokens(topk[t], ps, cap)
        assert np.array_equal(pages[t], ref), t
        assert counts[t] == n, t


def test_topk_pages_reports_out_of_range(dsa):
    topk = torch.tensor([[3, 70, 64 * 10, -1]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pages, counts = dsa.dsa_topk_pages_from_tokens(topk, ps=64, max_pages=4, cap=4, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 4  # DSA_STATUS_BAD_INDEX
    assert pages.cpu().tolist() == [[0, 1, -1, -1]] and counts.item() == 2
