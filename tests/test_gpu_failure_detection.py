"""Failure detection without a GPU fault: a bounded pipeline wait on a
barrier that nothing arrives on runs out, reports DSA_STATUS_TIMEOUT in the
device status word, and the kernel returns normally: the context stays
usable and the next call computes correctly. Host-side fault injection
(malformed metadata, out-of-range pages, overflowing unions, a shared layer
before any full one) is covered by the parity and ABI tests."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def test_bounded_wait_reports_timeout_and_context_survives(dsa):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.dsa_selftest_wait_timeout(st, limit_clocks=2_000_000)  # about a millisecond
    torch.cuda.synchronize()
    assert st.item() & 8  # DSA_STATUS_TIMEOUT
    # the same context keeps working
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.tensor([[130, 5, -1, 64]], dtype=torch.int32, device="cuda")
    pages, counts = dsa.dsa_topk_pages_from_tokens(topk, ps=64, max_pages=8, cap=4, dev_status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    assert pages.cpu().tolist() == [[0, 1, 2, -1]] and counts.item() == 3
