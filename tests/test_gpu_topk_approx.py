"""Approximate token top-k (dsa_indexer_topk_approx) against the oracle's
approx_topk_of_row. The bin maxima are decided on fp32 scores, which the
GPU and the oracle round differently, so the check is: the count is exact;
every selected position is the largest score of its bin up to the score
tolerance; the selection equals the oracle's except where a decision is
within the score tolerance (a near-tie inside a bin or at the k-th bin
maximum); with enough bins it is the exact top-k. The recall against the
exact top-k is reported."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import SCORE_RTOL, f32, meta_np, meta_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _near(a, b, scale):
    return abs(float(a) - float(b)) <= SCORE_RTOL * scale


@pytest.mark.parametrize("over", [1, 4])
def test_approx_topk_against_oracle(dsa, over, capsys):
    dev = torch.device("cuda")
    wl = DI.random_small(71 + over, [1, 1, 1, 30], [5000, 900, 130, 3000], k=256)
    rg = wl.rg
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = dsa.dsa_indexer_topk_approx(wl.q_idx.to(dev), wl.w.to(dev), wl.kcache[0].to(dev), *meta_to(rg, dev),
                                      k=wl.k, max_kv=int(rg.seq_lens.max()), over=over, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = got.cpu().numpy()
    scores = O.indexer_scores(f32(wl.q_idx), f32(wl.w), f32(wl.kcache[0]), **meta_np(rg))
    hits = tot = 0
    for t, s in enumerate(scores):
        n, k = len(s), wl.k
        g = got[t][got[t] >= 0]
        assert len(g) == min(k, n) and np.all(np.diff(g) > 0), t
        ref = O.approx_topk_of_row(s, k, over)
        ref = ref[ref >= 0]
        scale = max(float(np.abs(s).max()), 1e-30)
        B = min(n, over * k)
        for j in g:  # the largest of its bin, up to the tolerance
            assert _near(s[j], s[np.arange(j % B, n, B)].max(), scale), (t, j)
        kth = np.sort([s[np.arange(b, n, B)].max() for b in range(B)])[::-1][min(k, B) - 1]
        for j in set(g.tolist()) ^ set(ref.tolist()):  # differences only at near-ties
            bmax = s[np.arange(j % B, n, B)].max()
            assert _near(s[j], bmax, scale) or _near(bmax, kth, scale), (t, j)
        exact = set(O.topk_of_row(s, k).tolist()) - {-1}
        hits += len(exact & set(g.tolist()))
        tot += len(exact)
    with capsys.disabled():
        print(f"\napprox top-k over={over}: recall {hits / max(tot, 1):.4f} against the exact top-k")
    if over >= 4:
        assert hits / tot >= 0.9
