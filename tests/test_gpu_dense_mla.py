"""Dense causal MLA fallback (dsa_dense_mla) against the oracle's dense_mla:
decode rows, a prefill and a ragged mix, page sizes 32/64, with and without
a sliding window and a logit soft cap, at the attention tolerance."""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import check_attention, f32, meta_np, meta_to

pytestmark = pytest.mark.gpu

CASES = {
    "decode": ([1, 1, 1], [700, 64, 2100]),
    "prefill": ([300], [300]),
    "mixed": ([1, 45, 0, 7], [500, 300, 40, 1000]),
}


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("ps,window,cap", [(64, 0, 0.0), (32, 0, 0.0), (64, 100, 0.0), (64, 0, 5.0),
                                           (64, 257, 2.0)])
def test_dense_mla_matches_oracle(dsa, case, ps, window, cap):
    dev = torch.device("cuda")
    q_lens, kv_lens = CASES[case]
    wl = DI.random_small(50 + ps + window + len(case), q_lens, kv_lens, H=128, page_size=ps)
    rg = wl.rg
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o = dsa.dsa_dense_mla(wl.q[0].to(dev), wl.kv[0].to(dev), *meta_to(rg, dev), max_kv=int(max(kv_lens)),
                          sm_scale=wl.sm_scale, sliding_window=window, soft_cap=cap, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = O.dense_mla(f32(wl.q[0]), f32(wl.kv[0]), **meta_np(rg), sm_scale=wl.sm_scale, Dv=512,
                      sliding_window=window or None, soft_cap=cap or None)
    check_attention(o, ref, f"dense {case} window={window} cap={cap}")
