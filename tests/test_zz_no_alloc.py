"""The no-allocation decode entry point (dsa_sparse_mla_decode_noalloc).

Some callers cannot allocate device memory on this path, for example a plugin
that an inference engine hands only its input and output buffers, or code
that must not allocate once it is running. For them the library keeps the
split-key scratch of the decode attention in a device array built into the
library. This checks, through the C ABI, that two calls in a row (the second
one finding the first call's leftovers in that array) give the same output
as the workspace-based entry point, within the attention tolerance of the
other parity tests, and that both match the CPU oracle. The shape is one
whose key lists are split across CTAs, so the built-in array is in use
(asserted through the workspace query, which is non-zero exactly when the
split path runs).

The file name sorts last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as DI
import oracle as O
from gpu_util import ATTN_MAX_ABS, ATTN_REL_L2, check_attention, meta_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _selection(rg, K, seed):
    rng = np.random.default_rng(seed)
    sel = np.full((rg.T, K), -1, np.int32)
    for t in range(rg.T):
        n = int(rg.seq_lens[t])  # decode: each token sees its whole request
        m = min(K, n)
        sel[t, :m] = np.sort(rng.choice(n, size=m, replace=False))
    return sel


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    return rel <= ATTN_REL_L2 and np.abs(a - b).max() <= ATTN_MAX_ABS, rel


def test_noalloc_matches_workspace_entry_point_twice(dsa):
    dev = torch.device("cuda")
    # four decode requests x 128 heads: few enough CTAs that the key list is
    # split across several CTAs, so the built-in scratch is in use
    wl = DI.random_small(901, [1, 1, 1, 1], [700, 2000, 300, 4000], H=128, k=256)
    rg = wl.rg
    assert dsa.dsa_sparse_mla_decode_workspace_size(rg.T, 128) > 0, "this shape must take the split-key path"
    meta = meta_to(rg, dev)
    q, kv = wl.q[0].to(dev), wl.kv[0].to(dev)
    q_np, kv_np = wl.q[0].float().numpy(), wl.kv[0].float().numpy()
    for call, seed in enumerate((1, 2)):
        sel = torch.from_numpy(_selection(rg, 256, seed)).to(dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        ref, ref_lse = dsa.dsa_sparse_mla_decode(q, kv, *meta, sel, unit=1, sm_scale=wl.sm_scale, want_lse=True)
        got, got_lse = dsa.dsa_sparse_mla_decode_noalloc(q, kv, *meta, sel, unit=1, sm_scale=wl.sm_scale,
                                                         want_lse=True, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"call {call}: device status {st.item():#x}"
        ok, rel = _close(got, ref)
        assert ok, f"call {call}: rel-L2 {rel:.3e} against dsa_sparse_mla_decode"
        o_ref, _ = O.sparse_mla(q_np, kv_np, rg.seq_lens, rg.cu_q_lens, rg.cu_kv_lens, rg.page_indices,
                                sel.cpu().numpy(), 1, wl.sm_scale, 512)
        check_attention(got, o_ref, f"call {call}: no-allocation entry point against the oracle")
        np.testing.assert_allclose(got_lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-5, atol=1e-5)
