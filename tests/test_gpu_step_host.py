"""The host-buffer step (LayerRunner.step_host: copies on two streams, then
the layer calls) gives the outputs of the resident step, called eagerly and
replayed from a CUDA graph; covers decode (split keys), prefill with
IndexShare, and repeated replays. Selections must match exactly; outputs to
one bf16 rounding, since the last CTA of a split-key row adds the splits
starting from its own, and which CTA is last may change from run to run."""
import pytest
import torch

import dsa_inputs as DI

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def _workload(kind):
    if kind == "decode":
        return DI.random_small(901, [1, 1, 1, 1], [900, 2100, 64, 3000], H=32, k=256, k_pages=4)
    wl = DI.random_small(902, [40, 1, 9], [300, 700, 1000], H=32, k=128, k_pages=3)
    # a second, shared layer (IndexShare: it reuses the first layer's tables)
    wl.q.append(DI.randn(tuple(wl.q[0].shape), 903, "q_layer1").to(torch.bfloat16))
    wl.kv.append(DI.randn(tuple(wl.kv[0].shape), 903, "kv_layer1").to(torch.bfloat16))
    wl.indexer_types = [0, 1]
    return wl


def _host(rn):
    pin = lambda t: t.detach().to("cpu").pin_memory()
    return dict(q_idx=pin(rn.q_idx), w=pin(rn.w), q=[pin(x) for x in rn.q], meta=[pin(m) for m in rn.meta],
                topk=torch.empty(rn.topk[0].shape, dtype=torch.int32).pin_memory(),
                o=[torch.empty(x.shape, dtype=torch.bfloat16).pin_memory() for x in rn.o])


def _same_outputs(got, ref):
    for a, b in zip(got, ref):
        torch.testing.assert_close(a.float(), b.float(), rtol=2.0 ** -7, atol=1e-4)


def _call(rn, h, side):
    rn.step_host(h["q_idx"], h["w"], h["q"], h["meta"], h["topk"], h["o"], side)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_step_host_matches_resident_step(dsa, kind):
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    dev = torch.device("cuda")
    wl = _workload(kind)
    if kind == "prefill":
        wl.QB, wl.u_max = 32, 0
    rn = LayerRunner(wl, dev, prefill=(kind == "prefill"))
    rn.step()
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    ref_topk = rn.topk[0].cpu().clone()
    ref_o = [x.cpu().clone() for x in rn.o]

    h = _host(rn)
    side = torch.cuda.Stream(dev)
    # clobber the device inputs and outputs: everything must come from the host buffers
    for t in [rn.q_idx, *rn.q]:
        t.zero_()
    for x in rn.o:
        x.fill_(7.0)
    _call(rn, h, side)
    torch.cuda.synchronize()
    assert rn.status.item() == 0
    assert torch.equal(h["topk"], ref_topk)
    _same_outputs(h["o"], ref_o)

    # the same step captured once and replayed: fresh host outputs each time
    s2 = torch.cuda.Stream(dev)
    s2.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s2):
        _call(rn, h, side)
    torch.cuda.synchronize()
    for _ in range(2):
        h["topk"].fill_(-5)
        for x in h["o"]:
            x.zero_()
        for t in [rn.q_idx, *rn.q]:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(h["topk"], ref_topk)
        _same_outputs(h["o"], ref_o)
