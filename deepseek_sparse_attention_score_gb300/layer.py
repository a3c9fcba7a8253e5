"""One DSA layer step on a resident batch, built from the C-ABI calls.

Every layer first writes its new tokens' rows into the paged caches (the
latent row of every layer, the indexer key on full layers; the backend's
_scatter_paged step that precedes the path). Decode batches then run indexer
-> token top-k (or page top-k with a page budget) -> sparse MLA decode.
Prefill / mixed batches run, on full layers, the indexer once for both the
page top-k (K_p = ceil(k/ps), what the attention consumes) and the token
top-k, then the block union and the query-block sparse MLA; shared layers
(IndexShare, ref.py build_index_share_map) reuse the top-k and union tables of
their source slot and run the attention only.

All buffers are allocated once up front, so a step only enqueues kernels and
can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import abi


class LayerRunner:
    def __init__(self, wl, device, page_budget=None, prefill=None):
        """``wl``: a dsa_inputs.Workload whose tensors already live on ``device``
        (or on the CPU; they are moved). ``page_budget``: decode page-budget
        mode with that many pages. ``prefill``: force the prefill path
        (default: any request with more than one new token)."""
        rg = wl.rg
        self.wl = wl
        self.dev = torch.device(device)
        dev = self.dev
        self.rg = rg
        self.T, self.S, self.P, self.PTW, self.ps = rg.T, rg.S, rg.num_pages, rg.PTW, rg.page_size
        self.max_kv = max(1, rg.max_kv)
        self.k = wl.k
        self.k_pages = wl.k_pages if page_budget is None else page_budget
        self.page_budget = page_budget
        self.prefill = bool((rg.q_lens > 1).any()) if prefill is None else prefill
        to = lambda a: torch.from_numpy(a).to(dev)
        self.meta = [to(rg.seq_lens), to(rg.cu_q_lens), to(rg.cu_kv_lens), to(rg.page_indices)]
        self.q_idx = wl.q_idx.to(dev)
        self.w = wl.w.to(dev)
        self.kcache = [c.to(dev) for c in wl.kcache]
        self.q = [x.to(dev) for x in wl.q]
        self.kv = [x.to(dev) for x in wl.kv]
        self.types = list(wl.indexer_types) if wl.indexer_types else [0]
        self.full_slot, self.src_slot, self.num_full = abi.dsa_index_build_share_map(self.types, len(self.types))
        # the new tokens' rows (latent rows per layer, indexer keys per full
        # slot): taken from the synthetic caches, which already hold them, so
        # writing them back leaves every cache as generated
        tseq, tpos = rg.token_seq(), rg.token_pos()
        ent = rg.cu_kv_lens[tseq] // rg.page_size + tpos // rg.page_size
        rows = torch.from_numpy(rg.page_indices[ent].astype("int64") * rg.page_size + tpos % rg.page_size).to(dev)
        self.new_kv = [c.view(-1, c.shape[-1]).index_select(0, rows)[:, :576].contiguous() for c in self.kv]
        self.new_k = [c.view(-1, c.shape[-1]).index_select(0, rows).contiguous() for c in self.kcache]
        T, H = self.T, wl.H
        self.H = H
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws_idx = torch.empty(max(1, abi.dsa_indexer_workspace_size(T, self.S, self.max_kv, self.ps)),
                                  dtype=torch.uint8, device=dev)
        self.ws_att = torch.empty(max(1, abi.dsa_sparse_mla_decode_workspace_size(T, H)), dtype=torch.uint8,
                                  device=dev)
        nl = len(self.types)
        self.topk = [torch.empty((T, self.k), dtype=torch.int32, device=dev) for _ in range(self.num_full)]
        self.topk_pages = [torch.empty((T, self.k_pages), dtype=torch.int32, device=dev)
                           for _ in range(self.num_full)]
        self.o = [torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
        if self.prefill:
            self.QB = wl.QB
            self.u_max = wl.u_max if wl.u_max > 0 else min(self.QB * self.k_pages, self.PTW)
            nqb = (T + self.QB - 1) // self.QB
            self.units = [torch.empty((nqb, self.u_max), dtype=torch.int32, device=dev) for _ in range(self.num_full)]
            self.member = [torch.empty((nqb, self.u_max, self.QB // 32), dtype=torch.int32, device=dev)
                           for _ in range(self.num_full)]
            self.counts = [torch.empty((nqb,), dtype=torch.int32, device=dev) for _ in range(self.num_full)]

    # -- stages ---------------------------------------------------------------
    def write_back(self, layer):
        """The layer's new latent rows, and on a full layer its new indexer
        keys, into their slots of the paged caches."""
        if self.full_slot[layer] >= 0:  # both caches share the page table: one launch
            slot = self.full_slot[layer]
            abi.dsa_paged_write_back_pair(self.new_kv[layer], self.kv[layer], self.new_k[slot], self.kcache[slot],
                                          *self.meta, D0=576, D1=128, dev_status=self.status)
        else:
            abi.dsa_paged_write_back(self.new_kv[layer], self.kv[layer], *self.meta, D=576, dev_status=self.status)

    def index(self, slot):
        if self.prefill or self.page_budget is not None:
            abi.dsa_indexer_page_topk(self.q_idx, self.w, self.kcache[slot], *self.meta, k_pages=self.k_pages,
                                      max_kv=self.max_kv, topk_pages=self.topk_pages[slot], k=self.k,
                                      topk=self.topk[slot] if self.prefill else None, ws=self.ws_idx,
                                      dev_status=self.status)
        else:
            abi.dsa_indexer_topk(self.q_idx, self.w, self.kcache[slot], *self.meta, k=self.k, max_kv=self.max_kv,
                                 topk=self.topk[slot], ws=self.ws_idx, dev_status=self.status)

    def union(self, slot):
        abi.dsa_build_block_union(self.topk_pages[slot], QB=self.QB, u_max=self.u_max, cu_q_lens=self.meta[1],
                                  cu_kv_lens=self.meta[2], ps=self.ps, PTW=self.PTW, units=self.units[slot],
                                  member=self.member[slot], counts=self.counts[slot], dev_status=self.status)

    def attend(self, layer, t_range=None):
        """The layer's attention; ``t_range=(b, e)`` (prefill batches) writes
        only the output rows of tokens b .. e-1."""
        slot = self.src_slot[layer]
        if self.prefill:
            abi.dsa_sparse_mla_prefill_qblock(self.q[layer], self.kv[layer], *self.meta, self.units[slot],
                                              self.member[slot], self.counts[slot], QB=self.QB,
                                              sm_scale=self.wl.sm_scale, o=self.o[layer], dev_status=self.status,
                                              t_range=t_range)
        elif self.page_budget is not None:
            abi.dsa_sparse_mla_decode(self.q[layer], self.kv[layer], *self.meta, self.topk_pages[slot],
                                      unit=self.ps, sm_scale=self.wl.sm_scale, o=self.o[layer], ws=self.ws_att,
                                      dev_status=self.status)
        else:
            abi.dsa_sparse_mla_decode(self.q[layer], self.kv[layer], *self.meta, self.topk[slot], unit=1,
                                      sm_scale=self.wl.sm_scale, o=self.o[layer], ws=self.ws_att,
                                      dev_status=self.status)

    def layer_step(self, layer):
        self.write_back(layer)
        if self.full_slot[layer] >= 0:
            slot = self.full_slot[layer]
            self.index(slot)
            if self.prefill:
                self.union(slot)
        self.attend(layer)

    def step(self):
        """Every layer of the workload once (IndexShare across layers)."""
        for layer in range(len(self.types)):
            self.layer_step(layer)

    def step_host(self, h_q_idx, h_w, h_q, h_meta, h_topk, h_o, side, h_new_kv=None, h_new_k=None, out_side=None,
                  last_chunks=4):
        """One step from and to pinned host buffers (same shapes as the device
        tensors). The indexer inputs, the metadata and the new tokens' rows
        are copied first, on the current stream: host-to-device copies of all
        streams share one copy queue, so anything issued after the queries
        would wait for them. Each layer's attention queries (the largest
        inputs, needed only by that layer's attention) follow on the stream
        ``side``, in layer order, while the earlier layers compute; each
        layer's output is read back on the stream ``out_side`` (one of the
        runner's own if None) as soon as that layer's attention has written it,
        and the token selections of the first full slot once they exist. On a
        prefill batch the first layer's queries arrive, and its attention runs,
        in ``last_chunks`` token ranges (the attention of the first range
        starts when its queries have landed, not all of them), and the last
        layer's attention runs in as many ranges, each read back as soon as it
        is written, so little of the final read-back is left after the last
        kernel. The current stream joins both side streams before it returns,
        so the step ends when every copy has landed. Can be captured in a CUDA
        graph."""
        cur = torch.cuda.current_stream(self.dev)
        if out_side is None:
            if getattr(self, "_out_side", None) is None:
                self._out_side = torch.cuda.Stream(self.dev)
            out_side = self._out_side
        nl = len(self.types)

        def ranges(layer):
            # token ranges on query-block boundaries (first and last layer of a
            # prefill batch), else the whole batch
            nch = max(1, min(last_chunks, self.T // self.QB)) if (self.prefill and layer in (0, nl - 1)) else 1
            if nch == 1:
                return [(0, self.T)]
            nqb = -(-self.T // self.QB)
            b = [min(self.T, (nqb * c // nch) * self.QB) for c in range(nch)] + [self.T]
            return list(zip(b[:-1], b[1:]))

        self.q_idx.copy_(h_q_idx, non_blocking=True)
        self.w.copy_(h_w, non_blocking=True)
        for d, h in zip(self.meta, h_meta):
            d.copy_(h, non_blocking=True)
        for d, h in zip(self.new_kv, h_new_kv or []):
            d.copy_(h, non_blocking=True)
        for d, h in zip(self.new_k, h_new_k or []):
            d.copy_(h, non_blocking=True)
        # the previous step's kernels have finished reading q (its read-backs
        # were joined into the current stream when it returned)
        side.wait_stream(cur)
        q_ready = []  # per layer: one event per token range of its attention
        with torch.cuda.stream(side):
            for layer, (d, h) in enumerate(zip(self.q, h_q)):
                evs = []
                for b, e in ranges(layer) if layer == 0 else [(0, self.T)]:
                    d[b:e].copy_(h[b:e], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(side)
                    evs.append(ev)
                q_ready.append(evs)
        topk_read = False
        for layer in range(nl):
            self.write_back(layer)
            if self.full_slot[layer] >= 0:
                slot = self.full_slot[layer]
                self.index(slot)
                if self.prefill:
                    self.union(slot)
                if not topk_read:
                    out_side.wait_stream(cur)
                    with torch.cuda.stream(out_side):
                        h_topk.copy_(self.topk[0], non_blocking=True)
                    topk_read = True
            rs = ranges(layer)
            for i, (b, e) in enumerate(rs):
                evs = q_ready[layer]
                cur.wait_event(evs[min(i, len(evs) - 1)])
                self.attend(layer, (b, e) if len(rs) > 1 else None)
                out_side.wait_stream(cur)
                with torch.cuda.stream(out_side):
                    h_o[layer][b:e].copy_(self.o[layer][b:e], non_blocking=True)
        cur.wait_stream(side)
        cur.wait_stream(out_side)
