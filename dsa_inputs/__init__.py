"""Seeded synthetic inputs for the DSA sparse-attention hot path.

This module only draws random numbers and lays out ragged metadata. It holds
none of the method's arithmetic (no scores, no selection, no softmax), so the
CPU oracle under ``oracle/`` and the CUDA library can both consume its output
without sharing any code of the method.

Every tensor comes from its own ``torch.Generator`` seeded with
``master_seed ^ crc32(name)``; the master seed of workload ``c`` is
``0xD5A0 + c``. Small workloads are drawn on the CPU (so the oracle sees the
exact host copy); large ones can be drawn straight on a CUDA device.

Layouts (all row-major):
  * indexer query ``q_idx`` bf16 ``[T, Hi, Di]``, weights ``w`` fp32 ``[T, Hi]``
  * indexer key cache ``kcache`` bf16 ``[P, ps, Di]``
  * MLA query ``q`` bf16 ``[T, H, 576]`` (``[q_nope(512) | q_rope(64)]``)
  * MLA latent cache ``kv`` bf16 ``[P, ps, 576]`` (``[c_kv(512) | k_rope(64)]``)
  * ragged metadata int32: ``seq_lens [S]`` (kv length including the new
    tokens), ``cu_q_lens [S+1]``, ``cu_kv_lens [S+1]`` (cumsum of page-aligned
    kv lengths), ``page_indices [PTW]`` (packed: sequence ``s`` owns entries
    ``cu_kv_lens[s]//ps ...``).
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

MASTER_SEED_BASE = 0xD5A0

# Model constants of the workloads (GLM-5-style DSA layer).
INDEX_HEADS = 32
INDEX_DIM = 128
KV_LORA_RANK = 512
ROPE_DIM = 64
DK = KV_LORA_RANK + ROPE_DIM  # 576-wide latent key
DV = KV_LORA_RANK  # 512-wide latent value
PAGE_SIZE = 64
SM_SCALE = 1.0 / math.sqrt(192.0)


def _gen(master_seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(master_seed) ^ zlib.crc32(name.encode())) & 0x7FFFFFFFFFFFFFFF)
    return g


def randn(shape, master_seed, name, device="cpu", dtype=torch.float32):
    g = _gen(master_seed, name, device)
    return torch.randn(shape, generator=g, device=device, dtype=dtype)


def rand(shape, master_seed, name, device="cpu"):
    g = _gen(master_seed, name, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def randint(low, high, shape, master_seed, name):
    """Integers uniform in [low, high] (inclusive), drawn on the CPU."""
    g = _gen(master_seed, name, "cpu")
    return torch.randint(low, high + 1, shape, generator=g, dtype=torch.int64)


def randperm(n, master_seed, name):
    g = _gen(master_seed, name, "cpu")
    return torch.randperm(n, generator=g, dtype=torch.int64)


def randn_bf16_chunked(shape, master_seed, name, device="cpu", chunk_rows=1 << 14):
    """N(0,1) rounded to bf16 (round-to-nearest-even), drawn in row chunks so
    multi-GB caches never need an fp32 copy of the whole tensor."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    g = _gen(master_seed, name, device)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device).to(torch.bfloat16)
    return out


@dataclass
class Ragged:
    """Packed ragged batch metadata (host numpy int32 arrays)."""

    seq_lens: np.ndarray
    cu_q_lens: np.ndarray
    cu_kv_lens: np.ndarray
    page_indices: np.ndarray
    page_size: int
    num_pages: int  # physical pages P in the pool

    @property
    def S(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu_q_lens[-1])

    @property
    def PTW(self) -> int:
        return int(self.page_indices.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_q_lens)

    @property
    def max_kv(self) -> int:
        return int(self.seq_lens.max()) if self.S else 0

    def token_seq(self) -> np.ndarray:
        """Request id of every query token (layout helper for input shaping)."""
        return np.repeat(np.arange(self.S, dtype=np.int64), self.q_lens)

    def token_pos(self) -> np.ndarray:
        """Absolute position of every query token: the new tokens are the
        last ``q_len`` positions of their request."""
        seq = self.token_seq()
        t = np.arange(self.T, dtype=np.int64)
        return (self.seq_lens[seq] - self.q_lens[seq] + (t - self.cu_q_lens[seq])).astype(np.int64)


def make_ragged(q_lens, kv_lens, page_size, num_pages=None, master_seed=0, name="pages",
                spare_pages=0) -> Ragged:
    """Build packed metadata: request ``s`` gets ``ceil(kv_len/ps)`` page-table
    entries taken consecutively from one seeded permutation of the pool."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    assert q_lens.shape == kv_lens.shape
    assert np.all(q_lens <= kv_lens)
    npages = (kv_lens + page_size - 1) // page_size
    cu_kv = np.zeros(len(kv_lens) + 1, dtype=np.int64)
    cu_kv[1:] = np.cumsum(npages * page_size)
    ptw = int(npages.sum())
    if num_pages is None:
        num_pages = ptw + spare_pages
    assert num_pages >= ptw
    perm = randperm(num_pages, master_seed, name).numpy()
    cu_q = np.zeros(len(q_lens) + 1, dtype=np.int64)
    cu_q[1:] = np.cumsum(q_lens)
    return Ragged(
        seq_lens=kv_lens.astype(np.int32),
        cu_q_lens=cu_q.astype(np.int32),
        cu_kv_lens=cu_kv.astype(np.int32),
        page_indices=perm[:ptw].astype(np.int32),
        page_size=int(page_size),
        num_pages=int(num_pages),
    )


@dataclass
class Workload:
    name: str
    rg: Ragged
    q_idx: torch.Tensor  # bf16 [T, Hi, Di]
    w: torch.Tensor  # fp32 [T, Hi]
    kcache: list  # bf16 [P, ps, Di] per indexer slot
    q: list  # bf16 [T, H, 576] per layer
    kv: list  # bf16 [P, ps, 576] per layer
    k: int  # token top-k
    k_pages: int  # page top-k budget
    QB: int = 256
    u_max: int = 0
    sm_scale: float = SM_SCALE
    indexer_types: list = field(default_factory=lambda: [0])
    # which requests use which bias recipe (informational)
    notes: str = ""

    @property
    def H(self) -> int:
        return int(self.q[0].shape[1])


def _logical_rows(rg: Ragged, s: int, positions: np.ndarray) -> np.ndarray:
    """Flat physical row (page*ps + offset) of sequence-local positions."""
    ps = rg.page_size
    base = int(rg.cu_kv_lens[s]) // ps
    pages = rg.page_indices[base + positions // ps].astype(np.int64)
    return pages * ps + positions % ps


def _bias_decode(rg: Ragged, qt: torch.Tensor, cache: torch.Tensor, seqs, coeff=0.5, sinks=128,
                 window=512, seed=0, name="bias"):
    """Sink/local-window bias of the decode workloads: keys at positions
    ``j < sinks`` and ``j >= kv_len - window`` become ``N(0,1) + coeff*m``
    where ``m`` is the head-mean of the request's (single) query token."""
    flat = cache.view(-1, cache.shape[-1])
    dev = cache.device
    for s in seqs:
        kv_len = int(rg.seq_lens[s])
        t_last = int(rg.cu_q_lens[s + 1]) - 1
        m = qt[t_last].float().mean(dim=0)  # [D]
        pos = np.unique(np.concatenate([np.arange(min(sinks, kv_len)),
                                        np.arange(max(0, kv_len - window), kv_len)]))
        rows = torch.from_numpy(_logical_rows(rg, s, pos)).to(dev)
        noise = randn((len(pos), cache.shape[-1]), seed, f"{name}/{s}", device=dev)
        flat[rows] = (noise + coeff * m[None, :]).to(torch.bfloat16)


def _ar1(n, dim, seed, name, rho):
    """Unit-variance AR(1) process a[p] = rho a[p-1] + sqrt(1-rho^2) xi_p, a[0]=xi_0."""
    from scipy.signal import lfilter

    xi = randn((n, dim), seed, name).numpy().astype(np.float64)
    a = np.empty_like(xi)
    a[0] = xi[0]
    if n > 1:
        a[1:], _ = lfilter([math.sqrt(1.0 - rho * rho)], [1.0, -rho], xi[1:], axis=0,
                           zi=(rho * a[0])[None, :])
    return torch.from_numpy(a.astype(np.float32))


def _bias_prefill(rg: Ragged, s: int, qt: torch.Tensor, cache: torch.Tensor, seed, name,
                  rho=1.0 - 1.0 / 256.0, sinks=128, coeff=0.5):
    """Sink + local-window structure of the prefill workloads, relative to each
    query's own position: per request a sink direction ``g`` and an AR(1)
    process ``a`` over absolute positions;
    ``q[t] = (eps + a[pos(t)] + g)/sqrt(3)`` (unit marginal variance) and
    ``k[j] = N(0,1) + coeff*(a[j] + [j<sinks] g)/sqrt(3)``."""
    dev = cache.device
    kv_len = int(rg.seq_lens[s])
    D = cache.shape[-1]
    a = _ar1(kv_len, D, seed, f"{name}/ar/{s}", rho).to(dev)
    g = randn((D,), seed, f"{name}/sink/{s}").to(dev)
    t0, t1 = int(rg.cu_q_lens[s]), int(rg.cu_q_lens[s + 1])
    pos = torch.from_numpy(rg.token_pos()[t0:t1]).to(dev)
    eps = randn((t1 - t0,) + tuple(qt.shape[1:]), seed, f"{name}/eps/{s}", device=dev)
    qt[t0:t1] = ((eps + a[pos][:, None, :] + g[None, None, :]) / math.sqrt(3.0)).to(torch.bfloat16)
    j = torch.arange(kv_len, device=dev)
    rows = torch.from_numpy(_logical_rows(rg, s, np.arange(kv_len))).to(dev)
    noise = randn((kv_len, D), seed, f"{name}/knoise/{s}", device=dev)
    extra = a + (j < sinks).float()[:, None] * g[None, :]
    cache.view(-1, D)[rows] = (noise + coeff * extra / math.sqrt(3.0)).to(torch.bfloat16)


def _base_tensors(rg: Ragged, seed, H, device, n_idx_caches=1, n_layers=1):
    T, P, ps = rg.T, rg.num_pages, rg.page_size
    q_idx = randn((T, INDEX_HEADS, INDEX_DIM), seed, "q_idx", device=device).to(torch.bfloat16)
    w = rand((T, INDEX_HEADS), seed, "w", device=device) / math.sqrt(INDEX_HEADS)
    kc = [randn_bf16_chunked((P, ps, INDEX_DIM), seed, f"kcache/{i}", device=device)
          for i in range(n_idx_caches)]
    q = [randn((T, H, DK), seed, f"q/{l}", device=device).to(torch.bfloat16) for l in range(n_layers)]
    kv = [randn_bf16_chunked((P, ps, DK), seed, f"kv/{l}", device=device) for l in range(n_layers)]
    return q_idx, w, kc, q, kv


def tiny_decode(device="cpu") -> Workload:
    """1 request, kv_len 1024, 16 pages (a permutation), k=256, 16 MLA heads."""
    seed = MASTER_SEED_BASE + 1
    rg = make_ragged([1], [1024], PAGE_SIZE, num_pages=16, master_seed=seed)
    q_idx, w, kc, q, kv = _base_tensors(rg, seed, 16, device)
    return Workload("tiny_decode", rg, q_idx, w, kc, q, kv, k=256, k_pages=4)


def batched_decode(device="cpu", B=32) -> Workload:
    """32 requests, kv_len ~ U{4096..8192}, pool of 8192 pages, biased sinks
    (first 128) and local window (last 512), k=2048, 128 MLA heads."""
    seed = MASTER_SEED_BASE + 2
    kv_lens = randint(4096, 8192, (B,), seed, "kv_lens").numpy()
    rg = make_ragged(np.ones(B, np.int64), kv_lens, PAGE_SIZE, num_pages=8192, master_seed=seed)
    q_idx, w, kc, q, kv = _base_tensors(rg, seed, 128, device)
    _bias_decode(rg, q_idx, kc[0], range(B), seed=seed, name="kbias")
    _bias_decode(rg, q[0], kv[0], range(B), seed=seed, name="kvbias")
    return Workload("batched_decode", rg, q_idx, w, kc, q, kv, k=2048, k_pages=32)


def long_decode(device="cpu", B=64, kv_len=131072) -> Workload:
    """64 requests of 131072 tokens over a pool of 131072 pages (one full
    permutation), decode bias as in the batched workload; token k=2048 and a
    32-page budget."""
    seed = MASTER_SEED_BASE + 3
    npages = B * kv_len // PAGE_SIZE
    rg = make_ragged(np.ones(B, np.int64), np.full(B, kv_len), PAGE_SIZE, num_pages=npages,
                     master_seed=seed)
    q_idx, w, kc, q, kv = _base_tensors(rg, seed, 128, device)
    _bias_decode(rg, q_idx, kc[0], range(B), seed=seed, name="kbias")
    _bias_decode(rg, q[0], kv[0], range(B), seed=seed, name="kvbias")
    return Workload("long_decode", rg, q_idx, w, kc, q, kv, k=2048, k_pages=32)


def single_prefill(device="cpu", T=8192) -> Workload:
    """One request, prefix 0, T=8192 new tokens, 128 pages; AR(1) local window
    plus sink bias for both the indexer and the MLA inputs; k=2048, 32 pages
    per query, QB=256, u_max=min(QB*32, 128)=128."""
    seed = MASTER_SEED_BASE + 4
    rg = make_ragged([T], [T], PAGE_SIZE, num_pages=T // PAGE_SIZE, master_seed=seed)
    q_idx, w, kc, q, kv = _base_tensors(rg, seed, 128, device)
    _bias_prefill(rg, 0, q_idx, kc[0], seed, "idx")
    _bias_prefill(rg, 0, q[0], kv[0], seed, "mla")
    k_pages = (2048 + PAGE_SIZE - 1) // PAGE_SIZE
    return Workload("single_prefill", rg, q_idx, w, kc, q, kv, k=2048, k_pages=k_pages, QB=256,
                    u_max=min(256 * k_pages, rg.PTW))


def ragged_mixed(device="cpu", n_decode=48, prefixes=(0, 16384, 65536, 110592), new=4096) -> Workload:
    """48 decode tokens (kv_len ~ U{8192..131072}) first, then 4 chunked-prefill
    extends adding 4096 tokens to prefixes 0/16384/65536/110592; packed page
    table over PTW+1 shuffled pages; four layers [full, shared, shared, full]
    with two indexer caches and four MLA caches."""
    seed = MASTER_SEED_BASE + 5
    dec_kv = randint(8192, 131072, (n_decode,), seed, "kv_lens").numpy()
    q_lens = np.concatenate([np.ones(n_decode, np.int64), np.full(len(prefixes), new)])
    kv_lens = np.concatenate([dec_kv, np.asarray(prefixes, np.int64) + new])
    rg = make_ragged(q_lens, kv_lens, PAGE_SIZE, master_seed=seed, spare_pages=1)
    q_idx, w, kc, q, kv = _base_tensors(rg, seed, 128, device, n_idx_caches=2, n_layers=4)
    dec = range(n_decode)
    for i in range(2):
        _bias_decode(rg, q_idx, kc[i], dec, seed=seed, name=f"kbias{i}")
        for s in range(n_decode, rg.S):
            _bias_prefill(rg, s, q_idx, kc[i], seed, f"idx{i}")
    for l in range(4):
        _bias_decode(rg, q[l], kv[l], dec, seed=seed, name=f"kvbias{l}")
        for s in range(n_decode, rg.S):
            _bias_prefill(rg, s, q[l], kv[l], seed, f"mla{l}")
    k_pages = (2048 + PAGE_SIZE - 1) // PAGE_SIZE
    return Workload("ragged_mixed", rg, q_idx, w, kc, q, kv, k=2048, k_pages=k_pages, QB=256,
                    u_max=min(256 * k_pages, rg.PTW), indexer_types=[0, 1, 1, 0])


def random_small(seed, q_lens, kv_lens, H=16, page_size=PAGE_SIZE, spare_pages=3, k=64,
                 k_pages=4, device="cpu", index_heads=INDEX_HEADS, index_dim=INDEX_DIM) -> Workload:
    """Small unstructured ragged batch for parity tests (N(0,1) everywhere)."""
    rg = make_ragged(q_lens, kv_lens, page_size, master_seed=seed, spare_pages=spare_pages)
    T, P, ps = rg.T, rg.num_pages, rg.page_size
    q_idx = randn((T, index_heads, index_dim), seed, "q_idx", device=device).to(torch.bfloat16)
    w = rand((T, index_heads), seed, "w", device=device) / math.sqrt(index_heads)
    kc = [randn((P, ps, index_dim), seed, "kcache", device=device).to(torch.bfloat16)]
    q = [randn((T, H, DK), seed, "q", device=device).to(torch.bfloat16)]
    kv = [randn((P, ps, DK), seed, "kv", device=device).to(torch.bfloat16)]
    return Workload(f"random_small_{seed}", rg, q_idx, w, kc, q, kv, k=k, k_pages=k_pages)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "batched_decode": batched_decode,
    "long_decode": long_decode,
    "single_prefill": single_prefill,
    "ragged_mixed": ragged_mixed,
}
