// Lightning-indexer score on tcgen05 (ref.py, streamindex_topk_ref /
// streamindex_page_topk_ref: s[t,j] = sum_h relu(q[t,h,:] . k[j,:]) * w[t,h]).
//
// Key-major contraction: one UMMA tile is D[128 keys x NQ*32 (query,head)] =
// K_tile[128 x 128] * Q_tile[NQ*32 x 128]^T, so every TMEM lane holds one key
// and the ReLU + weighted head sum runs in-thread over its 32 head columns.
// NQ = 1 serves decode-like tiles (HBM-bound streaming of paged keys), NQ = 8
// serves prefill tiles (tensor-bound). Keys arrive page by page through 2-D
// TMA with 128-byte swizzle into a multi-stage ring; the epilogue writes the
// fp32 token scores and/or the maximum of every 32-key granule (the page top-k
// folds a page's granules into its max-pooled score).
//
// A device-side planner turns the ragged metadata into work items
// (query tile, key chunk) so the persistent kernels never read metadata the
// host cannot see.
#include "common.cuh"
#include "indexer.cuh"

namespace dsa {

// ------------------------------------------------------------------ planner
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    int y = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_warp[lane] = y;
  }
  __syncthreads();
  const int excl = x - v + (w > 0 ? s_warp[w - 1] : 0);
  *total = s_warp[nw - 1];
  __syncthreads();
  return excl;
}

constexpr int kPlanStageS = 4096;  // requests whose query offsets the planner keeps in shared memory

// one_token: every token becomes a one-token tile (the launch has as many
// tokens as requests, so it is a decode batch but for requests without new
// tokens; the eight-query kernel is then not launched at all)
__global__ void __launch_bounds__(1024) indexer_plan_kernel(IndexerMeta m, IndexerPlan pl, int ch1, int ch8,
                                                            int one_token) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int s_warp[32];
  __shared__ int s_cuq[kPlanStageS + 1];
  __shared__ int s_off[1024];
  __shared__ int4 s_tile[1024];
  const int T = m.T, S = m.S, ps = m.ps;
  // token -> request searches run against a shared-memory copy of cu_q_lens
  // when it fits (a chain of dependent global loads otherwise)
  const bool staged = S <= kPlanStageS;
  if (staged)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) s_cuq[i] = __ldg(m.cu_q_lens + i);
  __syncthreads();
  auto seq_of = [&](int t) -> int {
    if (!staged) return seq_of_token(m.cu_q_lens, S, t);
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cuq[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // 1. visible prefix of every token, clamped to the request's page-table span
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    TokenGeom g = token_geom(m.seq_lens, m.cu_q_lens, m.cu_kv_lens, S, ps, m.max_kv, t, m.dev_status, seq_of(t));
    long long cap = (long long)(m.PTW - g.page_base) * ps;
    int nv = g.n_vis;
    if (g.page_base < 0 || (long long)nv > cap) {
      set_status(m.dev_status, DSA_STATUS_BAD_METADATA);
      nv = cap < 0 || g.page_base < 0 ? 0 : (int)cap;
    }
    pl.nvis[t] = nv;
  }
  if (threadIdx.x == 0 && (__ldg(m.cu_q_lens) != 0 || __ldg(m.cu_q_lens + S) != T))
    set_status(m.dev_status, DSA_STATUS_BAD_METADATA);
  __syncthreads();
  // 2. per-request tile counts: tiles of up to 8 consecutive tokens; a final
  //    one-token tile goes to the decode (NQ = 1) list.
  int carry_d = 0, carry_p = 0;
  for (int s0 = 0; s0 < S; s0 += blockDim.x) {
    const int s = s0 + threadIdx.x;
    int nd = 0, np = 0;
    if (s < S) {
      const int ql = staged ? s_cuq[s + 1] - s_cuq[s] : __ldg(m.cu_q_lens + s + 1) - __ldg(m.cu_q_lens + s);
      if (ql > 0 && one_token) {
        nd = ql;
      } else if (ql > 0) {
        const int nt = (ql + 7) / 8;
        nd = (ql - 8 * (nt - 1)) == 1 ? 1 : 0;
        np = nt - nd;
      }
    }
    int td, tp;
    const int ed = block_excl_scan(nd, s_warp, &td);
    const int ep = block_excl_scan(np, s_warp, &tp);
    if (s < S) pl.seq_tile_off[s] = make_int2(carry_d + ed, carry_p + ep);
    carry_d += td;
    carry_p += tp;
  }
  __syncthreads();
  const int n_dec_tiles = carry_d, n_pre_tiles = carry_p;
  // 3. tile descriptors {first token, ntok, request, visible keys of the last token}
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const int s = seq_of(t);
    const int q0 = staged ? s_cuq[s] : __ldg(m.cu_q_lens + s);
    const int ql = (staged ? s_cuq[s + 1] : __ldg(m.cu_q_lens + s + 1)) - q0;
    const int r = t - q0;
    const int2 off = pl.seq_tile_off[s];
    if (one_token) {
      pl.dec_tiles[off.x + r] = make_int4(t, 1, s, pl.nvis[t]);
      continue;
    }
    if (r % 8) continue;
    const int ntok = min(8, ql - r);
    const int nvmax = pl.nvis[t + ntok - 1];
    if (ntok == 1) pl.dec_tiles[off.x] = make_int4(t, ntok, s, nvmax);
    else pl.pre_tiles[off.y + r / 8] = make_int4(t, ntok, s, nvmax);
  }
  __syncthreads();
  // 4. expand tiles into (tile, key chunk) items
  for (int list = 0; list < 2; ++list) {
    const int ntiles = list == 0 ? n_dec_tiles : n_pre_tiles;
    const int4* tiles = list == 0 ? pl.dec_tiles : pl.pre_tiles;
    int4* items = list == 0 ? pl.dec_items : pl.pre_items;
    const int ch = list == 0 ? ch1 : ch8;
    int carry = 0;
    for (int i0 = 0; i0 < ntiles; i0 += blockDim.x) {
      const int i = i0 + threadIdx.x;
      int4 tl = make_int4(0, 0, 0, 0);
      int n = 0;
      if (i < ntiles) {
        tl = tiles[i];
        n = (tl.w + ch - 1) / ch;
      }
      int tot;
      const int e = block_excl_scan(n, s_warp, &tot);
      // every thread writes items (coalesced), finding its tile by a search
      // over this batch's item offsets
      s_off[threadIdx.x] = i < ntiles ? e : 0x7fffffff;
      s_tile[threadIdx.x] = tl;
      __syncthreads();
      const int nb = min((int)blockDim.x, ntiles - i0);
      for (int j = threadIdx.x; j < tot; j += blockDim.x) {
        int lo = 0, hi = nb - 1;  // last tile whose offset is <= j
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_off[mid] <= j) lo = mid; else hi = mid - 1;
        }
        const int4 tj = s_tile[lo];
        const int kb = (j - s_off[lo]) * ch, ke = min(tj.w, kb + ch);
        items[carry + j] = make_int4(tj.x, (tj.y << 24) | tj.z, kb, ke);
      }
      __syncthreads();
      carry += tot;
    }
    if (threadIdx.x == 0) pl.counts[list] = carry;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ scorer
// Item ii of a launch without a planner (every request has one new token, so
// token t is request t unless some requests have none): token, request, key
// range and the token's visible length, clamped to its page-table span as
// the planner clamps it. Returns false for an empty key range.
__device__ __forceinline__ bool direct_item(const IndexerMeta& m, int ii, int& t, int& seq, int& kb, int& ke,
                                            int& nv) {
  t = ii / m.direct_nch;
  const int c = ii - t * m.direct_nch;
  const int a = __ldg(m.cu_q_lens + t), b = __ldg(m.cu_q_lens + t + 1);
  seq = (a == t && b == t + 1) ? t : seq_of_token(m.cu_q_lens, m.S, t);
  const TokenGeom g = token_geom(m.seq_lens, m.cu_q_lens, m.cu_kv_lens, m.S, m.ps, m.max_kv, t, m.dev_status, seq);
  const long long cap = (long long)(m.PTW - g.page_base) * m.ps;
  nv = g.n_vis;
  if (g.page_base < 0 || (long long)nv > cap) {
    set_status(m.dev_status, DSA_STATUS_BAD_METADATA);
    nv = cap < 0 || g.page_base < 0 ? 0 : (int)cap;
  }
  kb = c * m.direct_ch;
  ke = min(nv, kb + m.direct_ch);
  return kb < ke;
}

template <int NQ>
struct IdxCfg {
  static constexpr int N = NQ * 32;                  // UMMA N: (query, head) columns
  static constexpr int EPI_WARPS = NQ == 1 ? 4 : 16;  // epilogue warps: 1 or 4 per TMEM lane quadrant
  static constexpr int QPW = NQ / (EPI_WARPS / 4);    // queries each epilogue warp scores per tile
  static constexpr int THREADS = 64 + EPI_WARPS * 32;
  static constexpr int STAGES = NQ == 1 ? 6 : 3;
  static constexpr int Q_BYTES = N * 256;            // N rows x 128 dims bf16
  static constexpr int STAGE_BYTES = 128 * 256;      // 128 keys x 128 dims bf16
  static constexpr int TMEM_COLS = NQ == 1 ? 64 : 512;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_STAGE = 2 * Q_BYTES;
  static constexpr int OFF_W = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_W + 2 * N * 4;
  static constexpr int NBAR = 2 * STAGES + 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC = make_idesc_bf16(128, N, false, false);
};

// Order-preserving map fp32 -> uint32 (larger float -> larger key; 0 is
// below every mapped value), and its inverse.
__device__ __forceinline__ uint32_t ordered_key_f32(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ordered_key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NQ>
__global__ void __launch_bounds__(IdxCfg<NQ>::THREADS, 1)
    indexer_score_kernel(IndexerMeta m, IndexerPlan pl, IndexerOut out, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap qmap) {
  using C = IdxCfg<NQ>;
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_launch_dependents();
  griddep_wait();
  const bool direct = NQ == 1 && m.direct_nch > 0;
  const int n_items = direct ? m.T * m.direct_nch : NQ == 1 ? pl.counts[0] : pl.counts[1];
  if ((int)blockIdx.x >= n_items) return;
  const int4* items = NQ == 1 ? pl.dec_items : pl.pre_items;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need 1 KB alignment
    if (threadIdx.x == 0) set_status(m.dev_status, DSA_STATUS_INTERNAL);
    return;
  }
  uint8_t* q_s = smem + C::OFF_Q;
  uint8_t* st_s = smem + C::OFF_STAGE;
  float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* qfull = bars + 2 * C::STAGES;
  uint64_t* qempty = qfull + 2;
  uint64_t* dfull = qfull + 4;
  uint64_t* dempty = qfull + 6;
  uint64_t* fin = qfull + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = warp_id(), lane = lane_id();
  constexpr int EPI_THREADS = C::EPI_WARPS * 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(qfull + i, 1);
      mbar_init(qempty + i, 1 + EPI_THREADS);
      mbar_init(dfull + i, 1);
      mbar_init(dempty + i, EPI_THREADS);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // The whole warp walks the items so that an item's page ids are resolved
    // with one batch of loads (up to 64 pages, two per lane); lane 0 issues
    // the TMA copies.
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&qmap);
    }
    int kt = 0, it = 0;
    bool ok = true;
    if (direct && blockIdx.x == 0 && lane == 0 &&
        (__ldg(m.cu_q_lens) != 0 || __ldg(m.cu_q_lens + m.S) != m.T))
      set_status(m.dev_status, DSA_STATUS_BAD_METADATA);
    for (int ii = blockIdx.x; ii < n_items && ok; ii += gridDim.x, ++it) {
      int t0, ntok, seq, kb, ke;
      if (direct) {
        int nvv;
        const bool live = direct_item(m, ii, t0, seq, kb, ke, nvv);
        if (lane == 0 && kb == 0) pl.nvis[t0] = nvv;  // the token's first item
        if (!live) {  // every role skips the same items
          --it;
          continue;
        }
        ntok = 1;
      } else {
        const int4 item = items[ii];
        t0 = item.x, ntok = item.y >> 24, seq = item.y & 0xFFFFFF, kb = item.z, ke = item.w;
      }
      const int qb = it & 1;
      int okl = 1;
      if (lane == 0) {
        okl = mbar_wait(qempty + qb, ((it >> 1) & 1) ^ 1, abort_flag) ? 1 : 0;
        if (okl) {
          mbar_arrive_expect_tx(qfull + qb, C::Q_BYTES + ntok * 128);
          tma_load_2d(q_s + qb * C::Q_BYTES, &qmap, qfull + qb, 0, t0 * 32);
          tma_load_2d(q_s + qb * C::Q_BYTES + C::N * 128, &qmap, qfull + qb, 64, t0 * 32);
          bulk_load(w_s + qb * C::N, m.w + (size_t)t0 * 32, ntok * 128, qfull + qb);
        }
      }
      if (!(ok = __shfl_sync(0xffffffffu, okl, 0) != 0)) break;
      const int ps = m.ps;
      const int page_base = __ldg(m.cu_kv_lens + seq) / ps;
      const int pg0 = kb / ps, npg = (ke - 1) / ps - pg0 + 1;  // <= 64 pages per item
      int pid[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pi = lane + 32 * h;
        pid[h] = -1;
        if (pi < npg) {
          const int p = __ldg(m.page_indices + page_base + pg0 + pi);
          if (p >= 0 && p < m.P) pid[h] = p;
          else set_status(m.dev_status, DSA_STATUS_BAD_METADATA);
        }
      }
      const int ppt = 128 / ps;  // pages per 128-key tile
      for (int tile = kb / 128; tile * 128 < ke; ++tile, ++kt) {
        const int s = kt % C::STAGES;
        int phys[4];
        int nload = 0;
#pragma unroll
        for (int pg = 0; pg < 4; ++pg) {
          phys[pg] = -1;
          const int key0 = tile * 128 + pg * ps;
          if (pg < ppt) {
            const int pi = key0 / ps - pg0;
            const int v0 = __shfl_sync(0xffffffffu, pid[0], pi & 31);
            const int v1 = __shfl_sync(0xffffffffu, pid[1], pi & 31);
            if (key0 < ke) {
              phys[pg] = pi < 32 ? v0 : v1;
              if (phys[pg] >= 0) ++nload;
            }
          }
        }
        if (lane == 0) {
          okl = mbar_wait(empty + s, ((kt / C::STAGES) & 1) ^ 1, abort_flag) ? 1 : 0;
          if (okl) {
            mbar_arrive_expect_tx(full + s, nload * ps * 256);
            uint8_t* dst = st_s + s * C::STAGE_BYTES;
            for (int pg = 0; pg < ppt; ++pg) {
              if (phys[pg] < 0) continue;
              tma_load_2d(dst + pg * ps * 128, &kmap, full + s, 0, phys[pg] * ps);
              tma_load_2d(dst + 16384 + pg * ps * 128, &kmap, full + s, 64, phys[pg] * ps);
            }
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, okl, 0) != 0)) break;
      }
    }
    // drain: make sure no TMA write is still landing in shared memory
    if (lane == 0) {
      for (int d = 1; d <= C::STAGES && d <= kt; ++d) {
        const int k2 = kt - d;
        mbar_wait_drain(full + k2 % C::STAGES, (k2 / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int kt = 0, dt = 0, it = 0;
      bool ok = true;
      for (int ii = blockIdx.x; ii < n_items && ok; ii += gridDim.x, ++it) {
        int kb, ke;
        if (direct) {
          int t_, s_, nv_;
          if (!direct_item(m, ii, t_, s_, kb, ke, nv_)) {
            --it;
            continue;
          }
        } else {
          const int4 item = items[ii];
          kb = item.z, ke = item.w;
        }
        const int qb = it & 1;
        if (!(ok = mbar_wait(qfull + qb, (it >> 1) & 1, abort_flag))) break;
        const uint32_t qaddr = smem_u32(q_s + qb * C::Q_BYTES);
        for (int tile = kb / 128; tile * 128 < ke; ++tile, ++kt, ++dt) {
          const int s = kt % C::STAGES, db = dt & 1;
          if (!(ok = mbar_wait(full + s, (kt / C::STAGES) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(dempty + db, ((dt >> 1) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t kaddr = smem_u32(st_s + s * C::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t a = make_sdesc(kaddr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
            const uint64_t b = make_sdesc(qaddr + (kk >> 2) * (C::N * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B);
            umma_bf16_ss(tmem + db * C::N, a, b, C::IDESC, kk > 0);
          }
          umma_commit(empty + s);
          umma_commit(dfull + db);
        }
        if (ok) umma_commit(qempty + qb);
      }
      // on an aborted run, wait (bounded) until every issued MMA retired
      if (!ok && dt > 0) {
        umma_commit(fin);
        mbar_wait_drain(fin, 0);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // Warp ew reads TMEM lane quadrant ew % 4 (keys quad*32 .. +31 of the
    // tile) and scores queries [QPW*qset, QPW*qset + QPW) of the tile: the
    // QPW 32-column slices are loaded together and waited for once, then each
    // score is a ReLU-weighted head sum with four independent accumulators
    // (head weights read four at a time from shared memory).
    const int ew = warp - 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int qset = ew >> 2;
    constexpr int QPW = C::QPW;
    int dt = 0, it = 0;
    bool ok = true;
    for (int ii = blockIdx.x; ii < n_items && ok; ii += gridDim.x, ++it) {
      int t0, ntok, kb, ke;
      int nv[QPW];
      if (direct) {
        int s_, nv_;
        if (!direct_item(m, ii, t0, s_, kb, ke, nv_)) {
          --it;
          continue;
        }
        ntok = 1;
#pragma unroll
        for (int j = 0; j < QPW; ++j) nv[j] = qset * QPW + j < ntok ? nv_ : 0;
      } else {
        const int4 item = items[ii];
        t0 = item.x, ntok = item.y >> 24, kb = item.z, ke = item.w;
#pragma unroll
        for (int j = 0; j < QPW; ++j) {
          const int q = qset * QPW + j;
          nv[j] = q < ntok ? pl.nvis[t0 + q] : 0;
        }
      }
      const int qb = it & 1;
      if (!(ok = mbar_wait(qfull + qb, (it >> 1) & 1, abort_flag))) break;
      const float* wq = w_s + qb * C::N;
      for (int tile = kb / 128; tile * 128 < ke; ++tile, ++dt) {
        const int db = dt & 1;
        if (!(ok = mbar_wait(dfull + db, (dt >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const int key = tile * 128 + quad * 32 + lane;
        uint32_t r[QPW][32];
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + db * C::N + qset * QPW * 32;
#pragma unroll
        for (int j = 0; j < QPW; ++j) tmem_ld32(taddr + j * 32, r[j]);
        tmem_ld_wait_regs(r[0]);
#pragma unroll
        for (int j = 1; j < QPW; ++j) reg_fence(r[j]);
        // the D buffer is free as soon as the values are in registers
        tc_fence_before();
        mbar_arrive(dempty + db);
#pragma unroll
        for (int j = 0; j < QPW; ++j) {
          const int q = qset * QPW + j;
          if (q >= ntok) break;  // warp-uniform
          const float4* w4 = reinterpret_cast<const float4*>(wq + q * 32);
          uint64_t acc[2] = {0ull, 0ull};  // four partial sums in two packed pairs
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wv = w4[h4];
            const float a0 = fmaxf(__uint_as_float(r[j][4 * h4 + 0]), 0.f);
            const float a1 = fmaxf(__uint_as_float(r[j][4 * h4 + 1]), 0.f);
            const float a2 = fmaxf(__uint_as_float(r[j][4 * h4 + 2]), 0.f);
            const float a3 = fmaxf(__uint_as_float(r[j][4 * h4 + 3]), 0.f);
            acc[0] = ffma2(f32x2_pack(a0, a1), f32x2_pack(wv.x, wv.y), acc[0]);
            acc[1] = ffma2(f32x2_pack(a2, a3), f32x2_pack(wv.z, wv.w), acc[1]);
          }
          float s0, s1, s2, s3;
          f32x2_unpack(acc[0], s0, s1);
          f32x2_unpack(acc[1], s2, s3);
          const float sc = (s0 + s1) + (s2 + s3);
          const bool valid = key >= kb && key < ke && key < nv[j];
          if (out.tok_scores && valid) out.tok_scores[(size_t)(t0 + q) * out.ld_tok + key] = sc;
          if (out.gran_scores) {
            // the maximum of this quadrant's 32 keys: one granule (a page
            // of ps keys is ps / 32 granules, folded by the page top-k)
            const float pm = warp_max_f32(valid ? sc : -INFINITY);
            const int qkey0 = tile * 128 + quad * 32;  // first key of this quadrant
            if (lane == 0 && qkey0 < nv[j] && qkey0 >= kb)
              out.gran_scores[(size_t)(t0 + q) * out.ld_gr + qkey0 / 32] = pm;
          }
        }
      }
      if (ok) mbar_arrive(qempty + qb);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Normal path: the epilogue consumed every D buffer, so the tensor pipe
    // is idle. Aborted path: the issuer drained its MMAs above.
    if (*abort_flag && lane == 0) set_status(m.dev_status, DSA_STATUS_TIMEOUT);
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host
IndexerLayout indexer_layout(int T, int S, int max_kv, int ps) {
  IndexerLayout L{};
  const long long ch1 = kChunkDecode, ch8 = kChunkPrefill;
  const long long nchunk1 = (max_kv + ch1 - 1) / ch1, nchunk8 = (max_kv + ch8 - 1) / ch8;
  const long long dec_tiles = S, pre_tiles = (T + 7) / 8 + S;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.counts = take(16);
  L.nvis = take((size_t)T * 4);
  L.seq_tile_off = take((size_t)S * 8);
  L.dec_tiles = take((size_t)dec_tiles * 16);
  L.pre_tiles = take((size_t)pre_tiles * 16);
  L.dec_items = take((size_t)(dec_tiles * nchunk1) * 16);
  L.pre_items = take((size_t)(pre_tiles * nchunk8) * 16);
  L.ld_tok = align_up((size_t)max_kv, 128);
  L.ld_gr = align_up((size_t)(max_kv + 31) / 32, 4);
  L.ld_pg = align_up((size_t)(max_kv + ps - 1) / ps, 4);
  L.tok_scores = take((size_t)T * L.ld_tok * 4);
  L.gran_scores = take((size_t)T * L.ld_gr * 4);
  L.page_scores = take((size_t)T * L.ld_pg * 4);
  L.total = off;
  return L;
}

int run_indexer(cudaStream_t stream, const IndexerMeta& m, const uint16_t* q, const uint16_t* kcache, void* ws,
                const IndexerLayout& L, bool want_tok, bool want_page, IndexerPlan* plan_out, IndexerOut* out_out) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  IndexerPlan pl;
  pl.counts = reinterpret_cast<int*>(base + L.counts);
  pl.nvis = reinterpret_cast<int*>(base + L.nvis);
  pl.seq_tile_off = reinterpret_cast<int2*>(base + L.seq_tile_off);
  pl.dec_tiles = reinterpret_cast<int4*>(base + L.dec_tiles);
  pl.pre_tiles = reinterpret_cast<int4*>(base + L.pre_tiles);
  pl.dec_items = reinterpret_cast<int4*>(base + L.dec_items);
  pl.pre_items = reinterpret_cast<int4*>(base + L.pre_items);
  IndexerOut out;
  out.tok_scores = want_tok ? reinterpret_cast<float*>(base + L.tok_scores) : nullptr;
  out.gran_scores = want_page ? reinterpret_cast<float*>(base + L.gran_scores) : nullptr;
  out.ld_tok = (long long)L.ld_tok;
  out.ld_gr = (long long)L.ld_gr;
  *plan_out = pl;
  *out_out = out;
  if (m.T == 0) return DSA_OK;

  CUtensorMap kmap, qmap;
  if (!encode_bf16_2d(&kmap, kcache, (uint64_t)m.P * m.ps, 128, m.ps, 128)) return DSA_ERR_CUDA;
  if (!encode_bf16_2d(&qmap, q, (uint64_t)m.T * 32, 128, 32, 128)) return DSA_ERR_CUDA;
  CUtensorMap qmap8;
  if (!encode_bf16_2d(&qmap8, q, (uint64_t)m.T * 32, 128, 256, 128)) return DSA_ERR_CUDA;

  const int sms = sm_count();
  // keys per one-token work item: 512, doubled while the decode keys (at most
  // T x max_kv) still give every SM four items or more, up to 64 pages
  // (measured: long-context decode 0.55 -> 0.44 ms with 4096-key items; fewer
  // item boundaries, where a persistent CTA waits on the next item's
  // metadata and query, in the key stream)
  int ch1 = kChunkDecode;
  const long long decode_keys = (long long)m.T * m.max_kv;
  while (ch1 < kChunkDecodeMax && 2 * ch1 <= 64 * m.ps && decode_keys / (2LL * ch1) >= 4LL * sms) ch1 *= 2;
  // as many tokens as requests: a decode batch (or requests without new
  // tokens beside multi-token ones, whose tokens are then scored one by one)
  const int one_token = m.T == m.S ? 1 : 0;
  IndexerMeta m1 = m;
  const long long nch = (m.max_kv + ch1 - 1) / ch1;
  if (one_token && (long long)m.T * nch < (1LL << 31)) {
    // no planner: the one-query kernel derives its items from the token index
    m1.direct_nch = (int)nch;
    m1.direct_ch = ch1;
  } else {
    DSA_LAUNCH_PDL(indexer_plan_kernel, dim3(1), dim3(1024), 0, stream, m, pl, ch1, kChunkPrefill, one_token);
  }
  {
    using C = IdxCfg<1>;
    set_smem_attr_once(reinterpret_cast<const void*>(indexer_score_kernel<1>), C::SMEM);
    DSA_LAUNCH_PDL(indexer_score_kernel<1>, dim3(sms), dim3(C::THREADS), C::SMEM, stream, m1, pl, out, kmap, qmap);
  }
  if (!one_token) {
    using C = IdxCfg<8>;
    set_smem_attr_once(reinterpret_cast<const void*>(indexer_score_kernel<8>), C::SMEM);
    DSA_LAUNCH_PDL(indexer_score_kernel<8>, dim3(sms), dim3(C::THREADS), C::SMEM, stream, m, pl, out, kmap, qmap8);
  }
  return DSA_OK;
}

}  // namespace dsa
