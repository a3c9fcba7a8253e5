// Absorbed-MLA sparse attention on tcgen05 (ref.py, sparse_mla_ref; and the
// query-block form of sparse_mla_prefill_qblock.py, _qblock_kernel).
//
// One CTA computes one query token x up to 128 heads x one half of the
// 512-wide latent value. Per 32-key tile:
//   S[128 heads x 32 keys] = Q[128 x 576] * K_tile[32 x 576]^T   (TMEM, fp32)
//   online softmax over the keys, in registers, one head per thread
//   O[128 x 256] += P[128 x 32] * V_tile[32 x 256]              (TMEM, fp32)
// O of all 512 value columns would fill the whole 512-column TMEM, leaving no
// room for S, so the value width is split across two CTAs that both form S
// (the pair reads the same keys; the second read is an L2 hit).
//
// Q[:, 0:448] is kept in TMEM and feeds QK^T as the A operand (tcgen05 "TS"
// form), which keeps shared memory free for five KV stages and removes most
// of the A-operand shared-memory traffic; Q[:, 448:576] stays in shared
// memory. Keys are gathered row by row (1152 bytes each) with cp.async into
// the ring of 128-byte-swizzled column blocks; the same bytes serve as the
// K-major B operand of QK^T and as the MN-major B operand of PV. One warp
// walks the key list ahead of the gather and prefetches the rows into L2.
// Key lists come from (a) token top-k rows, (b) page top-k rows, or (c) a
// query block's union + membership bitmap (qblock form). Masked keys are
// zero-filled and get probability 0.
#include "common.cuh"
#include "attend.cuh"

namespace dsa {

namespace {
constexpr int kThreads = 256;  // warp 0 MMA, warp 1 key generator, warps 2-3 gather, warps 4-7 softmax
constexpr int kCopyThreads = 64;
constexpr int kTileKeys = 32;
constexpr int kStages = 5;   // KV tiles resident in shared memory
constexpr int kRing = 8;     // key-address tiles generated (and L2-prefetched) ahead of the gather
constexpr int kDk = 576, kDv = 512, kDvHalf = 256;
constexpr int kQTmemDims = 448;  // Q[:, 0:448] lives in TMEM (224 columns), Q[:, 448:576] in smem
constexpr int kQTmemSteps = kQTmemDims / 16;  // 28 of the 36 K-steps read A from TMEM
constexpr int kQsBytes = 128 * (kDk - kQTmemDims) * 2;  // 32768: 2 column blocks x 16 KB
constexpr int kStageBytes = kTileKeys * kDk * 2;        // 36864: 9 column blocks x 4 KB
constexpr int kPBytes = 128 * kTileKeys * 2;            // 8192
constexpr int OFF_QS = 0;
constexpr int OFF_ST = OFF_QS + kQsBytes;
constexpr int OFF_P = OFF_ST + kStages * kStageBytes;
constexpr int OFF_RING = OFF_P + kPBytes;         // int32 [kRing][32] physical rows
constexpr int OFF_RINFO = OFF_RING + kRing * 32 * 4;  // uint32 mask[kRing], end[kRing]
constexpr int OFF_SINFO = OFF_RINFO + kRing * 8;      // uint32 mask[kStages], end[kStages]
constexpr int OFF_BAR = (OFF_SINFO + kStages * 8 + 7) & ~7;
constexpr int NBAR = 2 * kStages + 2 * kRing + 5;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int kSmem = OFF_MISC + 16;
constexpr uint32_t kIdescQK = make_idesc_bf16(128, kTileKeys, false, false);
constexpr uint32_t kIdescPV = make_idesc_bf16(128, kDvHalf, false, true);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;    // 224 columns of packed bf16 pairs
constexpr uint32_t kColS = 224;  // 32 fp32 columns
constexpr uint32_t kColO = 256;  // 256 fp32 columns
constexpr float kRescaleThreshold = 8.f;  // log2 units: p stays <= 256
}  // namespace

// Warp-wide generator of 32-key tiles. Every lane gets the flat physical row
// of "its" key (or -1) and the ballot of valid keys; returns false when the
// CTA's key list is exhausted. Runs on one full warp.
struct TileGen {
  const AttendParams* p;
  int mode, t, seq, pos, kv_len, n_vis, page_base;
  // token / page modes
  int e, e1, sub;
  uint32_t pend;      // page mode: entries of the current 32-window still to visit
  int win;            // page / qblock: start of the current 32-window
  int cur, cur_valid; // current page entry (page mode) or unit (qblock)
  // qblock
  int b, qq, cnt;

  __device__ void init(const AttendParams& prm, int tok, int split) {
    p = &prm;
    mode = prm.mode;
    t = tok;
    TokenGeom g = token_geom(prm.seq_lens, prm.cu_q_lens, prm.cu_kv_lens, prm.S, prm.ps, 0x3fffffff, tok,
                             prm.dev_status);
    seq = g.seq;
    pos = g.pos;
    kv_len = g.kv_len;
    n_vis = g.n_vis;
    page_base = g.page_base;
    sub = 0;
    pend = 0;
    cur = -1;
    cur_valid = 0;
    if (mode == kModeQblock) {
      b = tok / prm.QB;
      qq = tok % prm.QB;
      cnt = min(__ldg(prm.counts + b), prm.u_max);
      win = 0;
    } else {
      const int per = ((prm.K + prm.nsplit - 1) / prm.nsplit + 31) & ~31;
      e = split * per;
      e1 = min(prm.K, e + per);
      win = e;
    }
  }

  // physical flat row of sequence-local key position j (page entry checked)
  __device__ __forceinline__ long long phys_row(int j) const {
    const int ent = page_base + j / p->ps;
    if (ent >= p->PTW) {
      set_status(p->dev_status, DSA_STATUS_BAD_INDEX);
      return -1;
    }
    const int pg = __ldg(p->page_indices + ent);
    if (pg < 0 || pg >= p->P) {
      set_status(p->dev_status, DSA_STATUS_BAD_METADATA);
      return -1;
    }
    return (long long)pg * p->ps + j % p->ps;
  }

  __device__ bool next(long long& row, uint32_t& mask) {
    const int lane = lane_id();
    const int tiles_per_unit = p->ps / kTileKeys;
    while (true) {
      if (mode == kModeToken) {
        if (e >= e1) return false;
        const int ee = e + lane;
        const int j = ee < e1 ? __ldg(p->sel + (size_t)t * p->K + ee) : -1;
        const bool v = j >= 0 && j < n_vis;
        row = v ? phys_row(j) : -1;
        mask = __ballot_sync(0xffffffffu, v && row >= 0);
        e += 32;
        if (mask) return true;
        continue;
      }
      // page and qblock modes walk units of ps keys, 32 keys per tile
      if (cur_valid && sub < tiles_per_unit) {
        const int k0 = sub * kTileKeys + lane;
        bool v;
        long long r = -1;
        if (mode == kModePage) {
          const int j = cur * p->ps + k0;
          v = j < n_vis;
          if (v) r = phys_row(j);
        } else {
          // qblock: unit g = cur, kp = g*ps + r - base_tok
          const long long kp = (long long)cur * p->ps + k0 - (long long)page_base * p->ps;
          v = kp <= pos && kp < kv_len;
          if (v) {
            const int pg = __ldg(p->page_indices + cur);
            if (pg < 0 || pg >= p->P) {
              set_status(p->dev_status, DSA_STATUS_BAD_METADATA);
              v = false;
            } else {
              r = (long long)pg * p->ps + k0;
            }
          }
        }
        ++sub;
        row = v ? r : -1;
        mask = __ballot_sync(0xffffffffu, v && r >= 0);
        if (mask) return true;
        continue;
      }
      // advance to the next unit
      cur_valid = 0;
      sub = 0;
      if (!pend) {
        // refill a window of 32 candidate units
        if (mode == kModePage) {
          if (win >= e1) return false;
          const int ee = win + lane;
          const int pg = ee < e1 ? __ldg(p->sel + (size_t)t * p->K + ee) : -1;
          pend = __ballot_sync(0xffffffffu, pg >= 0 && (long long)pg * p->ps < n_vis);
        } else {
          if (win >= cnt) return false;
          const int u = win + lane;
          bool has = false;
          if (u < cnt) {
            const uint32_t wd =
                __ldg(p->member + ((size_t)b * p->u_max + u) * (p->QB / 32) + (qq >> 5));
            has = (wd >> (qq & 31)) & 1u;
          }
          pend = __ballot_sync(0xffffffffu, has);
        }
        win += 32;
        continue;
      }
      const int bit = __ffs(pend) - 1;
      pend &= pend - 1u;
      const int idx = win - 32 + bit;
      if (mode == kModePage) {
        cur = __ldg(p->sel + (size_t)t * p->K + idx);
        cur_valid = 1;
      } else {
        const int g = __ldg(p->units + (size_t)b * p->u_max + idx);
        if (g < 0 || g >= p->PTW) {
          if (lane == 0) set_status(p->dev_status, DSA_STATUS_BAD_INDEX);
          continue;
        }
        cur = g;
        cur_valid = 1;
      }
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const AttendParams prm) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(prm.dev_status, DSA_STATUS_INTERNAL);
    return;
  }
  const int warp = warp_id(), lane = lane_id(), tid = threadIdx.x;
  const int half = blockIdx.x & 1, hg = blockIdx.x >> 1;
  const int t = blockIdx.y, split = blockIdx.z;
  const int h0 = hg * 128;
  uint8_t* qs_s = smem + OFF_QS;
  uint8_t* st_s = smem + OFF_ST;
  uint8_t* p_s = smem + OFF_P;
  int* ring_rows = reinterpret_cast<int*>(smem + OFF_RING);
  volatile uint32_t* ring_mask = reinterpret_cast<volatile uint32_t*>(smem + OFF_RINFO);
  volatile uint32_t* ring_end = ring_mask + kRing;
  volatile uint32_t* st_mask = reinterpret_cast<volatile uint32_t*>(smem + OFF_SINFO);
  volatile uint32_t* st_end = st_mask + kStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;                  // [kStages] 64 async + 1 leader arrivals
  uint64_t* empty = bars + kStages;       // [kStages] PV commit
  uint64_t* rfull = bars + 2 * kStages;   // [kRing] generator
  uint64_t* rempty = rfull + kRing;       // [kRing] 64 gather threads
  uint64_t* sfull = rempty + kRing;       // QK commit
  uint64_t* sempty = sfull + 1;           // 128 softmax threads
  uint64_t* pfull = sfull + 2;            // 128 softmax threads
  uint64_t* pempty = sfull + 3;           // PV commit
  uint64_t* fin = sfull + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full + i, kCopyThreads + 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(rfull + i, 1);
      mbar_init(rempty + i, kCopyThreads);
    }
    mbar_init(sfull, 1);
    mbar_init(sempty, 128);
    mbar_init(pfull, 128);
    mbar_init(pempty, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  const int nh = min(128, prm.H - h0);
  const uint16_t* qt = prm.q + ((size_t)t * prm.H + h0) * kDk;
  // Q[:, 448:576] -> two 128-byte-swizzled column blocks in shared memory
  {
    const uint32_t qbase = smem_u32(qs_s);
    constexpr int CH = (kDk - kQTmemDims) / 8;  // 16 chunks of 16 bytes per row
    for (int c = tid; c < 128 * CH; c += kThreads) {
      const int r = c / CH, ch = c % CH;
      const bool ok = r < nh;
      const uint16_t* src = ok ? qt + (size_t)r * kDk + kQTmemDims + ch * 8 : prm.q;
      cp_async16(qbase + (ch >> 3) * 16384 + sw128_offset(r, ch & 7), src, ok ? 16u : 0u);
    }
    cp_async_commit();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 4) {
    // Q[:, 0:448] -> TMEM lanes (one head row per lane), bf16 pairs per column
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint4* src = reinterpret_cast<const uint4*>(qt + (size_t)r * kDk);
#pragma unroll 1
    for (int c0 = 0; c0 < kQTmemDims / 2; c0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 x = r < nh ? __ldg(src + c0 / 4 + j) : make_uint4(0, 0, 0, 0);
        v[4 * j] = x.x;
        v[4 * j + 1] = x.y;
        v[4 * j + 2] = x.z;
        v[4 * j + 3] = x.w;
      }
      tmem_st32(tmem + lane_base + kColQ + c0, v);
    }
    tmem_st_wait();
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t qsaddr = smem_u32(qs_s), paddr = smem_u32(p_s);
      auto issue_qk = [&](int i) {
        const uint32_t kaddr = smem_u32(st_s + (i % kStages) * kStageBytes);
#pragma unroll 4
        for (int kk = 0; kk < kQTmemSteps; ++kk) {
          const uint64_t b = make_sdesc(kaddr + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          umma_bf16_ts(tmem + kColS, tmem + kColQ + kk * 8, b, kIdescQK, kk > 0);
        }
#pragma unroll
        for (int kk = kQTmemSteps; kk < kDk / 16; ++kk) {
          const int k2 = kk - kQTmemSteps;
          const uint64_t a = make_sdesc(qsaddr + (k2 >> 2) * 16384 + (k2 & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t b = make_sdesc(kaddr + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          umma_bf16_ss(tmem + kColS, a, b, kIdescQK, 1u);
        }
        umma_commit(sfull);
      };
      auto issue_pv = [&](int i) {
        const int s = i % kStages;
        const uint32_t vaddr = smem_u32(st_s + s * kStageBytes) + half * 4 * 4096;
#pragma unroll
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
          const uint64_t a = make_sdesc(paddr + ks * 2 * 128, 128, 512, kSwizzleNone);
          const uint64_t b = make_sdesc(vaddr + ks * 16 * 128, 4096, 1024, kSwizzle128B);
          umma_bf16_ss(tmem + kColO, a, b, kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(empty + s);
        umma_commit(pempty);
      };
      bool ok = mbar_wait(full + 0, 0, abort_flag);
      int issued = 0;
      if (ok && !st_end[0]) {
        fence_proxy_async_smem();  // cp.async data -> async proxy
        tc_fence_after();
        issue_qk(0);
        issued = 1;
        for (int i = 0;; ++i) {
          const int s1 = (i + 1) % kStages;
          if (!(ok = mbar_wait(full + s1, ((i + 1) / kStages) & 1, abort_flag))) break;
          const bool end1 = st_end[s1] != 0;
          if (!end1) {
            fence_proxy_async_smem();
            // single S buffer: softmax must have read S(i)
            if (!(ok = mbar_wait(sempty, i & 1, abort_flag))) break;
            tc_fence_after();
            issue_qk(i + 1);
          }
          if (!(ok = mbar_wait(pfull, i & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(i);
          if (end1) break;
        }
      }
      if (!ok && issued) {
        umma_commit(fin);
        mbar_wait_drain(fin, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ key generator + L2 prefetch
    TileGen gen;
    gen.init(prm, t, split);
    for (int j = 0;; ++j) {
      long long row = -1;
      uint32_t mask = 0;
      const bool more = gen.next(row, mask);
      const int slot = j % kRing;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(rempty + slot, ((j / kRing) & 1) ^ 1, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ring_rows[slot * 32 + lane] = more ? (int)row : -1;
      if (more && row >= 0) prefetch_l2_bulk(prm.kv + (size_t)row * prm.row_stride, kDk * 2);
      if (lane == 0) {
        ring_mask[slot] = mask;
        ring_end[slot] = more ? 0u : 1u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rfull + slot);
      if (!more) break;
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ gather
    const int ctid = tid - 64;
    const uint32_t stbase = smem_u32(st_s);
    for (int i = 0;; ++i) {
      const int slot = i % kRing, s = i % kStages;
      if (!mbar_wait(rfull + slot, (i / kRing) & 1, abort_flag)) break;
      const bool end = ring_end[slot] != 0;
      const uint32_t mask = ring_mask[slot];
      if (!mbar_wait(empty + s, ((i / kStages) & 1) ^ 1, abort_flag)) break;
      if (!end) {
        const uint32_t dst0 = stbase + s * kStageBytes;
        for (int c = ctid; c < kTileKeys * 72; c += kCopyThreads) {
          const int key = c / 72, ch = c % 72;
          const int r = ring_rows[slot * 32 + key];
          const uint16_t* src = r >= 0 ? prm.kv + (size_t)r * prm.row_stride + ch * 8 : prm.kv;
          cp_async16(dst0 + (ch >> 3) * 4096 + sw128_offset(key, ch & 7), src, r >= 0 ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(full + s);
      } else {
        mbar_arrive(full + s);
      }
      if (ctid == 0) {
        st_mask[s] = mask;
        st_end[s] = end ? 1u : 0u;
        mbar_arrive(full + s);
      }
      mbar_arrive(rempty + slot);
      if (end) break;
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = (warp & 3) * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = prm.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0;
    bool ok = true;
    for (int i = 0;; ++i) {
      const int s = i % kStages;
      if (!(ok = mbar_wait(full + s, (i / kStages) & 1, abort_flag))) break;
      if (st_end[s]) break;
      const uint32_t mask = st_mask[s];
      if (!(ok = mbar_wait(sfull, i & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base + kColS, sv);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(sempty);
      float x[32];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = ((mask >> j) & 1u) ? __uint_as_float(sv[j]) * sl2 : -INFINITY;
        mt = fmaxf(mt, x[j]);
      }
      const float m_new = fmaxf(m_run, mt);
      const bool need = m_new > m_run + kRescaleThreshold;  // also true when m_run == -inf
      const float m_use = need ? m_new : m_run;
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      float psum = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = exp2f(x[j] - m_use), p1 = exp2f(x[j + 1] - m_use);
        psum += p0 + p1;
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        pk[j >> 1] = *reinterpret_cast<uint32_t*>(&b2);
      }
      l_run = l_run * alpha + psum;
      m_run = m_use;
      if (i > 0) {
        if (!(ok = mbar_wait(pempty, (i - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < kDvHalf / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tmem_st32(tmem + lane_base + kColO + c * 32, ov);
          }
          tmem_st_wait();
        }
      }
      // P row -> no-swizzle K-major core matrices: (r/8)*512 + (j/8)*128 + (r%8)*16
      uint8_t* prow = p_s + (r >> 3) * 512 + (r & 7) * 16;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + c * 128) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(pfull);
      n = i + 1;
    }
    // epilogue
    if (ok && n > 0) ok = mbar_wait(pempty, (n - 1) & 1, abort_flag);
    tc_fence_after();
    const int h = h0 + r;
    const bool hv = h < prm.H;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const size_t orow = ((size_t)t * prm.H + h) * kDv + half * kDvHalf;
    const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    if (prm.nsplit == 1) {
      for (int c = 0; c < kDvHalf / 32; ++c) {
        uint32_t ov[32];
        if (n > 0 && ok) {
          tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        if (hv) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            __nv_bfloat162 b2 =
                __floats2bfloat162_rn(__uint_as_float(ov[j]) * inv_l, __uint_as_float(ov[j + 1]) * inv_l);
            pk[j >> 1] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(prm.o + orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (hv && half == 0 && prm.lse) prm.lse[(size_t)t * prm.H + h] = lse_v;
    } else {
      float* op = prm.o_part + ((size_t)split * prm.T * prm.H) * kDv;
      for (int c = 0; c < kDvHalf / 32; ++c) {
        uint32_t ov[32];
        if (n > 0 && ok) {
          tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        if (hv) {
          float4* dst = reinterpret_cast<float4*>(op + orow + c * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(ov[4 * v]) * inv_l, __uint_as_float(ov[4 * v + 1]) * inv_l,
                                 __uint_as_float(ov[4 * v + 2]) * inv_l, __uint_as_float(ov[4 * v + 3]) * inv_l);
        }
      }
      if (hv && half == 0) prm.lse_part[((size_t)split * prm.T + t) * prm.H + h] = lse_v;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (*abort_flag && lane == 0) set_status(prm.dev_status, DSA_STATUS_TIMEOUT);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge split-key partials: o = sum_z e^{lse_z - M} o_z / sum_z e^{lse_z - M}.
__global__ void __launch_bounds__(256) combine_splits_kernel(const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part, int nsplit, int T,
                                                             int H, uint16_t* __restrict__ o, float* __restrict__ lse) {
  const int th = blockIdx.x;  // (t, h)
  if (th >= T * H) return;
  __shared__ float wts[16];
  __shared__ float s_lse;
  if (threadIdx.x == 0) {
    float mx = -INFINITY;
    for (int z = 0; z < nsplit; ++z) mx = fmaxf(mx, lse_part[(size_t)z * T * H + th]);
    float tot = 0.f;
    for (int z = 0; z < nsplit; ++z) {
      const float l = lse_part[(size_t)z * T * H + th];
      const float wz = (mx == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - mx);
      wts[z] = wz;
      tot += wz;
    }
    for (int z = 0; z < nsplit; ++z) wts[z] = tot > 0.f ? wts[z] / tot : 0.f;
    s_lse = tot > 0.f ? mx + __logf(tot) : -INFINITY;
  }
  __syncthreads();
  const int c = threadIdx.x * 2;  // 256 threads x 2 columns = 512
  float a0 = 0.f, a1 = 0.f;
  for (int z = 0; z < nsplit; ++z) {
    const float2 v = *reinterpret_cast<const float2*>(o_part + ((size_t)z * T * H + th) * kDv + c);
    a0 = fmaf(wts[z], v.x, a0);
    a1 = fmaf(wts[z], v.y, a1);
  }
  __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
  *reinterpret_cast<__nv_bfloat162*>(o + (size_t)th * kDv + c) = b2;
  if (lse && threadIdx.x == 0) lse[th] = s_lse;
}

int attend_num_splits(int T, int H, int K, int mode) {
  if (mode == kModeQblock) return 1;
  const int ctas = T * 2 * ((H + 127) / 128);
  const int target = 2 * sm_count();
  int z = ctas >= target ? 1 : (target + ctas - 1) / ctas;
  const int max_by_k = mode == kModeToken ? max(1, (K + 31) / 32) : max(1, K);
  z = min(z, min(16, max_by_k));
  return max(1, z);
}

size_t attend_workspace_bytes(int T, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  return align_up((size_t)nsplit * T * H * kDv * 4, 256) + align_up((size_t)nsplit * T * H * 4, 256);
}

int run_attend(cudaStream_t stream, AttendParams prm, void* ws, size_t ws_bytes) {
  if (prm.T == 0 || prm.H == 0) return DSA_OK;
  if (prm.nsplit > 1) {
    if (!ws || ws_bytes < attend_workspace_bytes(prm.T, prm.H, prm.nsplit)) return DSA_ERR_WORKSPACE;
    prm.o_part = static_cast<float*>(ws);
    prm.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                            align_up((size_t)prm.nsplit * prm.T * prm.H * kDv * 4, 256));
  }
  cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  dim3 grid(2 * ((prm.H + 127) / 128), prm.T, prm.nsplit);
  sparse_mla_kernel<<<grid, kThreads, kSmem, stream>>>(prm);
  DSA_CHECK_LAUNCH();
  if (prm.nsplit > 1) {
    combine_splits_kernel<<<prm.T * prm.H, 256, 0, stream>>>(prm.o_part, prm.lse_part, prm.nsplit, prm.T, prm.H,
                                                            prm.o, prm.lse);
    DSA_CHECK_LAUNCH();
  }
  return DSA_OK;
}

}  // namespace dsa
