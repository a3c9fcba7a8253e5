// Absorbed-MLA sparse attention on tcgen05 (ref.py, sparse_mla_ref; and the
// query-block form of sparse_mla_prefill_qblock.py, _qblock_kernel).
//
// One CTA computes one query token x up to 128 heads x one half of the
// 512-wide latent value. Per 64-key tile:
//   S[128 heads x 64 keys] = Q[128 x 576] * K_tile[64 x 576]^T   (TMEM, fp32)
//   online softmax over the keys, in registers, one head per thread
//   O[128 x 256] += P[128 x 64] * V_tile[64 x 256]              (TMEM, fp32)
// O of all 512 value columns would fill the whole 512-column TMEM, leaving no
// room for S, so the value width is split across two CTAs that both form S
// (the pair reads the same keys; the second read is an L2 hit).
//
// A tcgen05.mma with M = 128 and K = 16 costs about the same for every N up
// to 64, so keys are multiplied 64 at a time: a 32-key tile would leave the
// tensor pipe idle half of the time. Q[:, 0:256] is kept in TMEM and feeds
// QK^T as the A operand (tcgen05 "TS" form); Q[:, 256:576] stays in shared
// memory. S is double-buffered in TMEM and the softmax writes P (bf16) back
// over its S buffer, where PV reads it as a TS-form A operand, so QK^T of the
// next tile never waits for the softmax. Each key tile is stored as nine
// 128-byte-swizzled column blocks of 64 dims; the same bytes are the K-major
// B operand of QK^T and the MN-major B operand of PV. The four blocks holding
// this CTA's value half (the "V part") are only released once PV has read
// them; the other five (the "K part") as soon as QK^T has.
//
// Keys are resolved 32 at a time by one warp (token top-k rows, page top-k
// rows, or a query block's union + membership bitmap). The page-run modes
// (page units, query blocks, dense) fetch every step, 32 consecutive rows of
// one page, with 2-D TMA boxes; token mode fetches its scattered rows with
// coalesced cp.async; each has an instantiation of its own. Masked keys are
// zero-filled or carry P = 0.
#include <atomic>

#include "common.cuh"
#include "attend.cuh"

namespace dsa {

namespace {
// warp 0 MMA, warp 1 key generator, warps 2-3 and 8.. gather, warps 4-7 softmax.
// Scattered token rows are copied by ten warps (512 threads: more copies in
// flight, measured 10% faster decode than six, as fast as eight); the
// page-run modes, whose steps are single TMA boxes, run with four (320
// threads) in an instantiation of their own (measured against 2, 3, 5, 6 and
// 8: query-block prefill 6.50 ms with six, 6.35 with four).
constexpr int kCopyWarpsToken = 10;
constexpr int kCopyWarpsRuns = 4;
constexpr int kSubKeys = 32;   // keys resolved / copied per generator step
constexpr int kTileKeys = 64;  // keys per MMA tile (two generator steps)
// generator steps buffered ahead of the gather: token mode keeps 32 physical
// rows per step, the page-run modes only a step's first row, so their ring
// can be deeper in the same shared memory
constexpr int kRingToken = 18;
constexpr int kRingRuns = 32;
constexpr int kDk = 576, kDv = 512, kDvHalf = 256;
constexpr int kBlk = kTileKeys * 128;   // one 64-dim column block of a tile: 8 KB
constexpr int kKBlocks = 5, kVBlocks = 4;
constexpr int kKStages = 2, kVStages = 2;
constexpr int kKStageBytes = kKBlocks * kBlk;  // 40960
constexpr int kVStageBytes = kVBlocks * kBlk;  // 32768
constexpr int kQTmemBlocks = 4;                // Q column blocks 0..3 in TMEM (128 columns)
constexpr int kQTmemDims = kQTmemBlocks * 64;  // 256
constexpr int kQsBytes = (kDk - kQTmemDims) / 64 * 16384;  // 5 column blocks x 16 KB
constexpr int OFF_QS = 0;
constexpr int OFF_KST = OFF_QS + kQsBytes;
constexpr int OFF_VST = OFF_KST + kKStages * kKStageBytes;
// the tail of the shared-memory layout, after the value stages: the
// generator ring (R steps; ROWS: with 32 physical rows per step), stage
// flags, barriers and a few words
template <int R, bool ROWS>
struct RingLayout {
  static constexpr int OFF_RING = OFF_VST + kVStages * kVStageBytes;  // int32 [R][32] physical rows (ROWS)
  static constexpr int OFF_RINFO = OFF_RING + (ROWS ? R * 32 * 4 : 0);  // uint32 mask[R], end[R]
  static constexpr int OFF_RBASE = OFF_RINFO + R * 8;   // int32 first row of each step [R]
  static constexpr int OFF_SINFO = OFF_RBASE + R * 4;   // uint32 kend[kKStages], vmask[kVStages][2], vend[kVStages]
  static constexpr int OFF_BAR = (OFF_SINFO + (kKStages + 3 * kVStages) * 4 + 7) & ~7;
  static constexpr int NBAR = 2 * kKStages + 2 * kVStages + 2 * R + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};
template <int kCopyW>
using LayoutOf = RingLayout<kCopyW == kCopyWarpsToken ? kRingToken : kRingRuns, kCopyW == kCopyWarpsToken>;
static_assert(OFF_KST % 1024 == 0 && OFF_VST % 1024 == 0, "swizzle atoms need 1 KB alignment");
constexpr uint32_t kIdescQK = make_idesc_bf16(128, kTileKeys, false, false);
constexpr uint32_t kIdescPV = make_idesc_bf16(128, kDvHalf, false, true);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;    // 128 columns of packed bf16 pairs
constexpr uint32_t kColS = 128;  // two S buffers of 64 fp32 columns; P (bf16 pairs) overwrites S
constexpr uint32_t kColO = 256;  // 256 fp32 columns
constexpr float kRescaleThreshold = 8.f;  // log2 units: p stays <= 256
constexpr int kMaxSplits = 8;
// epilogue stage: 128 rows of 256 fp32 values, rows padded to 1040 bytes so
// that eight lanes writing eight rows hit eight different bank groups
constexpr int kStageLd = kDvHalf + 4;
constexpr int OFF_STAGE = 0;
constexpr int OFF_WTS = OFF_STAGE + 128 * kStageLd * 4;  // fp32 merge weights [kMaxSplits][128]
static_assert(OFF_WTS + kMaxSplits * 128 * 4 <= OFF_VST, "the stage must stay clear of the value stages");
// every full barrier completes after two generator steps' worth of arrivals:
// each gather thread once per step, plus one more by the leader per step
__device__ __forceinline__ uint32_t full_arrivals(int copy_threads) { return 2u * (uint32_t)(copy_threads + 1); }

}  // namespace

// Warp-wide generator of 32-key tiles. Every lane gets the flat physical row
// of "its" key (or -1) and the ballot of valid keys; returns false when the
// CTA's key list is exhausted. Runs on one full warp. Loads are batched so a
// whole window of selections (8 x 32 token entries, or 32 pages / union
// slots) resolves to physical rows in two or three dependent global loads.
struct TileGen {
  static constexpr int GB = 8;  // token windows resolved per refill
  const AttendParams* p;
  int mode, t, seq, pos, kv_len, n_vis, page_base;
  int e, e1;          // token / page modes: next entry, end of this CTA's range
  int win;            // page / qblock: start of the next 32-window
  // token mode: buffered tiles
  int buf_row[GB];
  uint32_t buf_mask[GB];
  uint32_t buf_pend;  // windows of the buffer with keys, not returned yet
  // page / qblock modes: current window
  uint32_t pend;      // units of the window still to visit
  int w_key0;         // this lane's unit: first key position (page) or kp base (qblock)
  int w_phys;         // this lane's unit: physical page, -1 if none
  int cur_key0, cur_phys, sub, cur_valid;
  int b, qq, cnt;     // qblock
  int ps_log2;        // the page size is a power of two
  int key_lo;         // dense: first key position inside the window

  __device__ void init(const AttendParams& prm, int tok, int split) {
    p = &prm;
    mode = prm.mode;
    ps_log2 = 31 - __clz(prm.ps);
    t = tok;
    const int sq = seq_of_token_warp(prm.cu_q_lens, prm.S, tok);
    TokenGeom g = token_geom(prm.seq_lens, prm.cu_q_lens, prm.cu_kv_lens, prm.S, prm.ps, 0x3fffffff, tok,
                             prm.dev_status, sq);
    seq = g.seq;
    pos = g.pos;
    kv_len = g.kv_len;
    n_vis = g.n_vis;
    page_base = g.page_base;
    buf_pend = 0;
    pend = 0;
    sub = 0;
    cur_valid = 0;
    key_lo = 0;
    if (mode == kModeDense) {
      // every page that holds a visible position inside the window, split
      // evenly across the CTAs of this token
      key_lo = prm.window > 0 ? max(0, pos - prm.window + 1) : 0;
      const int p_lo = key_lo / prm.ps, p_hi = (n_vis + prm.ps - 1) / prm.ps;
      const int per = (max(0, p_hi - p_lo) + prm.nsplit - 1) / prm.nsplit;
      e = min(p_hi, p_lo + split * per);
      e1 = min(p_hi, e + per);
      win = e;
    } else if (mode == kModeQblock) {
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

  // physical page of packed page-table entry `ent` (checked), or -1
  __device__ __forceinline__ int page_of(int ent) const {
    if (ent < 0 || ent >= p->PTW) {
      set_status(p->dev_status, DSA_STATUS_BAD_INDEX);
      return -1;
    }
    const int pg = __ldg(p->page_indices + ent);
    if (pg < 0 || pg >= p->P) {
      set_status(p->dev_status, DSA_STATUS_BAD_METADATA);
      return -1;
    }
    return pg;
  }

  // base: first physical row of the tile when its 32 keys are 32 consecutive
  // rows of one page (page and qblock modes), else -1
  __device__ bool next(long long& row, uint32_t& mask, long long& base) {
    const int lane = lane_id();
    const int ps = p->ps;
    base = -1;
    if (mode == kModeToken) {
      while (!buf_pend) {
        if (e >= e1) return false;
        int j[GB];
#pragma unroll
        for (int g = 0; g < GB; ++g) {
          const int ee = e + 32 * g + lane;
          j[g] = ee < e1 ? __ldg(p->sel + (size_t)t * p->K + ee) : -1;
        }
        int pg[GB];
#pragma unroll
        for (int g = 0; g < GB; ++g) pg[g] = (j[g] >= 0 && j[g] < n_vis) ? page_of(page_base + (j[g] >> ps_log2)) : -1;
        // every array index below is a compile-time constant, so the buffer
        // stays in registers
#pragma unroll
        for (int g = 0; g < GB; ++g) {
          const bool v = pg[g] >= 0;
          const uint32_t m = __ballot_sync(0xffffffffu, v);
          buf_row[g] = v ? pg[g] * ps + (j[g] & (ps - 1)) : -1;
          buf_mask[g] = m;
          buf_pend |= (m ? 1u : 0u) << g;
        }
        e += 32 * GB;
      }
      const int gsel = __ffs(buf_pend) - 1;
      buf_pend &= buf_pend - 1u;
      int r = -1;
      uint32_t m = 0;
#pragma unroll
      for (int g = 0; g < GB; ++g)
        if (g == gsel) {
          r = buf_row[g];
          m = buf_mask[g];
        }
      row = r;
      mask = m;
      return true;
    }
    const int tiles_per_unit = ps / kSubKeys;
    while (true) {
      if (cur_valid && sub < tiles_per_unit) {
        const int k0 = sub * kSubKeys + lane;
        bool v;
        if (mode == kModePage) {
          v = cur_key0 + k0 < n_vis;
        } else if (mode == kModeDense) {
          v = cur_key0 + k0 < n_vis && cur_key0 + k0 >= key_lo;
        } else {
          const int kp = cur_key0 + k0;  // kp = g*ps + r - base_tok
          v = kp <= pos && kp < kv_len;
        }
        base = (long long)cur_phys * ps + sub * kSubKeys;
        ++sub;
        row = v ? (long long)cur_phys * ps + k0 : -1;
        mask = __ballot_sync(0xffffffffu, v);
        if (mask) return true;
        continue;
      }
      cur_valid = 0;
      sub = 0;
      if (!pend) {
        // resolve a window of 32 candidate units to physical pages
        if (mode == kModeDense) {
          if (win >= e1) return false;
          const int pgl = win + lane;
          w_phys = pgl < e1 ? page_of(page_base + pgl) : -1;
          w_key0 = pgl * ps;
        } else if (mode == kModePage) {
          if (win >= e1) return false;
          const int ee = win + lane;
          const int pgl = ee < e1 ? __ldg(p->sel + (size_t)t * p->K + ee) : -1;
          const bool v = pgl >= 0 && (long long)pgl * ps < n_vis;
          w_phys = v ? page_of(page_base + pgl) : -1;
          w_key0 = pgl * ps;
        } else {
          if (win >= cnt) return false;
          const int u = win + lane;
          bool has = false;
          int g = -1;
          if (u < cnt) {
            const uint32_t wd = __ldg(p->member + ((size_t)b * p->u_max + u) * (p->QB / 32) + (qq >> 5));
            g = __ldg(p->units + (size_t)b * p->u_max + u);
            has = (wd >> (qq & 31)) & 1u;
          }
          w_phys = has ? page_of(g) : -1;
          w_key0 = (g - page_base) * ps;
        }
        pend = __ballot_sync(0xffffffffu, w_phys >= 0);
        win += 32;
        continue;
      }
      const int bit = __ffs(pend) - 1;
      pend &= pend - 1u;
      cur_phys = __shfl_sync(0xffffffffu, w_phys, bit);
      cur_key0 = __shfl_sync(0xffffffffu, w_key0, bit);
      cur_valid = 1;
    }
  }
};

// The MMA issuer (one thread). Every operand descriptor is a base register
// plus a compile-time offset, so issuing an MMA costs a couple of
// instructions: a single thread that has to build descriptors, branch and
// wait on dependent integer ops between MMAs cannot keep the tensor pipe fed
// at these small N. The value half is a template argument for that reason.
//
// Order per tile i: QK^T(i) over the K part, then over the V part (into S
// buffer i % 2), then PV(i-1) with P(i-1) read from TMEM. With two S buffers
// QK^T(i) never waits for the softmax of tile i-1, whose TMEM read of S
// takes on the order of a thousand cycles to land.
struct MmaBars {
  uint64_t *kfull, *kempty, *vfull, *vempty, *sfull, *pfull, *pempty, *fin;
};

template <int HALF>
__device__ __forceinline__ void mma_issuer(uint32_t tmem, uint32_t qs_addr, uint32_t kst_addr, uint32_t vst_addr,
                                           const MmaBars& br, volatile uint32_t* kst_end, volatile int* abort_flag) {
  const uint64_t dq = make_sdesc(qs_addr, 16, 1024, kSwizzle128B);
  const uint64_t dk[2] = {make_sdesc(kst_addr, 16, 1024, kSwizzle128B),
                          make_sdesc(kst_addr + kKStageBytes, 16, 1024, kSwizzle128B)};
  const uint64_t dv[2] = {make_sdesc(vst_addr, 16, 1024, kSwizzle128B),
                          make_sdesc(vst_addr + kVStageBytes, 16, 1024, kSwizzle128B)};
  // the V part as the MN-major B operand of PV: 64-column blocks kBlk apart
  const uint64_t dvn[2] = {make_sdesc(vst_addr, kBlk, 1024, kSwizzle128B),
                           make_sdesc(vst_addr + kVStageBytes, kBlk, 1024, kSwizzle128B)};
  static_assert(kKStages == 2 && kVStages == 2, "stage selection below assumes two stages");
  const uint32_t tO = tmem + kColO, tQ = tmem + kColQ;
  // descriptors address shared memory in 16-byte units in their low bits
  auto qk_block = [&](const uint32_t tS, const int c, const uint64_t b0, const bool first) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t b = b0 + (uint64_t)((kk * 32) >> 4);
      const uint32_t acc = (first && kk == 0) ? 0u : 1u;
      if (c < kQTmemBlocks)
        umma_bf16_ts(tS, tQ + c * 32 + kk * 8, b, kIdescQK, acc);
      else
        umma_bf16_ss(tS, dq + (uint64_t)(((c - kQTmemBlocks) * 16384 + kk * 32) >> 4), b, kIdescQK, acc);
    }
  };
  bool ok = true;
  int issued = 0;
  for (int i = 0;; ++i) {
    const int ks = i & 1, vs = i & 1;
    if (!(ok = mbar_wait(br.kfull + ks, (i >> 1) & 1, abort_flag))) break;
    const bool end = kst_end[ks] != 0;
    if (!end) {
      // S buffer i % 2 last held P(i-2), which PV(i-2) (issued before this
      // point, and the tensor pipe runs in order) has read
      const uint32_t tS = tmem + kColS + (uint32_t)(i & 1) * kTileKeys;
      fence_proxy_async_smem();  // cp.async data -> async proxy
      tc_fence_after();
      const uint64_t kb = ks ? dk[1] : dk[0];
#pragma unroll
      for (int pos = 0; pos < kKBlocks; ++pos)
        qk_block(tS, HALF == 0 ? 4 + pos : (pos < 4 ? pos : 8), kb + (uint64_t)((pos * kBlk) >> 4), pos == 0);
      umma_commit(br.kempty + ks);
      issued = 1;
      if (!(ok = mbar_wait(br.vfull + vs, (i >> 1) & 1, abort_flag))) break;
      fence_proxy_async_smem();
      tc_fence_after();
      const uint64_t vb = vs ? dv[1] : dv[0];
#pragma unroll
      for (int pos = 0; pos < kVBlocks; ++pos)
        qk_block(tS, 4 * HALF + pos, vb + (uint64_t)((pos * kBlk) >> 4), false);
      umma_commit(br.sfull + (i & 1));
    }
    if (i > 0) {
      const int j = i - 1;
      if (!(ok = mbar_wait(br.pfull + (j & 1), (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t tP = tmem + kColS + (uint32_t)(j & 1) * kTileKeys;  // P(j): 32 columns of bf16 pairs
      const uint64_t vb = (j & 1) ? dvn[1] : dvn[0];
#pragma unroll
      for (int k2 = 0; k2 < kTileKeys / 16; ++k2)
        umma_bf16_ts(tO, tP + k2 * 8, vb + (uint64_t)((k2 * 16 * 128) >> 4), kIdescPV, (j > 0 || k2 > 0) ? 1u : 0u);
      umma_commit(br.vempty + (j & 1));
      umma_commit(br.pempty);
    }
    if (end) break;
  }
  if (!ok && issued) {
    umma_commit(br.fin);
    mbar_wait_drain(br.fin, 0);
  }
}

// kSoftCap: the logit cap of the dense fallback, a separate instantiation
// so that the common path carries none of its code
// kCopyW: copier warps (kCopyWarpsToken or kCopyWarpsRuns); the block has
// (6 + kCopyW) warps
template <bool kSoftCap, int kCopyW>
__global__ void __launch_bounds__((6 + kCopyW) * 32, 1)
    sparse_mla_kernel(const AttendParams prm, const __grid_constant__ CUtensorMap kvmap,
                      const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(prm.dev_status, DSA_STATUS_INTERNAL);
    return;
  }
  griddep_launch_dependents();
  const int warp = warp_id(), lane = lane_id(), tid = threadIdx.x;
  constexpr int n_copy_warps = kCopyW;
  constexpr int n_copy_threads = n_copy_warps * 32;
  const int half = blockIdx.x & 1, hg = blockIdx.x >> 1;
  const int t = prm.t0 + (int)blockIdx.y, split = blockIdx.z;
  const int h0 = hg * 128;
  uint8_t* qs_s = smem + OFF_QS;
  uint8_t* kst_s = smem + OFF_KST;
  uint8_t* vst_s = smem + OFF_VST;
  using L = LayoutOf<kCopyW>;
  constexpr int kRing = kCopyW == kCopyWarpsToken ? kRingToken : kRingRuns;
  constexpr bool kRows = kCopyW == kCopyWarpsToken;  // page-run steps carry only their first row
  int* ring_rows = reinterpret_cast<int*>(smem + L::OFF_RING);
  volatile uint32_t* ring_mask = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_RINFO);
  volatile uint32_t* ring_end = ring_mask + kRing;
  volatile int* ring_base = reinterpret_cast<volatile int*>(smem + L::OFF_RBASE);
  volatile uint32_t* kst_end = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_SINFO);
  volatile uint32_t* vst_mask = kst_end + kKStages;   // [kVStages][2]
  volatile uint32_t* vst_end = vst_mask + 2 * kVStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kfull = bars;                 // [kKStages] full_arrivals + tx bytes
  uint64_t* kempty = kfull + kKStages;    // [kKStages] commit after the K-part MMAs
  uint64_t* vfull = kempty + kKStages;    // [kVStages] full_arrivals + tx bytes
  uint64_t* vempty = vfull + kVStages;    // [kVStages] commit after PV
  uint64_t* rfull = vempty + kVStages;    // [kRing] generator
  uint64_t* rempty = rfull + kRing;       // [kRing] gather threads
  uint64_t* sfull = rempty + kRing;       // [2] QK^T commit, one per S buffer
  uint64_t* pfull = sfull + 2;            // [2] 128 softmax threads (P written over S)
  uint64_t* pempty = sfull + 4;           // PV commit
  uint64_t* fin = sfull + 5;
  uint64_t* qbar = sfull + 6;             // the query block's TMA copy
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(kfull + i, full_arrivals(n_copy_threads));
      mbar_init(kempty + i, 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(vfull + i, full_arrivals(n_copy_threads));
      mbar_init(vempty + i, 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(rfull + i, 1);
      mbar_init(rempty + i, n_copy_threads);
    }
    mbar_init(sfull, 1);
    mbar_init(sfull + 1, 1);
    mbar_init(pfull, 128);
    mbar_init(pfull + 1, 128);
    mbar_init(pempty, 1);
    mbar_init(fin, 1);
    mbar_init(qbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // barrier initialisation must be visible before the Q copy signals one
  __syncthreads();
  // the local set-up above overlaps the previous kernel of the stream; global
  // memory is touched only after it has completed
  griddep_wait();
  // Q rows h0..h0+127 of token t (rows past H belong to the next token or
  // lie past the tensor, where TMA fills zeros; their outputs are never
  // stored) as nine 128-byte-swizzled column blocks: Q[:, 256:576] stays in
  // shared memory, Q[:, 0:256] waits in the still unused key stages until
  // the softmax warps move it into TMEM.
  uint8_t* qstage = kst_s;
  static_assert(kQTmemBlocks * 16384 <= kKStages * kKStageBytes, "Q staging fits");
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, (kDk / 64) * 16384);
#pragma unroll 1
    for (int c = 0; c < kDk / 64; ++c)
      tma_load_2d(c < kQTmemBlocks ? qstage + c * 16384 : qs_s + (c - kQTmemBlocks) * 16384, &qmap, qbar, c * 64,
                  t * prm.H + h0);
  }
  // The key generator (warp 1) resolves its first window of selections while
  // Q arrives; it publishes steps only after the barrier below. (Measured:
  // calling TileGen::next from the generator loop alone, which halves its
  // inlined code, made the query-block prefill 60% slower; the time of this
  // kernel follows its code layout as much as its instruction count.)
  TileGen gen;
  bool gen_more = false;
  long long gen_row = -1, gen_base = -1;
  uint32_t gen_mask = 0;
  if (warp == 1) {
    gen.init(prm, t, split);
    gen_more = gen.next(gen_row, gen_mask, gen_base);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 4 && warp < 8) {
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    if (mbar_wait(qbar, 0, abort_flag)) {
#pragma unroll 1
      for (int c = 0; c < kQTmemBlocks; ++c) {
        const uint8_t* row = qstage + c * 16384 + r * 128;
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
          v[4 * j] = x.x;
          v[4 * j + 1] = x.y;
          v[4 * j + 2] = x.z;
          v[4 * j + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + kColQ + c * 32, v);
      }
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const MmaBars br{kfull, kempty, vfull, vempty, sfull, pfull, pempty, fin};
      mbar_wait(qbar, 0, abort_flag);
      if (half == 0)
        mma_issuer<0>(tmem, smem_u32(qs_s), smem_u32(kst_s), smem_u32(vst_s), br, kst_end, abort_flag);
      else
        mma_issuer<1>(tmem, smem_u32(qs_s), smem_u32(kst_s), smem_u32(vst_s), br, kst_end, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ key generator
    // Steps are published in pairs (one MMA tile); a list that ends after an
    // odd number of steps gets one empty step (no keys) to complete its tile.
    int j = 0;
    auto publish = [&](long long row, uint32_t mask, long long base, bool end) -> bool {
      const int slot = j % kRing;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(rempty + slot, ((j / kRing) & 1) ^ 1, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      if constexpr (kRows) ring_rows[slot * 32 + lane] = end ? -1 : (int)row;
      if (lane == 0) {
        ring_mask[slot] = end ? 0u : mask;
        ring_end[slot] = end ? 1u : 0u;
        ring_base[slot] = end ? -1 : (int)base;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rfull + slot);
      ++j;
      return true;
    };
    for (bool first = true;; first = false) {
      long long row = gen_row, base = gen_base;
      uint32_t mask = gen_mask;
      const bool more = first ? gen_more : gen.next(row, mask, base);
      // decode rows come from all over HBM: start pulling this step's rows
      // into L2 now, a whole ring ahead of the gather (union pages of a query
      // block are shared by its queries and are L2-resident anyway)
      if (more && row >= 0 && (prm.mode == kModeToken || prm.mode == kModePage)) {
        const char* rp = reinterpret_cast<const char*>(prm.kv + (size_t)row * prm.row_stride);
#pragma unroll
        for (int l = 0; l < kDk * 2 / 128; ++l) prefetch_l2_line(rp + l * 128);
      }
      if (!more && (j & 1)) {
        // its first row -32: a page-run box of rows -32..-1 lies wholly
        // outside the tensor and is zero-filled (no stray cache row is read)
        if (!publish(-1, 0u, -kSubKeys, false)) break;
      }
      if (!publish(row, mask, base, !more)) break;
      if (!more) break;
    }
  } else if (warp < 4 || warp >= 8) {
    // ------------------------------------------------------------ gather
    // Tile by tile (two generator steps): the K parts of both steps as soon
    // as the K stage is free, then the V parts once PV has released the V
    // stage, so a K part is never held up behind the V stage.
    const int cw = warp < 4 ? warp - 2 : warp - 6;  // 0 .. n_copy_warps - 1
    const int ctid = cw * 32 + lane;
    // scattered rows: copier warp cw copies keys cw, cw+n, ... of a step; per
    // key the K part is 40 16-byte chunks (lanes 0..31, then 0..7 again) and
    // the V part 32 (one per lane), each a contiguous run of the row
    const int kc1 = lane + 32;
    const int kpos0 = lane >> 3, kpos1 = kc1 >> 3;
    const int kcol0 = half == 0 ? 4 + kpos0 : kpos0;            // kpos0 < 4
    const int kcol1 = half == 0 ? 4 + kpos1 : (kpos1 < 4 ? kpos1 : 8);
    const int vcol = 4 * half + (lane >> 3);
    const int src_k0 = kcol0 * 64 + (lane & 7) * 8, src_k1 = kcol1 * 64 + (kc1 & 7) * 8;
    const int src_v = vcol * 64 + (lane & 7) * 8;
    const uint32_t dst_k0 = kpos0 * kBlk, dst_k1 = kpos1 * kBlk, dst_v = (lane >> 3) * kBlk;
    for (int ti = 0;; ++ti) {
      const int j0 = 2 * ti, s0 = j0 % kRing, s1 = (j0 + 1) % kRing;
      const int ks = ti % kKStages, vs = ti % kVStages;
      if (!mbar_wait(rfull + s0, (j0 / kRing) & 1, abort_flag)) break;
      if (ring_end[s0]) {
        // the end marker stands for a whole tile: both steps' arrivals
        if (!mbar_wait(kempty + ks, ((ti / kKStages) & 1) ^ 1, abort_flag)) break;
        if (!mbar_wait(vempty + vs, ((ti / kVStages) & 1) ^ 1, abort_flag)) break;
        if (ctid == 0) {
          kst_end[ks] = 1u;
          vst_end[vs] = 1u;
          mbar_arrive(kfull + ks);
          mbar_arrive(vfull + vs);
          mbar_arrive(kfull + ks);
          mbar_arrive(vfull + vs);
        }
        mbar_arrive(kfull + ks);
        mbar_arrive(vfull + vs);
        mbar_arrive(kfull + ks);
        mbar_arrive(vfull + vs);
        mbar_arrive(rempty + s0);
        break;
      }
      if (!mbar_wait(rfull + s1, ((j0 + 1) / kRing) & 1, abort_flag)) break;
      const int base0 = ring_base[s0], base1 = ring_base[s1];
      // ---- K parts
      if (!mbar_wait(kempty + ks, ((ti / kKStages) & 1) ^ 1, abort_flag)) break;
      const uint32_t kd = smem_u32(kst_s + ks * kKStageBytes);
#pragma unroll 1
      for (int sb = 0; sb < 2; ++sb) {
        const int slot = sb ? s1 : s0, cbase = sb ? base1 : base0;
        const uint32_t d = kd + sb * (kSubKeys * 128);
        // page-run modes: every step is 32 consecutive rows of one page, one
        // 2-D TMA box (64 cols x 32 rows) per block; token mode: every step
        // is 32 scattered rows
        if constexpr (!kRows) {
          if (ctid == 0) {
            mbar_arrive_expect_tx(kfull + ks, kKBlocks * kSubKeys * 128);
#pragma unroll 1
            for (int pos = 0; pos < kKBlocks; ++pos) {
              const int c = half == 0 ? 4 + pos : (pos < 4 ? pos : 8);
              tma_load_2d(kst_s + ks * kKStageBytes + sb * (kSubKeys * 128) + pos * kBlk, &kvmap, kfull + ks,
                          c * 64, cbase);
            }
          } else {
            mbar_arrive(kfull + ks);
          }
        } else {
#pragma unroll 2
          for (int key = cw; key < kSubKeys; key += n_copy_warps) {
            const int r = ring_rows[slot * 32 + key];
            const uint16_t* rb = r >= 0 ? prm.kv + (size_t)r * prm.row_stride : prm.kv;
            const uint32_t nb = r >= 0 ? 16u : 0u;
            cp_async16(d + dst_k0 + sw128_offset(key, lane & 7), rb + src_k0, nb);
            if (lane < 8) cp_async16(d + dst_k1 + sw128_offset(key, kc1 & 7), rb + src_k1, nb);
          }
          cp_async_mbar_arrive_noinc(kfull + ks);
        }
      }
      if (ctid == 0) {
        kst_end[ks] = 0u;
        mbar_arrive(kfull + ks);
        mbar_arrive(kfull + ks);
      }
      // ---- V parts
      if (!mbar_wait(vempty + vs, ((ti / kVStages) & 1) ^ 1, abort_flag)) break;
      const uint32_t vd = smem_u32(vst_s + vs * kVStageBytes);
#pragma unroll 1
      for (int sb = 0; sb < 2; ++sb) {
        const int slot = sb ? s1 : s0, cbase = sb ? base1 : base0;
        const uint32_t d = vd + sb * (kSubKeys * 128);
        if constexpr (!kRows) {
          if (ctid == 0) {
            mbar_arrive_expect_tx(vfull + vs, kVBlocks * kSubKeys * 128);
#pragma unroll 1
            for (int pos = 0; pos < kVBlocks; ++pos)
              tma_load_2d(vst_s + vs * kVStageBytes + sb * (kSubKeys * 128) + pos * kBlk, &kvmap, vfull + vs,
                          (4 * half + pos) * 64, cbase);
          } else {
            mbar_arrive(vfull + vs);
          }
        } else {
#pragma unroll 2
          for (int key = cw; key < kSubKeys; key += n_copy_warps) {
            const int r = ring_rows[slot * 32 + key];
            const uint16_t* rb = r >= 0 ? prm.kv + (size_t)r * prm.row_stride : prm.kv;
            cp_async16(d + dst_v + sw128_offset(key, lane & 7), rb + src_v, r >= 0 ? 16u : 0u);
          }
          cp_async_mbar_arrive_noinc(vfull + vs);
        }
      }
      if (ctid == 0) {
        vst_mask[2 * vs] = ring_mask[s0];
        vst_mask[2 * vs + 1] = ring_mask[s1];
        vst_end[vs] = 0u;
        mbar_arrive(vfull + vs);
        mbar_arrive(vfull + vs);
      }
      mbar_arrive(rempty + s0);
      mbar_arrive(rempty + s1);
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
      const int vs = i % kVStages;
      if (!(ok = mbar_wait(vfull + vs, (i / kVStages) & 1, abort_flag))) break;
      if (vst_end[vs]) break;
      const uint32_t mlo = vst_mask[2 * vs], mhi = vst_mask[2 * vs + 1];
      if (!(ok = mbar_wait(sfull + (i & 1), (i >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + kColS + (uint32_t)(i & 1) * kTileKeys;
      uint32_t sa[32], sb[32];
      tmem_ld32(tS, sa);
      tmem_ld32(tS + 32, sb);
      tmem_ld_wait();
      // scaled, masked logits in place (log2 units); independent partial
      // maxima keep the dependency chains short
      float sc = sl2;
      if (kSoftCap) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          sa[j] = __float_as_uint(prm.cap_log2 * tanh_approx(__uint_as_float(sa[j]) * prm.inv_cap_scale));
          sb[j] = __float_as_uint(prm.cap_log2 * tanh_approx(__uint_as_float(sb[j]) * prm.inv_cap_scale));
        }
        sc = 1.f;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if ((mlo & mhi) == 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float a = __uint_as_float(sa[j]) * sc, b = __uint_as_float(sb[j]) * sc;
          sa[j] = __float_as_uint(a);
          sb[j] = __float_as_uint(b);
          mx4[j & 1] = fmaxf(mx4[j & 1], a);
          mx4[2 + (j & 1)] = fmaxf(mx4[2 + (j & 1)], b);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float a = ((mlo >> j) & 1u) ? __uint_as_float(sa[j]) * sc : -INFINITY;
          const float b = ((mhi >> j) & 1u) ? __uint_as_float(sb[j]) * sc : -INFINITY;
          sa[j] = __float_as_uint(a);
          sb[j] = __float_as_uint(b);
          mx4[j & 1] = fmaxf(mx4[j & 1], a);
          mx4[2 + (j & 1)] = fmaxf(mx4[2 + (j & 1)], b);
        }
      }
      const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m_run, mt);
      const bool need = m_new > m_run + kRescaleThreshold;  // also true when m_run == -inf
      const float m_use = need ? m_new : m_run;
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      // rescaling O must wait until PV(i-1) has added into it; P(i) goes to
      // the other S buffer than P(i-1), so without a rescale nothing waits
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        if (!(ok = mbar_wait(pempty, (i - 1) & 1, abort_flag))) break;
        tc_fence_after();
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
      // P row r as bf16 pairs (lower key in the low half) over the first 32
      // columns of its S buffer: the A operand of PV in the tcgen05 TS form
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float x0 = __uint_as_float(c < 16 ? sa[2 * c] : sb[2 * c - 32]);
        const float x1 = __uint_as_float(c < 16 ? sa[2 * c + 1] : sb[2 * c - 31]);
        const float p0 = ex2_approx(x0 - m_use), p1 = ex2_approx(x1 - m_use);
        ps4[c & 3] += p0 + p1;
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        pw[c] = *reinterpret_cast<uint32_t*>(&b2);
      }
      tmem_st32(tS, pw);
      tmem_st_wait();
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      l_run = l_run * alpha + psum;
      m_run = m_use;
      tc_fence_before();
      mbar_arrive(pfull + (i & 1));
      n = i + 1;
    }
    // epilogue
    if (ok && n > 0) ok = mbar_wait(pempty, (n - 1) & 1, abort_flag);
    tc_fence_after();
    const int h = h0 + r;
    const bool hv = h < prm.H;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    const bool have_o = n > 0 && ok;
    // O is read back from TMEM 64 columns at a time (one wait per two loads)
    auto load_o64 = [&](int c0, uint32_t (&oa)[32], uint32_t (&ob)[32]) {
      if (have_o) {
        tmem_ld32(tmem + lane_base + kColO + c0, oa);
        tmem_ld32(tmem + lane_base + kColO + c0 + 32, ob);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) oa[j] = ob[j] = 0u;
      }
    };
    if (prm.nsplit == 1) {
      // one split: the warp stages its 32 head rows as bf16 in the idle key
      // stage (four 128-byte-swizzled boxes of 64 columns) and one lane
      // writes them with four TMA stores; rows past H lie outside the tensor
      // map and are not written. (Each thread storing its own row made every
      // warp store touch 32 lines.)
      uint8_t* stg = kst_s + (warp & 3) * 16384;
      const uint32_t stg_a = smem_u32(stg);
#pragma unroll 1
      for (int c0 = 0; c0 < kDvHalf; c0 += 64) {
        uint32_t oa[32], ob[32];
        load_o64(c0, oa, ob);
        const uint32_t box = stg_a + (uint32_t)(c0 / 64) * 4096u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t x0 = j < 4 ? oa[8 * j + 2 * e] : ob[8 * (j - 4) + 2 * e];
            const uint32_t x1 = j < 4 ? oa[8 * j + 2 * e + 1] : ob[8 * (j - 4) + 2 * e + 1];
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(x0) * inv_l, __uint_as_float(x1) * inv_l);
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          st_shared_v4(box + sw128_offset((uint32_t)lane, (uint32_t)j), pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int hw = h0 + (warp & 3) * 32;  // first head row of this warp
      if (lane == 0 && hw < prm.H) {
#pragma unroll 1
        for (int c = 0; c < kDvHalf / 64; ++c) tma_store_3d(&omap, stg + c * 4096, half * kDvHalf + c * 64, hw, t);
        bulk_commit();
        bulk_wait_read();
      }
      __syncwarp();
      if (hv && half == 0 && prm.lse) prm.lse[(size_t)t * prm.H + h] = lse_v;
    } else {
      // split keys: each CTA stages its normalised partial (rows scaled by
      // 1/l) in shared memory; below, every warp of the CTA writes it out and,
      // in the last CTA of the (token, value half) group, merges all splits.
      // The stage reuses the Q and key buffers, idle once the last PV has
      // completed; its rows are padded to 1040 bytes against bank conflicts.
      float* stg = reinterpret_cast<float*>(smem + OFF_STAGE) + (warp & 3) * 32 * kStageLd;
#pragma unroll 1
      for (int c0 = 0; c0 < kDvHalf; c0 += 64) {
        uint32_t oa[32], ob[32];
        load_o64(c0, oa, ob);
        float4* srow = reinterpret_cast<float4*>(stg + lane * kStageLd + c0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          srow[v] = make_float4(__uint_as_float(oa[4 * v]) * inv_l, __uint_as_float(oa[4 * v + 1]) * inv_l,
                                __uint_as_float(oa[4 * v + 2]) * inv_l, __uint_as_float(oa[4 * v + 3]) * inv_l);
          srow[8 + v] = make_float4(__uint_as_float(ob[4 * v]) * inv_l, __uint_as_float(ob[4 * v + 1]) * inv_l,
                                    __uint_as_float(ob[4 * v + 2]) * inv_l, __uint_as_float(ob[4 * v + 3]) * inv_l);
        }
      }
      // lse of this split as seen by this CTA (both value halves compute the
      // same logits, so each group merges with its own copies)
      prm.lse_part[(size_t)gridDim.x * 128 + (((size_t)split * prm.T + t) * gridDim.x + blockIdx.x) * 128 + r] =
          lse_v;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (*abort_flag && lane == 0) {
      set_status(prm.dev_status, DSA_STATUS_TIMEOUT);
      mbar_wait_drain(qbar, 0);  // the Q copy must not land after the CTA exits
    }
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (prm.nsplit > 1) {
    // Split keys, with every warp of the CTA (the staged partial is complete
    // and every role has finished at the barrier above). A warp moves one
    // 1 KB head row at a time, 32 lanes over consecutive 16-byte pieces, so
    // that every store and every load covers whole cache lines; the merge
    // runs its loads on all warps because each round of them waits on L2
    // (on the four softmax warps alone the merging CTA took about twice as
    // long as the others).
    const int nw = (int)(blockDim.x >> 5);
    const float* stg = reinterpret_cast<const float*>(smem + OFF_STAGE);
    const int nrows = max(0, min(128, prm.H - h0));  // head rows that exist
    const size_t orow0 = ((size_t)t * prm.H + h0) * kDv + half * kDvHalf;  // element offset of row h0
    const size_t zstride = (size_t)prm.T * prm.H * kDv;
    float* op = prm.o_part + (size_t)split * zstride + orow0;
#pragma unroll 2
    for (int i = warp; i < nrows; i += nw) {
      const float* sr = stg + i * kStageLd;
      float4* dst = reinterpret_cast<float4*>(op + (size_t)i * kDv);
      dst[lane] = *reinterpret_cast<const float4*>(sr + 4 * lane);
      dst[32 + lane] = *reinterpret_cast<const float4*>(sr + 128 + 4 * lane);
    }
    __threadfence();
    __syncthreads();
    volatile int* s_last = abort_flag + 1;
    if (tid == 0) {
      int* ctr = prm.counters + (size_t)t * gridDim.x + blockIdx.x;
      const int old = atomicAdd(ctr, 1);
      const int last = old == prm.nsplit - 1;
      if (last) *ctr = 0;  // ready for the next call
      *s_last = last;
    }
    __syncthreads();
    if (*s_last) {  // uniform over the CTA
      __threadfence();
      // per head row: the weight of each split's partial, in shared memory
      float* wts = reinterpret_cast<float*>(smem + OFF_WTS);
      if (tid < 128) {
        const float* lsep = prm.lse_part + (size_t)gridDim.x * 128;
        auto lse_of = [&](int z) {
          return __ldcg(lsep + (((size_t)z * prm.T + t) * gridDim.x + blockIdx.x) * 128 + tid);
        };
        float mx = -INFINITY;
#pragma unroll 1
        for (int z = 0; z < prm.nsplit; ++z) mx = fmaxf(mx, lse_of(z));
        float tot = 0.f;
#pragma unroll 1
        for (int z = 0; z < prm.nsplit; ++z) {
          const float lz = lse_of(z);
          const float w = (mx == -INFINITY || lz == -INFINITY) ? 0.f : exp2f((lz - mx) * 1.4426950408889634f);
          wts[z * 128 + tid] = w;
          tot += w;
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll 1
        for (int z = 0; z < prm.nsplit; ++z) wts[z * 128 + tid] *= inv;
        if (tid < nrows && half == 0 && prm.lse)
          prm.lse[(size_t)t * prm.H + h0 + tid] = tot > 0.f ? mx + logf(tot) : -INFINITY;
      }
      __syncthreads();
      // every warp merges groups of four rows; this CTA's own split is read
      // from the stage, the others from the partials. The splits are added
      // in the fixed order 0, 1, ..., so an output does not depend on which
      // CTA of its row merges.
      auto store_bf16_4 = [&](uint16_t* dst, float4 a) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      };
      const float* parts = prm.o_part + orow0;
#pragma unroll 1
      for (int i0 = 4 * warp; i0 < nrows; i0 += 4 * nw) {
        float4 acc[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc[u][0] = make_float4(0.f, 0.f, 0.f, 0.f);
          acc[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 1
        for (int z = 0; z < prm.nsplit; ++z) {
          float4 va[4][2];
          if (z == split) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* sr = stg + (i0 + u) * kStageLd;
              va[u][0] = *reinterpret_cast<const float4*>(sr + 4 * lane);
              va[u][1] = *reinterpret_cast<const float4*>(sr + 128 + 4 * lane);
            }
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool live = i0 + u < nrows;
              const float4* src = reinterpret_cast<const float4*>(parts + z * zstride + (size_t)(i0 + u) * kDv);
              va[u][0] = live ? __ldcg(src + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
              va[u][1] = live ? __ldcg(src + 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float w = wts[z * 128 + i0 + u];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              acc[u][e].x = fmaf(w, va[u][e].x, acc[u][e].x);
              acc[u][e].y = fmaf(w, va[u][e].y, acc[u][e].y);
              acc[u][e].z = fmaf(w, va[u][e].z, acc[u][e].z);
              acc[u][e].w = fmaf(w, va[u][e].w, acc[u][e].w);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (i0 + u < nrows) {
            uint16_t* dst = prm.o + orow0 + (size_t)(i0 + u) * kDv;
            store_bf16_4(dst + 4 * lane, acc[u][0]);
            store_bf16_4(dst + 128 + 4 * lane, acc[u][1]);
          }
        }
      }
    }
  }
}

// Split the key list only as far as one wave of CTAs (one per SM) allows:
// more splits cost partial-output traffic and leave a quantised tail.
int attend_num_splits(int T, int H, int K, int mode) {
  if (mode == kModeQblock) return 1;
  const int ctas = T * 2 * ((H + 127) / 128);
  int z = max(1, sm_count() / max(1, ctas));
  const int max_by_k = mode == kModeToken ? max(1, (K + 31) / 32) : max(1, K);  // dense: K = pages
  z = min(z, min(kMaxSplits, max_by_k));
  return max(1, z);
}

// Split-key workspace: fp32 partial outputs [nsplit, T, H, 512], per-CTA lse
// copies [nsplit, T, CTAs per token, 128] (offset by one CTA row of padding),
// and one arrival counter per (token, CTA column).
static size_t part_bytes(int T, int H, int nsplit) { return align_up((size_t)nsplit * T * H * kDv * 4, 256); }
static size_t lse_bytes(int T, int H, int nsplit) {
  const size_t cols = 2 * (size_t)((H + 127) / 128);
  return align_up(((size_t)nsplit * T * cols + cols) * 128 * 4, 256);
}
size_t attend_workspace_bytes(int T, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  const size_t cols = 2 * (size_t)((H + 127) / 128);
  return part_bytes(T, H, nsplit) + lse_bytes(T, H, nsplit) + align_up((size_t)T * cols * 4, 256);
}

int run_attend(cudaStream_t stream, AttendParams prm, void* ws, size_t ws_bytes) {
  if (prm.T == 0 || prm.H == 0) return DSA_OK;
  if (prm.ps < kSubKeys || (prm.ps & (prm.ps - 1))) return DSA_ERR_UNSUPPORTED;  // pages: 2^n rows, n >= 5
  const int cols = 2 * ((prm.H + 127) / 128);
  if (prm.nsplit > 1) {
    if (!ws || ws_bytes < attend_workspace_bytes(prm.T, prm.H, prm.nsplit)) return DSA_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(ws);
    prm.o_part = reinterpret_cast<float*>(base);
    prm.lse_part = reinterpret_cast<float*>(base + part_bytes(prm.T, prm.H, prm.nsplit));
    prm.counters = reinterpret_cast<int*>(base + part_bytes(prm.T, prm.H, prm.nsplit) +
                                          lse_bytes(prm.T, prm.H, prm.nsplit));
    if (cudaMemsetAsync(prm.counters, 0, (size_t)prm.T * cols * 4, stream) != cudaSuccess) return DSA_ERR_CUDA;
  }
  CUtensorMap kvmap, qmap;
  if (!encode_bf16_2d(&kvmap, prm.kv, (uint64_t)prm.P * prm.ps, (uint64_t)prm.row_stride, 32, kDk))
    return DSA_ERR_CUDA;
  if (!encode_bf16_2d(&qmap, prm.q, (uint64_t)prm.T * prm.H, kDk, 128, kDk)) return DSA_ERR_CUDA;
  CUtensorMap omap;  // the output [T][H][512] in boxes of 64 columns x 32 head rows
  if (!encode_bf16_3d(&omap, prm.o, kDv, (uint64_t)prm.H, (uint64_t)prm.T, 32)) return DSA_ERR_CUDA;
  dim3 grid(cols, prm.tn > 0 ? prm.tn : prm.T, prm.nsplit);
  void (*kern)(AttendParams, CUtensorMap, CUtensorMap, CUtensorMap);
  int threads, smem_bytes;
  if (prm.soft_cap_on) {  // dense mode only: page runs
    kern = sparse_mla_kernel<true, kCopyWarpsRuns>;
    threads = (6 + kCopyWarpsRuns) * 32;
    smem_bytes = LayoutOf<kCopyWarpsRuns>::SMEM;
  } else if (prm.mode == kModeToken) {
    kern = sparse_mla_kernel<false, kCopyWarpsToken>;
    threads = (6 + kCopyWarpsToken) * 32;
    smem_bytes = LayoutOf<kCopyWarpsToken>::SMEM;
  } else {
    kern = sparse_mla_kernel<false, kCopyWarpsRuns>;
    threads = (6 + kCopyWarpsRuns) * 32;
    smem_bytes = LayoutOf<kCopyWarpsRuns>::SMEM;
  }
  set_smem_attr_once(reinterpret_cast<const void*>(kern), smem_bytes);
  DSA_LAUNCH_PDL(kern, grid, dim3(threads), smem_bytes, stream, prm, kvmap, qmap, omap);
  return DSA_OK;
}

// ---------------------------------------------------------------------------
// No-allocation variant of the split-key decode path. Its scratch (the split
// partials, their lse values and the merge counters) lives in a file-scope
// device array instead of a caller workspace, so a caller that cannot
// allocate device memory can still run the split path. The array is part of
// the module image: every device that loads the library holds it until the
// process exits.
constexpr size_t kStaticScratchBytes = 24u << 20;  // 24 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of the array on the current device. In host code the name
// g_static_scratch is only a host-side stand-in, so the address is resolved
// once per device, with that device current, the first time it is needed.
// Host threads may race to resolve it: each gets the same address, and the
// atomic slots keep the race benign. Devices 0..kMaxScratchDevices-1 only.
constexpr int kMaxScratchDevices = 64;
static void* static_scratch_address() {
  static std::atomic<void*> addr[kMaxScratchDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
  void* cur = addr[dev].load(std::memory_order_acquire);
  if (!cur) {
    if (cudaGetSymbolAddress(&cur, g_static_scratch) != cudaSuccess) return nullptr;
    addr[dev].store(cur, std::memory_order_release);
  }
  return cur;
}

int run_attend_static_scratch(cudaStream_t stream, AttendParams prm) {
  if (prm.T == 0 || prm.H == 0) return DSA_OK;
  if (prm.nsplit <= 1) return run_attend(stream, prm, nullptr, 0);
  if (attend_workspace_bytes(prm.T, prm.H, prm.nsplit) > kStaticScratchBytes) return DSA_ERR_SCRATCH_LIMIT;
  void* p = static_scratch_address();
  if (!p) return DSA_ERR_CUDA;
  return run_attend(stream, prm, p, kStaticScratchBytes);
}

}  // namespace dsa
