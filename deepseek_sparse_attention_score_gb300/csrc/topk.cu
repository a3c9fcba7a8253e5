// Exact per-row top-k (ref.py, streamindex_topk_ref / streamindex_page_topk_ref
// with exact selection): the k largest of a row's visible scores, ties to the
// lower index, written in ascending index order and -1 padded.
//
// One CTA per row. A 4-pass most-significant-digit radix select (8-bit
// digits, per-warp shared-memory histograms) finds the exact k-th largest key
// K* and how many copies of K* are needed; a final pass of warp ballots and
// two block scans emits every index with key > K* plus the lowest-index
// copies of K*, already in ascending order. Rows that fit are first staged in
// shared memory. Longer rows are read once: a threshold from a strided
// sample of the row bounds a candidate list that then takes the select; when
// the sample misleads (fewer than k or too many candidates) a two-read path
// with an 11-bit histogram, and last a path that re-reads the row from L2 per
// radix pass, take over.
#include "common.cuh"
#include "indexer.cuh"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkThreadsShort = 128;  // threads per row when every row has at most 2048 keys
constexpr int kTopkThreadsMany = 256;   // threads per row for many rows of any length

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 and +0
// map to the same key so they tie like equal scores.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Page score from 32-key granule maxima: unit i of a row covers granules
// fold*i .. fold*i + fold - 1 (fold = 2 or 4), of which only those starting
// below the row's visible length nraw hold scores. The row starts 16-byte
// aligned and its stride is a multiple of four granules.
__device__ __forceinline__ float fold_max(const float* __restrict__ g, int i, int fold, int nraw) {
  const int g0 = i * fold;
  if (fold == 2) {
    const float2 a = __ldg(reinterpret_cast<const float2*>(g) + i);
    return 32 * (g0 + 1) < nraw ? fmaxf(a.x, a.y) : a.x;
  }
  const float4 a = __ldg(reinterpret_cast<const float4*>(g) + i);
  float mx = a.x;
  if (32 * (g0 + 1) < nraw) mx = fmaxf(mx, a.y);
  if (32 * (g0 + 2) < nraw) mx = fmaxf(mx, a.z);
  if (32 * (g0 + 3) < nraw) mx = fmaxf(mx, a.w);
  return mx;
}

template <int TPB>
__device__ __forceinline__ int block_scan_warps(int v, int* s_tmp, int* total) {
  // exclusive scan of one value per warp (lane 0 holds it) across the block
  constexpr int kTopkWarps = TPB / 32;
  const int w = warp_id(), lane = lane_id();
  if (lane == 0) s_tmp[w] = v;
  __syncthreads();
  if (w == 0) {
    int x = lane < kTopkWarps ? s_tmp[lane] : 0;
    const int orig = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kTopkWarps) s_tmp[32 + lane] = x - orig;
    if (lane == kTopkWarps - 1) s_tmp[64] = x;
  }
  __syncthreads();
  const int r = s_tmp[32 + w];
  *total = s_tmp[64];
  __syncthreads();
  return r;
}

// Histogram update into the calling warp's own 256-bin histogram. All lanes
// of the warp must call it (it used to aggregate equal digits with a warp
// match; a plain shared-memory atomic is cheaper for the digit spreads that
// score rows have).
__device__ __forceinline__ void hist_add(uint32_t* wh, uint32_t key, bool valid, uint32_t prefix, uint32_t mask,
                                         int shift) {
  if (valid && (key & mask) == prefix) atomicAdd(wh + ((key >> shift) & 255u), 1u);
}

// Pick the digit holding the rank-`remaining` key from the 256-bin histogram
// (summed over warps) and update prefix / mask / remaining. Block-wide.
template <int TPB>
__device__ __forceinline__ void pick_digit(uint32_t* hist, int shift, uint32_t& prefix, uint32_t& mask,
                                           int& remaining, int* s_sel) {
  constexpr int kTopkWarps = TPB / 32;
  const int tid = threadIdx.x, w = warp_id(), lane = lane_id();
  for (int b = tid; b < 256; b += TPB) {
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < kTopkWarps; ++j) c += hist[j * 256 + b];
    hist[kTopkWarps * 256 + b] = c;
  }
  __syncthreads();
  if (w == 0) {
    const uint32_t* h = hist + kTopkWarps * 256;
    uint32_t local[8];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      local[j] = h[255 - (lane * 8 + j)];
      sum += local[j];
    }
    uint32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    uint32_t above = x - sum;  // keys in digits above this lane's group
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (above < (uint32_t)remaining && above + local[j] >= (uint32_t)remaining) {
        s_sel[0] = 255 - (lane * 8 + j);
        s_sel[1] = (int)above;
      }
      above += local[j];
    }
  }
  __syncthreads();
  const uint32_t d = (uint32_t)s_sel[0];
  remaining -= s_sel[1];
  prefix |= d << shift;
  mask |= 255u << shift;
  __syncthreads();
}

// Ordered emission: every index with key > kstar, plus the lowest-index
// need_eq copies of kstar, in ascending index order. Warp w owns a contiguous
// segment; two block scans give each warp its output offset.
// With s_idx, entry i of the staged keys stands for row position s_idx[i]
// (a compacted candidate list kept in ascending position order).
template <bool kStaged, int TPB>
__device__ void emit_ordered(const float* __restrict__ g, const uint32_t* __restrict__ s_row, int n,
                             uint32_t kstar, int need_eq, int32_t* __restrict__ out_idx, float* __restrict__ out_val,
                             int* s_tmp, const int* __restrict__ s_idx = nullptr) {
  constexpr int kTopkWarps = TPB / 32;
  const int w = warp_id(), lane = lane_id();
  auto key_at = [&](int i) -> uint32_t { return kStaged ? s_row[i] : ordered_key(__ldg(g + i)); };
  const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int seg0 = min(n, w * seg), seg1 = min(n, seg0 + seg);
  const int seg_end = seg1 + ((32 - (seg1 - seg0) % 32) % 32);
  int gt = 0, eq = 0;
  for (int i = seg0 + lane; i < seg_end; i += 32) {
    const bool in = i < seg1;
    const uint32_t key = in ? key_at(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, in && key > kstar));
    eq += __popc(__ballot_sync(0xffffffffu, in && key == kstar));
  }
  int tot;
  const int eq_base = block_scan_warps<TPB>(eq, s_tmp, &tot);
  const int take_eq = max(0, min(need_eq - eq_base, eq));
  const int out_base = block_scan_warps<TPB>(gt + take_eq, s_tmp, &tot);
  const uint32_t lt = (1u << lane) - 1u;
  int eq_run = eq_base, sel_run = out_base;
  for (int i = seg0 + lane; i < seg_end; i += 32) {
    const bool in = i < seg1;
    const uint32_t key = in ? key_at(i) : 0u;
    const bool is_gt = in && key > kstar, is_eq = in && key == kstar;
    const uint32_t eqb = __ballot_sync(0xffffffffu, is_eq);
    const int my_eq_rank = eq_run + __popc(eqb & lt);
    const bool sel = is_gt || (is_eq && my_eq_rank < need_eq);
    const uint32_t selb = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int pos = sel_run + __popc(selb & lt);
      const int j = s_idx ? s_idx[i] : i;
      out_idx[pos] = j;
      if (out_val) out_val[pos] = __ldg(g + j);
    }
    eq_run += __popc(eqb);
    sel_run += __popc(selb);
  }
}

// Bitonic sort of n_pow2 ints in shared memory (ascending), block-wide.
__device__ void bitonic_sort_smem(int* a, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2 / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const int x = a[lo], y = a[hi];
        if ((x > y) == up) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

constexpr int kUnroll = 16;  // float4 loads in flight per thread on the global path

// Row longer than shared memory: radix passes read it from global memory
// (L2) with many loads in flight; the final pass collects the winners
// unordered and sorts them.
template <int TPB>
__device__ void select_row_global(const float* __restrict__ g, int n, int k, int32_t* __restrict__ out_idx,
                                  float* __restrict__ out_val, uint32_t* hist, int* s_tmp, int* lists,
                                  int list_cap) {
  constexpr int kTopkThreads = TPB, kTopkWarps = TPB / 32;
  const int tid = threadIdx.x, w = warp_id();
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  __shared__ int s_sel[2];
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const int n4 = n / 4;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    uint32_t* wh = hist + w * 256;
    for (int b0 = 0; b0 < n4; b0 += kTopkThreads * kUnroll) {
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i4 = b0 + u * kTopkThreads + tid;
        v[u] = i4 < n4 ? __ldg(g4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const bool in = b0 + u * kTopkThreads + tid < n4;
        hist_add(wh, ordered_key(v[u].x), in, prefix, mask, shift);
        hist_add(wh, ordered_key(v[u].y), in, prefix, mask, shift);
        hist_add(wh, ordered_key(v[u].z), in, prefix, mask, shift);
        hist_add(wh, ordered_key(v[u].w), in, prefix, mask, shift);
      }
    }
    if (w == 0) {
      // the < 4 tail elements (rows are not always a multiple of 4 long)
      const int i = n4 * 4 + (tid & 31);
      const bool in = i < n;
      hist_add(wh, in ? ordered_key(__ldg(g + i)) : 0u, in, prefix, mask, shift);
    }
    __syncthreads();
    pick_digit<TPB>(hist, shift, prefix, mask, remaining, s_sel);
  }
  const uint32_t kstar = prefix;
  const int need_eq = remaining;
  const int n_gt = k - need_eq;
  // unordered collection of the winners
  int* s_cnt = s_tmp + 68;  // [0] greater, [1] equal
  int* gt_list = lists;                  // list_cap entries
  int* eq_list = lists + list_cap;       // list_cap entries
  if (tid == 0) {
    s_cnt[0] = 0;
    s_cnt[1] = 0;
  }
  __syncthreads();
  const uint32_t lt = (1u << (tid & 31)) - 1u;
  for (int b0 = 0; b0 < n; b0 += kTopkThreads * 4) {
    float vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = b0 + u * kTopkThreads + tid;
      vv[u] = i < n ? __ldg(g + i) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = b0 + u * kTopkThreads + tid;
      const uint32_t key = ordered_key(vv[u]);
      const bool in = i < n;
      const bool is_gt = in && key > kstar, is_eq = in && key == kstar;
      const uint32_t gb = __ballot_sync(0xffffffffu, is_gt), eb = __ballot_sync(0xffffffffu, is_eq);
      int gbase = 0, ebase = 0;
      if ((tid & 31) == 0) {
        if (gb) gbase = atomicAdd(&s_cnt[0], __popc(gb));
        if (eb) ebase = atomicAdd(&s_cnt[1], __popc(eb));
      }
      gbase = __shfl_sync(0xffffffffu, gbase, 0);
      ebase = __shfl_sync(0xffffffffu, ebase, 0);
      if (is_gt) {
        // a selection larger than the list is emitted in order below instead
        const int pos = gbase + __popc(gb & lt);
        if (pos < list_cap) gt_list[pos] = i;
      }
      if (is_eq) {
        const int pos = ebase + __popc(eb & lt);
        if (pos < list_cap) eq_list[pos] = i;
      }
    }
  }
  __syncthreads();
  const int neq = s_cnt[1];
  if (neq > list_cap || k > list_cap) {
    // too many winners or ties to collect (the lists stopped at list_cap
    // entries): ordered emission straight from global memory
    emit_ordered<false, TPB>(g, nullptr, n, kstar, need_eq, out_idx, out_val, s_tmp);
    return;
  }
  // lowest-index need_eq ties: sort the tie list, then the k winners
  int p2 = 1;
  while (p2 < neq) p2 <<= 1;
  for (int i = neq + tid; i < p2; i += kTopkThreads) eq_list[i] = 0x7fffffff;
  __syncthreads();
  bitonic_sort_smem(eq_list, p2);
  for (int i = tid; i < need_eq; i += kTopkThreads) gt_list[n_gt + i] = eq_list[i];
  int q2 = 1;
  while (q2 < k) q2 <<= 1;
  for (int i = k + tid; i < q2; i += kTopkThreads) gt_list[i] = 0x7fffffff;
  __syncthreads();
  bitonic_sort_smem(gt_list, q2);
  for (int i = tid; i < k; i += kTopkThreads) {
    const int idx = gt_list[i];
    out_idx[i] = idx;
    if (out_val) out_val[i] = __ldg(g + idx);
  }
}

// The key of rank `rank` (1 = largest) among m ordered keys in shared
// memory, by a most-significant-digit radix select; `remaining` returns how
// many copies of that key belong to the top `rank`. Digits above the first
// bit in which the keys differ are skipped (a candidate list near the top of
// a row shares its leading digits, and a pass over one shared digit would
// send every atomic of a warp to one bin). With last_pass < 3 the select
// stops after that digit and returns the lower bound of the bin that holds
// the rank-`rank` key (at most that key). Block-wide.
template <int TPB>
__device__ uint32_t rank_key(const uint32_t* __restrict__ keys, int m, int rank, uint32_t* hist, int& remaining,
                             int last_pass = 3) {
  constexpr int W = TPB / 32;
  __shared__ int s_sel[2];
  __shared__ uint32_t s_ao[2][W];
  const int tid = threadIdx.x, w = warp_id(), lane = lane_id();
  uint32_t a = 0xffffffffu, o = 0u;
  for (int i = tid; i < m; i += TPB) {
    a &= keys[i];
    o |= keys[i];
  }
  a = __reduce_and_sync(0xffffffffu, a);
  o = __reduce_or_sync(0xffffffffu, o);
  if (lane == 0) {
    s_ao[0][w] = a;
    s_ao[1][w] = o;
  }
  __syncthreads();
  a = 0xffffffffu;
  o = 0u;
#pragma unroll
  for (int ww = 0; ww < W; ++ww) {
    a &= s_ao[0][ww];
    o |= s_ao[1][ww];
  }
  remaining = rank;
  const uint32_t diff = a ^ o;
  if (diff == 0u) return a;  // every key is equal (m > 0)
  const int first = __clz(diff) >> 3;  // the first digit in which keys differ
  uint32_t mask = first ? ~0u << (32 - 8 * first) : 0u;
  uint32_t prefix = a & mask;
  const int mround = (m + TPB - 1) / TPB * TPB;
  for (int pass = first; pass <= last_pass; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < W * 256; i += TPB) hist[i] = 0;
    __syncthreads();
    uint32_t* wh = hist + w * 256;
    for (int i = tid; i < mround; i += TPB) hist_add(wh, i < m ? keys[i] : 0u, i < m, prefix, mask, shift);
    __syncthreads();
    pick_digit<TPB>(hist, shift, prefix, mask, remaining, s_sel);
  }
  return prefix;
}

// Exact top-k of a row from a candidate list in shared memory (ordered keys
// ckey and row positions cidx, ascending in position) that holds every
// winner: the rank-k key, then the ordered emission over the list.
template <int TPB>
__device__ void select_candidates(const float* __restrict__ g, const uint32_t* __restrict__ ckey,
                                  const int* __restrict__ cidx, int m, int k, int32_t* __restrict__ out_idx,
                                  float* __restrict__ out_val, uint32_t* hist, int* s_tmp) {
  int remaining;
  const uint32_t kstar = rank_key<TPB>(ckey, m, k, hist, remaining);
  emit_ordered<true, TPB>(g, ckey, m, kstar, remaining, out_idx, out_val, s_tmp, cidx);
}

// Row longer than shared memory, in two reads of the row instead of one per
// radix digit:
//  A. every warp histograms the top kWideBits bits of the keys of its own
//     contiguous segment of the row (a 2048-bin histogram per warp); the sums
//     give the bin b* that holds the rank-k key;
//  B. every warp copies, in position order, the keys of its segment whose top
//     bits are >= b* (exactly the candidates: every winner, plus the rest of
//     bin b*) into a shared-memory list; the per-warp histograms give each
//     warp its offset, so the list is in ascending position order;
//  C. the exact radix select and the ordered emission run on that list.
// Returns false (before writing anything) when the candidates would not fit;
// the caller then takes the multi-pass path.
constexpr int kWideBits = 11;
constexpr int kWideBins = 1 << kWideBits;
constexpr int kWideShift = 32 - kWideBits;
// The staging area of a TPB-thread block holds (TPB / 32) * kWideBins keys:
// exactly the per-warp wide histograms, and then the candidate list (keys and
// positions) of half as many entries.
template <int TPB>
__host__ __device__ constexpr int stage_cap() { return TPB / 32 * kWideBins; }

template <int TPB>
__device__ bool select_row_two_pass(const float* __restrict__ g, int n, int k, int32_t* __restrict__ out_idx,
                                    float* __restrict__ out_val, uint32_t* hist, uint32_t* area, int* s_tmp) {
  constexpr int kTopkThreads = TPB, kTopkWarps = TPB / 32;
  constexpr int kCandCap = stage_cap<TPB>() / 2;
  constexpr int BPT = kWideBins / TPB;  // wide bins per thread in the scan
  const int tid = threadIdx.x, w = warp_id(), lane = lane_id();
  __shared__ int s_sel[2];
  __shared__ int s_woff[kTopkWarps + 1];
  uint32_t* whist = area + w * kWideBins;  // [kTopkWarps][kWideBins] over the staging area
  for (int i = tid; i < kTopkWarps * kWideBins; i += kTopkThreads) area[i] = 0;
  __syncthreads();
  // segments of whole float4 groups (rows start 16-byte aligned)
  const int n4 = (n + 3) / 4;
  const int seg4 = (n4 + kTopkWarps - 1) / kTopkWarps;
  const int s0 = min(n4, w * seg4), s1 = min(n4, s0 + seg4);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  constexpr int U = 8;  // float4 loads in flight per lane
  // ---- A
  for (int b = s0; b < s1; b += 32 * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = b + u * 32 + lane;
      v[u] = i4 < s1 ? __ldg(g4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = 4 * (b + u * 32 + lane);
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (i + c < n && i < 4 * s1) atomicAdd(whist + (ordered_key(e[c]) >> kWideShift), 1u);
    }
  }
  __syncthreads();
  // bin totals, scanned from the top bin down: thread tid owns bins
  // 2047 - BPT*tid .. 2048 - BPT*(tid + 1)
  uint32_t cnt[BPT], tot = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int bin = kWideBins - 1 - (BPT * tid + j);
    uint32_t c = 0;
#pragma unroll 4
    for (int ww = 0; ww < kTopkWarps; ++ww) c += area[ww * kWideBins + bin];
    cnt[j] = c;
    tot += c;
  }
  // block-wide exclusive scan of the per-thread totals
  uint32_t x = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[w] = (int)x;
  __syncthreads();
  if (w == 0) {
    uint32_t y = lane < kTopkWarps ? (uint32_t)s_tmp[lane] : 0u;
    const uint32_t orig = y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    if (lane < kTopkWarps) s_tmp[32 + lane] = (int)(y - orig);
  }
  __syncthreads();
  uint32_t above = (uint32_t)s_tmp[32 + w] + (x - tot);  // keys in bins above this thread's first bin
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    if (above < (uint32_t)k && above + cnt[j] >= (uint32_t)k) {
      s_sel[0] = kWideBins - 1 - (BPT * tid + j);
      s_sel[1] = (int)(above + cnt[j]);  // candidates: keys in bins >= b*
    }
    above += cnt[j];
  }
  __syncthreads();
  const int bstar = s_sel[0];
  const int m = s_sel[1];
  if (m > kCandCap) return false;  // uniform over the block
  // per-warp candidate counts (suffix sums of the warp's own histogram) and offsets
  uint32_t mine = 0;
  for (int bin = bstar + lane; bin < kWideBins; bin += 32) mine += whist[bin];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_woff[w] = (int)mine;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int ww = 0; ww < kTopkWarps; ++ww) {
      const int c = s_woff[ww];
      s_woff[ww] = acc;
      acc += c;
    }
    s_woff[kTopkWarps] = acc;
  }
  __syncthreads();  // the histograms are dead from here on: the area holds the list
  uint32_t* ckey = area;
  int* cidx = reinterpret_cast<int*>(area + kCandCap);
  // ---- B: ordered compaction of this warp's segment
  int run = s_woff[w];
  for (int b = s0; b < s1; b += 32 * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = b + u * 32 + lane;
      v[u] = i4 < s1 ? __ldg(g4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = 4 * (b + u * 32 + lane);
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t key[4];
      int c = 0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        key[cc] = ordered_key(e[cc]);
        const bool in = i + cc < n && i < 4 * s1 && (int)(key[cc] >> kWideShift) >= bstar;
        c += in ? 1 : 0;
      }
      // lanes hold consecutive groups of four positions: an exclusive scan of
      // the per-lane counts keeps the list in position order
      int xs = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
      }
      int pos = run + xs - c;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const bool in = i + cc < n && i < 4 * s1 && (int)(key[cc] >> kWideShift) >= bstar;
        if (in) {
          ckey[pos] = key[cc];
          cidx[pos] = i + cc;
          ++pos;
        }
      }
      run += __shfl_sync(0xffffffffu, xs, 31);
    }
  }
  __syncthreads();
  // ---- C
  select_candidates<TPB>(g, ckey, cidx, m, k, out_idx, out_val, hist, s_tmp);
  return true;
}

// Row longer than shared memory, in one read: a threshold t0 from a strided
// sample of the row bounds the candidates.
//  A. kSample keys at evenly spaced positions; r is chosen so that about
//     min(2k, (k + capacity) / 2) keys of the row are expected at or above
//     the sample's key of rank r, and t0 is the lower bound of that key's
//     16-bit bin (so a little below it);
//  B. one pass over the row in block-wide chunks copies every key >= t0,
//     in position order, into the candidate list (per chunk, each warp takes
//     a contiguous run; a scan over the warps gives the offsets);
//  C. if at least k keys were copied, the k-th largest key is >= t0, so the
//     list holds every winner: exact select and ordered emission on it.
// Returns false (before writing anything) when fewer than k or more than the
// list capacity were found (massive ties, unusual score distributions); the
// caller then takes the two-pass path.
constexpr int kSample = 1024;
constexpr int kAhead = 2;  // chunks of the row prefetched into L2 ahead of the pass

template <int TPB>
__device__ bool select_row_sampled(const float* __restrict__ g, int n, int k, int32_t* __restrict__ out_idx,
                                   float* __restrict__ out_val, uint32_t* hist, uint32_t* area, int* s_tmp) {
  constexpr int W = TPB / 32;
  constexpr int kCandCap = stage_cap<TPB>() / 2;
  static_assert(kSample <= kCandCap, "the sample fits the candidate list");
  if (2 * k > kCandCap) return false;  // a list of (k + cap) / 2 expected entries would crowd the cap
  const int tid = threadIdx.x, w = warp_id(), lane = lane_id();
  __shared__ int s_wcnt[2][W];
  const int n4 = (n + 3) / 4;
  const float4* g4 = reinterpret_cast<const float4*>(g);
  constexpr int U = 4;                  // float4 groups per lane per chunk
  constexpr int kChunk4 = TPB * U;      // float4 groups per chunk
  // the first chunks of the row start their way into L2 under the sample
  // (one 128-byte line per prefetch, kAhead chunks ahead of the pass)
  auto prefetch_chunk = [&](int c0) {
    for (int l = tid; l < kChunk4 / 8; l += TPB) {
      const int i4 = c0 + 8 * l;
      if (i4 < n4) prefetch_l2(g4 + i4);
    }
  };
#pragma unroll 1
  for (int c = 0; c < kAhead; ++c) prefetch_chunk(c * kChunk4);
  // ---- A
  uint32_t* skey = area;
  for (int j = tid; j < kSample; j += TPB) skey[j] = ordered_key(__ldg(g + (int)(((long long)j * n) / kSample)));
  __syncthreads();
  const long long target = min(2LL * k, (long long)(k + kCandCap) / 2);
  const int r = (int)max(1LL, min((long long)kSample, (target * kSample + n / 2) / n));
  int rem_unused;
  // two digits resolve t0 to its 16-bit bin (sign, exponent and seven
  // mantissa bits): t0 is that bin's lower bound, a little below the sample's
  // rank-r key, which only adds the keys within the bin
  const uint32_t t0 = rank_key<TPB>(skey, kSample, r, hist, rem_unused, 1);
  __syncthreads();  // the sample is dead: the area holds the list
  uint32_t* ckey = area;
  int* cidx = reinterpret_cast<int*>(area + kCandCap);
  // ---- B
  int run = 0;                          // candidates before this chunk (block-uniform)
  float4 v[U];
  auto load = [&](int c0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = c0 + w * 32 * U + u * 32 + lane;
      v[u] = i4 < n4 ? __ldg(g4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
  };
  load(0);
  for (int c0 = 0, par = 0; c0 < n4; c0 += kChunk4, par ^= 1) {
    uint32_t fl[U];  // per group: bit cc set when position 4*i4 + cc is a candidate
    uint32_t key[U][4];
    int wtot = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = 4 * (c0 + w * 32 * U + u * 32 + lane);
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      fl[u] = 0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        key[u][cc] = ordered_key(e[cc]);
        if (i + cc < n && key[u][cc] >= t0) fl[u] |= 1u << cc;
      }
      wtot += __popc(fl[u]);
    }
    if (c0 + kChunk4 < n4) load(c0 + kChunk4);  // the next chunk's loads fly during the scans
    prefetch_chunk(c0 + kAhead * kChunk4);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wtot += __shfl_xor_sync(0xffffffffu, wtot, o);
    if (lane == 0) s_wcnt[par][w] = wtot;
    __syncthreads();
    int woff = run, ctot = 0;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) {
      const int c = s_wcnt[par][ww];
      woff += ww < w ? c : 0;
      ctot += c;
    }
    // lanes hold consecutive groups of four positions: an exclusive scan of
    // the per-lane counts keeps the list in position order
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = __popc(fl[u]);
      int xs = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
      }
      int pos = woff + xs - c;
      const int i = 4 * (c0 + w * 32 * U + u * 32 + lane);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        if ((fl[u] >> cc) & 1u) {
          if (pos < kCandCap) {
            ckey[pos] = key[u][cc];
            cidx[pos] = i + cc;
          }
          ++pos;
        }
      }
      woff += __shfl_sync(0xffffffffu, xs, 31);
    }
    run += ctot;
    // s_wcnt alternates between two buffers: the next chunk's counts never
    // overwrite ones a slower warp is still reading
  }
  __syncthreads();
  if (run < k || run > kCandCap) return false;  // uniform over the block
  // ---- C
  select_candidates<TPB>(g, ckey, cidx, run, k, out_idx, out_val, hist, s_tmp);
  return true;
}

// Row staged in shared memory as ordered keys; the histograms of the first
// pass (top digit) were counted while staging.
template <int TPB>
__device__ void select_row_staged(const float* __restrict__ g, const uint32_t* __restrict__ s_row, int n, int k,
                                  int32_t* __restrict__ out_idx, float* __restrict__ out_val, uint32_t* hist,
                                  int* s_tmp) {
  constexpr int W = TPB / 32;
  const int tid = threadIdx.x, w = warp_id();
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  __shared__ int s_sel[2];
  const int nround = (n + TPB - 1) / TPB * TPB;
  pick_digit<TPB>(hist, 24, prefix, mask, remaining, s_sel);
  for (int pass = 1; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < W * 256; i += TPB) hist[i] = 0;
    __syncthreads();
    uint32_t* wh = hist + w * 256;
    for (int i = tid; i < nround; i += TPB) hist_add(wh, i < n ? s_row[i] : 0u, i < n, prefix, mask, shift);
    __syncthreads();
    pick_digit<TPB>(hist, shift, prefix, mask, remaining, s_sel);
  }
  emit_ordered<true, TPB>(g, s_row, n, prefix, remaining, out_idx, out_val, s_tmp);
}

// TPB threads per row: kTopkThreads (a few rows longer than 2048: the
// shortest per-row time), kTopkThreadsMany (many such rows: three resident
// per SM instead of one) or kTopkThreadsShort (rows of at most 2048 keys)
template <int TPB>
__global__ void __launch_bounds__(TPB, TPB == kTopkThreadsMany ? 3 : 1)
    topk_rows_kernel(const float* __restrict__ scores, long long ld, const int* __restrict__ nvis, int div, int k,
                     int32_t* __restrict__ out_idx, float* __restrict__ out_val, int cap, int fold) {
  constexpr int W = TPB / 32;
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_tmp[72];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);  // (warps + 1) * 256
  uint32_t* s_row = hist + (W + 1) * 256;               // cap keys
  const int row = blockIdx.x;
  const int nraw = nvis[row];
  int n = nraw;
  if (div > 1) n = (n + div - 1) / div;
  const float* g = scores + (size_t)row * ld;
  int32_t* oi = out_idx + (size_t)row * k;
  float* ov = out_val ? out_val + (size_t)row * k : nullptr;
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
      oi[i] = i < n ? i : -1;
      if (ov) ov[i] = i < n ? __ldg(g + i) : -INFINITY;
    }
    return;
  }
  if (n <= cap) {
    // stage with many independent loads in flight, counting the top digit of
    // every key on the way (the first radix pass)
    for (int i = threadIdx.x; i < W * 256; i += TPB) hist[i] = 0;
    __syncthreads();
    uint32_t* wh = hist + warp_id() * 256;
    for (int b0 = 0; b0 < n; b0 += TPB * 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = b0 + u * TPB + threadIdx.x;
        v[u] = i >= n ? 0.f : fold == 1 ? __ldg(g + i) : fold_max(g, i, fold, nraw);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = b0 + u * TPB + threadIdx.x;
        if (i < n) {
          const uint32_t key = ordered_key(v[u]);
          s_row[i] = key;
          atomicAdd(wh + (key >> 24), 1u);
        }
      }
    }
    __syncthreads();
    select_row_staged<TPB>(g, s_row, n, k, oi, ov, hist, s_tmp);
  } else if constexpr (TPB != kTopkThreadsShort) {
    if (cap < stage_cap<TPB>() || (!select_row_sampled<TPB>(g, n, k, oi, ov, hist, s_row, s_tmp) &&
                                   !select_row_two_pass<TPB>(g, n, k, oi, ov, hist, s_row, s_tmp)))
      select_row_global<TPB>(g, n, k, oi, ov, hist, s_tmp, reinterpret_cast<int*>(s_row), cap / 2);
  }
  // (the short-row instantiation is only launched when every row fits cap)
}

// The block size for a launch: rows of at most 2048 keys take 128-thread
// blocks (six rows per SM, cheap block barriers); launches with many longer
// rows take 256-thread blocks (three rows per SM); a few longer rows keep
// the 512-thread block, the shortest time per row (measured: 32 rows of 4-8 K
// keys took 61 us with short blocks, 41 us wide; 8192 causal rows of up to
// 8192 keys 0.545 ms with short blocks, 0.530 with 256-thread ones).
static int topk_tier(int T, int max_len) {
  if (max_len <= 2048) return kTopkThreadsShort;
  return T >= 2 * sm_count() ? kTopkThreadsMany : kTopkThreads;
}

static int topk_stage_cap(int tpb) {
  return tpb == kTopkThreadsShort ? stage_cap<kTopkThreadsShort>()
         : tpb == kTopkThreadsMany ? stage_cap<kTopkThreadsMany>() : stage_cap<kTopkThreads>();
}

static int launch_topk(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int div, int k,
                       int32_t* out_idx, float* out_val, int max_len, int fold) {
  if (T == 0) return DSA_OK;
  // rows longer than the staging capacity are read as float4: every row must
  // start 16-byte aligned
  if ((ld & 3) || (reinterpret_cast<uintptr_t>(scores) & 15)) return DSA_ERR_ALIGNMENT;
  // rows longer than the staging capacity use the staging area as two
  // winner lists of cap/2 entries each; the staging capacity of a block size
  // is its wide-histogram area (stage_cap)
  auto launch = [&](auto tpb_c) -> int {
    constexpr int TPB = decltype(tpb_c)::value;
    constexpr int W = TPB / 32;
    const int cap = max_len > stage_cap<TPB>() ? stage_cap<TPB>() : max(0, max_len);
    const size_t smem = (size_t)(W + 1) * 256 * 4 + (size_t)cap * 4;
    set_smem_attr_once(reinterpret_cast<const void*>(topk_rows_kernel<TPB>),
                       (W + 1) * 256 * 4 + stage_cap<TPB>() * 4);
    DSA_LAUNCH_PDL(topk_rows_kernel<TPB>, dim3(T), dim3(TPB), smem, stream, scores, ld, nvis, div, k, out_idx,
                   out_val, cap, fold);
    return DSA_OK;
  };
  const int tier = topk_tier(T, max_len);
  if (tier == kTopkThreadsShort) return launch(std::integral_constant<int, kTopkThreadsShort>{});
  if (tier == kTopkThreadsMany) return launch(std::integral_constant<int, kTopkThreadsMany>{});
  return launch(std::integral_constant<int, kTopkThreads>{});
}

int run_topk(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int div, int k,
             int32_t* out_idx, float* out_val, int max_len) {
  return launch_topk(stream, scores, ld, nvis, T, div, k, out_idx, out_val, max_len, 1);
}

// page maxima from granule maxima, for page rows longer than a stage
__global__ void fold_pages_kernel(const float* __restrict__ gran, long long ld_gr, const int* __restrict__ nvis, int T,
                                  int ps, float* __restrict__ pages, long long ld_pg, int max_pages) {
  griddep_launch_dependents();
  griddep_wait();
  const int fold = ps / 32;
  const long long total = (long long)T * max_pages;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / max_pages), i = (int)(e % max_pages);
    const int nraw = nvis[t];
    if ((long long)i * ps < nraw) pages[(size_t)t * ld_pg + i] = fold_max(gran + (size_t)t * ld_gr, i, fold, nraw);
  }
}

int run_page_topk(cudaStream_t stream, const float* gran, long long ld_gr, const int* nvis, int T, int ps, int k_pages,
                  int32_t* out_idx, float* page_buf, long long ld_pg, int max_pages) {
  if (T == 0) return DSA_OK;
  const int fold = ps / 32;
  if (fold == 1) return launch_topk(stream, gran, ld_gr, nvis, T, ps, k_pages, out_idx, nullptr, max_pages, 1);
  // staged rows fold their granules while they are staged; longer rows take
  // a folding pass first
  if (max_pages <= topk_stage_cap(topk_tier(T, max_pages)))
    return launch_topk(stream, gran, ld_gr, nvis, T, ps, k_pages, out_idx, nullptr, max_pages, fold);
  if ((ld_gr & 3) || (reinterpret_cast<uintptr_t>(gran) & 15)) return DSA_ERR_ALIGNMENT;
  const long long total = (long long)T * max_pages;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 8LL * sm_count());
  DSA_LAUNCH_PDL(fold_pages_kernel, dim3(blocks), dim3(256), 0, stream, gran, ld_gr, nvis, T, ps, page_buf, ld_pg,
                 max_pages);
  return launch_topk(stream, page_buf, ld_pg, nvis, T, ps, k_pages, out_idx, nullptr, max_pages, 1);
}

}  // namespace dsa
