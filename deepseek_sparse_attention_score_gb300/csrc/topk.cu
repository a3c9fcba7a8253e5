// Exact per-row top-k (ref.py, streamindex_topk_ref / streamindex_page_topk_ref
// with exact selection): the k largest of a row's visible scores, ties to the
// lower index, written in ascending index order and -1 padded.
//
// One CTA per row. A 4-pass most-significant-digit radix select (8-bit
// digits, per-warp shared-memory histograms) finds the exact k-th largest key
// K* and how many copies of K* are needed; a final pass of warp ballots and
// two block scans emits every index with key > K* plus the lowest-index
// copies of K*, already in ascending order. Rows that fit are first staged in
// shared memory; longer rows are re-read from global memory (L2) per pass.
#include "common.cuh"
#include "indexer.cuh"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkSmemCap = 32768;  // row elements staged in shared memory

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 and +0
// map to the same key so they tie like equal scores.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ int block_scan_warps(int v, int* s_tmp, int* total) {
  // exclusive scan of one value per warp (lane 0 holds it) across the block
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

template <bool kStaged>
__device__ void select_row(const float* __restrict__ g, const uint32_t* __restrict__ s_row, int n, int k,
                           int32_t* __restrict__ out_idx, float* __restrict__ out_val, uint32_t* hist,
                           int* s_tmp) {
  const int tid = threadIdx.x, w = warp_id(), lane = lane_id();
  auto key_at = [&](int i) -> uint32_t { return kStaged ? s_row[i] : ordered_key(__ldg(g + i)); };
  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // rank (1-based) of the wanted key among keys matching prefix
  __shared__ int s_sel[2];
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    uint32_t* wh = hist + w * 256;
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(wh + ((key >> shift) & 255u), 1u);
    }
    __syncthreads();
    // reduce the per-warp histograms into hist[0..255] and pick the digit
    if (tid < 256) {
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < kTopkWarps; ++j) c += hist[j * 256 + tid];
      hist[kTopkWarps * 256 + tid] = c;
    }
    __syncthreads();
    if (w == 0) {
      // suffix sums from the top digit down, 8 digits per lane
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
  const uint32_t kstar = prefix;
  const int need_eq = remaining;  // copies of K* to take, lowest index first
  // warp w owns the contiguous segment [seg0, seg1)
  const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int seg0 = min(n, w * seg), seg1 = min(n, seg0 + seg);
  int gt = 0, eq = 0;
  for (int i = seg0 + lane; i < seg1 + ((32 - (seg1 - seg0) % 32) % 32); i += 32) {
    const bool in = i < seg1;
    const uint32_t key = in ? key_at(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, in && key > kstar));
    eq += __popc(__ballot_sync(0xffffffffu, in && key == kstar));
  }
  int tot;
  const int eq_base = block_scan_warps(eq, s_tmp, &tot);
  const int take_eq = max(0, min(need_eq - eq_base, eq));
  const int out_base = block_scan_warps(gt + take_eq, s_tmp, &tot);
  const uint32_t lt = (1u << lane) - 1u;
  int eq_run = eq_base, sel_run = out_base;
  for (int i = seg0 + lane; i < seg1 + ((32 - (seg1 - seg0) % 32) % 32); i += 32) {
    const bool in = i < seg1;
    const uint32_t key = in ? key_at(i) : 0u;
    const bool is_gt = in && key > kstar, is_eq = in && key == kstar;
    const uint32_t eqb = __ballot_sync(0xffffffffu, is_eq);
    const int my_eq_rank = eq_run + __popc(eqb & lt);
    const bool sel = is_gt || (is_eq && my_eq_rank < need_eq);
    const uint32_t selb = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int pos = sel_run + __popc(selb & lt);
      out_idx[pos] = i;
      if (out_val) out_val[pos] = kStaged ? __ldg(g + i) : __ldg(g + i);
    }
    eq_run += __popc(eqb);
    sel_run += __popc(selb);
  }
  // k <= n here, so exactly k entries were written
}

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const float* __restrict__ scores, long long ld,
                                                                 const int* __restrict__ nvis, int div, int k,
                                                                 int32_t* __restrict__ out_idx,
                                                                 float* __restrict__ out_val, int cap) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_tmp[72];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);                  // (warps + 1) * 256
  uint32_t* s_row = hist + (kTopkWarps + 1) * 256;                      // cap keys
  const int row = blockIdx.x;
  int n = nvis[row];
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
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_row[i] = ordered_key(__ldg(g + i));
    __syncthreads();
    select_row<true>(g, s_row, n, k, oi, ov, hist, s_tmp);
  } else {
    select_row<false>(g, s_row, n, k, oi, ov, hist, s_tmp);
  }
}

int run_topk(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int div, int k,
             int32_t* out_idx, float* out_val, int max_len) {
  if (T == 0) return DSA_OK;
  const int cap = max(0, min(max_len, kTopkSmemCap));
  const size_t smem = (size_t)(kTopkWarps + 1) * 256 * 4 + (size_t)cap * 4;
  cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  topk_rows_kernel<<<T, kTopkThreads, smem, stream>>>(scores, ld, nvis, div, k, out_idx, out_val, cap);
  DSA_CHECK_LAUNCH();
  return DSA_OK;
}

}  // namespace dsa
