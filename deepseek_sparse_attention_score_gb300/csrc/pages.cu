// Token top-k -> page list (dsa_sparse_backend.py, compute_topk_pages, used
// by its page-level decode): per query, the ascending unique pages
// (position / ps) of its selected tokens, the first `cap` of them, -1 padded.
//
// One CTA per query row. The row's pages are marked in a shared-memory
// bitmap over the request's pages; a block scan of per-word popcounts then
// gives every set page its output slot, so the list comes out sorted without
// a sort, whatever the order of the token row.
#include "common.cuh"

namespace dsa {

namespace {
constexpr int kPgThreads = 256;
constexpr int kPgWarps = kPgThreads / 32;

__global__ void __launch_bounds__(kPgThreads) topk_pages_kernel(const int32_t* __restrict__ topk, int K, int ps,
                                                                int max_pages, int cap, int32_t* __restrict__ pages,
                                                                int32_t* __restrict__ counts, int32_t* dev_status) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ uint32_t bm[];
  __shared__ int s_warp[kPgWarps + 1];
  const int row = blockIdx.x, tid = threadIdx.x, lane = lane_id(), w = warp_id();
  const int words = (max_pages + 31) / 32;
  for (int i = tid; i < words; i += kPgThreads) bm[i] = 0u;
  __syncthreads();
  const int32_t* src = topk + (size_t)row * K;
  bool bad = false;
  for (int i = tid; i < K; i += kPgThreads) {
    const int j = __ldg(src + i);
    if (j < 0) continue;
    const int p = j / ps;
    if (p >= max_pages) {
      bad = true;
      continue;
    }
    atomicOr(bm + (p >> 5), 1u << (p & 31));
  }
  if (bad) set_status(dev_status, DSA_STATUS_BAD_INDEX);
  __syncthreads();
  // each thread owns a contiguous run of bitmap words
  const int per = (words + kPgThreads - 1) / kPgThreads;
  const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
  int mine = 0;
  for (int i = w0; i < w1; ++i) mine += __popc(bm[i]);
  int x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int k = 0; k < kPgWarps; ++k) {
      const int v = s_warp[k];
      s_warp[k] = acc;
      acc += v;
    }
    s_warp[kPgWarps] = acc;
  }
  __syncthreads();
  int slot = s_warp[w] + x - mine;
  const int total = s_warp[kPgWarps];
  int32_t* out = pages + (size_t)row * cap;
  for (int i = w0; i < w1 && slot < cap; ++i) {
    uint32_t b = bm[i];
    while (b && slot < cap) {
      const int bit = __ffs(b) - 1;
      b &= b - 1u;
      out[slot++] = i * 32 + bit;
    }
  }
  for (int i = total + tid; i < cap; i += kPgThreads) out[i] = -1;
  if (tid == 0 && counts) counts[row] = total;
}
}  // namespace

constexpr int kTopkPagesMaxPages = 1 << 20;  // 128 KB of bitmap
size_t topk_pages_smem(int max_pages) { return (size_t)((max_pages + 31) / 32) * 4; }

int topk_pages_max_pages() { return kTopkPagesMaxPages; }

int run_topk_pages(cudaStream_t stream, const int32_t* topk, int T, int K, int ps, int max_pages, int cap,
                   int32_t* pages, int32_t* counts, int32_t* dev_status) {
  if (T == 0) return DSA_OK;
  const size_t smem = topk_pages_smem(max_pages);
  set_smem_attr_once(reinterpret_cast<const void*>(topk_pages_kernel), (int)topk_pages_smem(kTopkPagesMaxPages));
  DSA_LAUNCH_PDL(topk_pages_kernel, dim3(T), dim3(kPgThreads), smem, stream, topk, K, ps, max_pages, cap, pages,
                 counts, dev_status);
  return DSA_OK;
}

}  // namespace dsa
