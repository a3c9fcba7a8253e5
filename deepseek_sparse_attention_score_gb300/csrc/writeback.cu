// Paged write-back of the new tokens' rows (dsa_sparse_backend.py,
// _scatter_paged; sparse_mla_prefill_qblock.py, paged_write_back): query
// token t of request s sits at absolute position
// pos = seq_lens[s] - q_len(s) + (t - cu_q_lens[s]), and its row goes to
// row pos % ps of physical page page_indices[cu_kv_lens[s] / ps + pos / ps].
//
// One warp per token: the request lookup is a warp-wide search over
// cu_q_lens and the row is copied as 16-byte chunks, one per lane per step,
// so every warp moves whole contiguous rows (pure HBM streaming; there is no
// reuse to stage through shared memory). Two caches that share the page
// table (a layer's latent rows and its indexer keys) can be written by one
// launch: the slot is found once and both rows are copied.
#include "common.cuh"

namespace dsa {

namespace {
constexpr int kWbThreads = 256;  // 8 tokens per CTA

struct WbTarget {
  const uint16_t* rows;  // [T, src_stride]
  long long src_stride;
  int D;                 // columns copied (0: nothing)
  uint16_t* cache;       // [P, ps, cache_stride]
  long long cache_stride;
};

__device__ __forceinline__ void copy_row(const WbTarget& w, int t, size_t slot, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(w.rows + (size_t)t * w.src_stride);
  uint4* dst = reinterpret_cast<uint4*>(w.cache + slot * w.cache_stride);
  const int n16 = w.D / 8;
  for (int c = lane; c < n16; c += 32) dst[c] = __ldg(src + c);
}

__global__ void __launch_bounds__(kWbThreads) paged_write_back_kernel(
    const WbTarget w0, const WbTarget w1, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q_lens,
    const int32_t* __restrict__ cu_kv_lens, const int32_t* __restrict__ page_indices, int T, int S, int P, int PTW,
    int ps, int32_t* dev_status) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = lane_id();
  const int t = blockIdx.x * (kWbThreads / 32) + warp_id();
  if (t >= T) return;
  const int s = seq_of_token_warp(cu_q_lens, S, t);
  const int q0 = __ldg(cu_q_lens + s), q1 = __ldg(cu_q_lens + s + 1);
  const int kv = __ldg(seq_lens + s);
  const int pos = kv - (q1 - q0) + (t - q0);
  const long long ent = (long long)(__ldg(cu_kv_lens + s) / ps) + pos / ps;
  if (pos < 0 || q1 - q0 > kv || ent < 0 || ent >= PTW) {
    if (lane == 0) set_status(dev_status, DSA_STATUS_BAD_METADATA);
    return;
  }
  const int pg = __ldg(page_indices + ent);
  if (pg < 0 || pg >= P) {
    if (lane == 0) set_status(dev_status, DSA_STATUS_BAD_METADATA);
    return;
  }
  const size_t slot = (size_t)pg * ps + pos % ps;
  copy_row(w0, t, slot, lane);
  if (w1.D) copy_row(w1, t, slot, lane);
}
}  // namespace

int run_paged_write_back(cudaStream_t stream, const uint16_t* rows, long long src_stride, int D, uint16_t* cache,
                         long long cache_stride, const uint16_t* rows1, long long src_stride1, int D1,
                         uint16_t* cache1, long long cache_stride1, const int32_t* seq_lens,
                         const int32_t* cu_q_lens, const int32_t* cu_kv_lens, const int32_t* page_indices, int T,
                         int S, int P, int PTW, int ps, int32_t* dev_status) {
  if (T == 0) return DSA_OK;
  const int per = kWbThreads / 32;
  const WbTarget w0{rows, src_stride, D, cache, cache_stride};
  const WbTarget w1{rows1, src_stride1, rows1 && cache1 ? D1 : 0, cache1, cache_stride1};
  DSA_LAUNCH_PDL(paged_write_back_kernel, dim3((T + per - 1) / per), dim3(kWbThreads), 0, stream, w0, w1, seq_lens,
                 cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps, dev_status);
  return DSA_OK;
}

}  // namespace dsa
