// Shared internals of the DSA library: status reporting, ragged-metadata
// lookups done on the device, and host launch helpers.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>

#include "../../include/dsa.h"
#include "ptx.cuh"

namespace dsa {

__device__ __forceinline__ void set_status(int32_t* dev_status, int bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// Request of query token t: the s with cu_q_lens[s] <= t < cu_q_lens[s+1]
// (binary search; empty requests are skipped naturally).
__device__ __forceinline__ int seq_of_token(const int32_t* cu_q_lens, int S, int t) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_q_lens + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Per-token geometry derived from the ragged metadata.
struct TokenGeom {
  int seq;       // request id
  int pos;       // absolute position of the query token
  int kv_len;    // seq_lens[seq], clamped to [0, max_kv]
  int n_vis;     // visible prefix length: min(kv_len, pos + 1), >= 0
  int page_base; // first packed page-table entry of the request
};

__device__ __forceinline__ TokenGeom token_geom(const int32_t* seq_lens, const int32_t* cu_q_lens,
                                                const int32_t* cu_kv_lens, int S, int ps, int max_kv, int t,
                                                int32_t* dev_status) {
  TokenGeom g;
  g.seq = seq_of_token(cu_q_lens, S, t);
  const int q0 = __ldg(cu_q_lens + g.seq), q1 = __ldg(cu_q_lens + g.seq + 1);
  int kv = __ldg(seq_lens + g.seq);
  if (kv < 0 || kv > max_kv || kv < q1 - q0) {
    set_status(dev_status, DSA_STATUS_BAD_METADATA);
    kv = kv < 0 ? 0 : (kv > max_kv ? max_kv : kv);
  }
  g.kv_len = kv;
  g.pos = kv - (q1 - q0) + (t - q0);
  int nv = g.pos + 1 < kv ? g.pos + 1 : kv;
  g.n_vis = nv < 0 ? 0 : nv;
  g.page_base = __ldg(cu_kv_lens + g.seq) / ps;
  return g;
}

}  // namespace dsa

namespace dsa {
void note_launch();  // process-wide count of enqueued kernels
}
// Host-side launch check: turns a launch error into DSA_ERR_CUDA and counts
// the launch.
#define DSA_CHECK_LAUNCH()                              \
  do {                                                  \
    if (cudaPeekAtLastError() != cudaSuccess) {         \
      (void)cudaGetLastError();                         \
      return DSA_ERR_CUDA;                              \
    }                                                   \
    ::dsa::note_launch();                               \
  } while (0)

namespace dsa {
int sm_count();  // cached per device
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace dsa
