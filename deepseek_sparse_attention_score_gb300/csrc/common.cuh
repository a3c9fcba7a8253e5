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

// Warp-cooperative version of seq_of_token: 32 boundaries per step, so a
// batch of S requests resolves in ceil(log32(S)) dependent loads. All lanes
// must call it with the same t; every lane gets the result.
__device__ __forceinline__ int seq_of_token_warp(const int32_t* cu_q_lens, int S, int t) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = S;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(cu_q_lens + idx) <= t;
    const uint32_t m = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz(m);  // lane 0 always qualifies (cu_q_lens[lo] <= t)
    lo = lo + last * step;
    hi = min(hi, lo + step);
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
                                                int32_t* dev_status, int seq = -1) {
  TokenGeom g;
  g.seq = seq >= 0 ? seq : seq_of_token(cu_q_lens, S, t);
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

// Launch with programmatic stream serialization (the kernel may start while
// the previous kernel of the stream is finishing; it waits for it with
// griddep_wait before touching global memory), turning a launch error into
// DSA_ERR_CUDA and counting the launch.
#define DSA_LAUNCH_PDL(kernel, grid, block, smem, stream, ...)                        \
  do {                                                                                \
    cudaLaunchConfig_t cfg_ = {};                                                     \
    cfg_.gridDim = (grid);                                                            \
    cfg_.blockDim = (block);                                                          \
    cfg_.dynamicSmemBytes = (smem);                                                   \
    cfg_.stream = (stream);                                                           \
    cudaLaunchAttribute attr_[1];                                                     \
    attr_[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                 \
    attr_[0].val.programmaticStreamSerializationAllowed = 1;                          \
    cfg_.attrs = attr_;                                                               \
    cfg_.numAttrs = 1;                                                                \
    if (cudaLaunchKernelEx(&cfg_, kernel, __VA_ARGS__) != cudaSuccess) {              \
      (void)cudaGetLastError();                                                       \
      return DSA_ERR_CUDA;                                                            \
    }                                                                                 \
    ::dsa::note_launch();                                                             \
  } while (0)

namespace dsa {
int sm_count();  // cached per device
// Raise a kernel's dynamic shared-memory limit once per device (not during
// stream capture after the first call).
void set_smem_attr_once(const void* func, int bytes);
// 2-D bf16 tensor map over a row-major matrix of `rows` rows whose rows are
// `row_elems` elements apart, exposing the first `used_cols` columns, with a
// [64 cols x box_rows] box and 128-byte swizzle.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems, uint32_t box_rows,
                    uint64_t used_cols);
// [groups][rows][cols] bf16 (contiguous), boxes of 64 columns x box_rows rows
// of one group, 128-byte swizzle
bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t groups,
                    uint32_t box_rows);
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace dsa
