// Sparse-MLA attention internals shared by the attention and API units.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>

namespace dsa {

enum : int { kModeToken = 0, kModePage = 1, kModeQblock = 2, kModeDense = 3 };

struct AttendParams {
  const uint16_t* q;   // bf16 [T, H, 576]
  const uint16_t* kv;  // bf16 [P, ps, row_stride]
  int row_stride;
  const int32_t* seq_lens;
  const int32_t* cu_q_lens;
  const int32_t* cu_kv_lens;
  const int32_t* page_indices;
  int T, S, P, PTW, ps, H;
  float scale_log2;  // sm_scale * log2(e)
  int mode;
  const int32_t* sel;  // token / page modes: [T, K]
  int K;
  const int32_t* units;  // qblock mode
  const uint32_t* member;
  const int32_t* counts;
  int QB, u_max;
  int window;           // dense mode: keep the `window` most recent positions (0 = all)
  int soft_cap_on;      // logits l -> cap * tanh(l / cap) before the softmax
  float inv_cap_scale;  // sm_scale / cap
  float cap_log2;       // cap * log2(e)
  int nsplit;
  int t0;  // first query token of the launch (grid.y walks tokens t0 .. t0 + tn - 1)
  int tn;  // tokens in the launch; 0 means all T
  uint16_t* o;      // bf16 [T, H, 512]
  float* lse;       // [T, H] or null
  float* o_part;    // [nsplit, T, H, 512] (set by run_attend)
  float* lse_part;  // per-CTA lse copies (set by run_attend)
  int* counters;    // split arrival counters (set by run_attend)
  int32_t* dev_status;
};

int attend_num_splits(int T, int H, int K, int mode);
size_t attend_workspace_bytes(int T, int H, int nsplit);
int run_attend(cudaStream_t stream, AttendParams prm, void* ws, size_t ws_bytes);
// Same as run_attend with the split scratch in a built-in device array.
int run_attend_static_scratch(cudaStream_t stream, AttendParams prm);

int run_block_union(cudaStream_t stream, const int32_t* topk_units, int T, int K, int QB, int u_max,
                    const int32_t* cu_q_lens, const int32_t* cu_kv_lens, int S, int ps, int PTW, int32_t* units,
                    uint32_t* member, int32_t* counts, int32_t* dev_status);

// Paged write-back of new token rows (writeback.cu).
// one or two caches sharing the page table (rows1 == NULL: one)
int run_paged_write_back(cudaStream_t stream, const uint16_t* rows, long long src_stride, int D, uint16_t* cache,
                         long long cache_stride, const uint16_t* rows1, long long src_stride1, int D1,
                         uint16_t* cache1, long long cache_stride1, const int32_t* seq_lens,
                         const int32_t* cu_q_lens, const int32_t* cu_kv_lens, const int32_t* page_indices, int T,
                         int S, int P, int PTW, int ps, int32_t* dev_status);

// Token top-k -> sorted unique page list per query (pages.cu).
int topk_pages_max_pages();
int run_topk_pages(cudaStream_t stream, const int32_t* topk, int T, int K, int ps, int max_pages, int cap,
                   int32_t* pages, int32_t* counts, int32_t* dev_status);

// Bounded-wait self-test (selftest.cu).
int run_wait_timeout_selftest(cudaStream_t stream, long long limit_clocks, int32_t* dev_status);

}  // namespace dsa
