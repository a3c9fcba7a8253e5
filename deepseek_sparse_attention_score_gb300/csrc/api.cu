// extern "C" entry points of include/dsa.h: host-side argument checks,
// workspace carving, and the kernel launches of each operation.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include <nvtx3/nvToolsExt.h>

#include "attend.cuh"
#include "common.cuh"
#include "indexer.cuh"

namespace dsa {

static std::atomic<long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

void set_smem_attr_once(const void* func, int bytes) {
  struct Entry {
    const void* f;
    int dev;
  };
  static Entry done[64];
  static int ndone = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < ndone; ++i)
    if (done[i].f == func && done[i].dev == dev) return;
  cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (ndone < 64) done[ndone++] = {func, dev};
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems, uint32_t box_rows,
                    uint64_t used_cols) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {used_cols, rows};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t groups,
                    uint32_t box_rows) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, groups};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool ps_supported(int ps) { return ps == 32 || ps == 64 || ps == 128; }

static int check_meta(const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                      const int32_t* page_indices, int T, int S, int P, int PTW, int ps) {
  if (T < 0 || S < 0 || P < 0 || PTW < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (T > 0 && (S < 1 || P < 1 || PTW < 1)) return DSA_ERR_INVALID_ARGUMENT;
  if (T > 0 && (!seq_lens || !cu_q_lens || !cu_kv_lens || !page_indices)) return DSA_ERR_INVALID_ARGUMENT;
  if (!ps_supported(ps)) return DSA_ERR_UNSUPPORTED;
  if ((long long)P * ps >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

static int indexer_common(cudaStream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di,
                          int max_kv, int k_pages, int32_t* topk_pages, int k, int32_t* topk, float* topk_scores,
                          void* ws, size_t ws_bytes, int32_t* dev_status) {
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  if (Hi != 32 || Di != 128) return DSA_ERR_UNSUPPORTED;
  if (max_kv < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (topk && k < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (topk_pages && k_pages < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (!topk && !topk_pages) return DSA_ERR_INVALID_ARGUMENT;
  if (T == 0) return DSA_OK;
  if (!q || !w || !kcache) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(w) || !aligned16(kcache)) return DSA_ERR_ALIGNMENT;
  if (T >= (1 << 24) || S >= (1 << 24)) return DSA_ERR_UNSUPPORTED;
  const IndexerLayout L = indexer_layout(T, S, max_kv, ps);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  IndexerMeta m{w, seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps, max_kv, dev_status, 0, 0};
  IndexerPlan pl;
  IndexerOut out;
  rc = run_indexer(stream, m, q, kcache, ws, L, topk != nullptr, topk_pages != nullptr, &pl, &out);
  if (rc) return rc;
  if (topk) {
    rc = run_topk(stream, out.tok_scores, out.ld_tok, pl.nvis, T, 1, k, topk, topk_scores, max_kv);
    if (rc) return rc;
  }
  if (topk_pages) {
    rc = run_page_topk(stream, out.gran_scores, out.ld_gr, pl.nvis, T, ps, k_pages, topk_pages,
                       reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.page_scores), (long long)L.ld_pg,
                       (max_kv + ps - 1) / ps);
    if (rc) return rc;
  }
  return DSA_OK;
}

static int attend_check(const uint16_t* q, const uint16_t* kv, int row_stride, int T, int H, int Dk, int Dv,
                        uint16_t* o) {
  if (H < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (Dk != 576 || Dv != 512) return DSA_ERR_UNSUPPORTED;
  if (row_stride != 576 && row_stride != 640) return DSA_ERR_UNSUPPORTED;
  if (T > 0 && H > 0 && (!q || !kv || !o)) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(o)) return DSA_ERR_ALIGNMENT;
  if (T > 65535) return DSA_ERR_UNSUPPORTED;  // grid.y
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

namespace {
// One NVTX range per device entry point, so a timeline tool shows the ABI
// calls around their kernels (header-only NVTX: free unless a tool attaches).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

extern "C" {

int dsa_device_sm_count(void) { return sm_count(); }

int dsa_selftest_wait_timeout(dsa_stream_t stream, long long limit_clocks, int32_t* dev_status) {
  if (!dev_status || limit_clocks < 1 || limit_clocks > 10000000000LL) return DSA_ERR_INVALID_ARGUMENT;
  return run_wait_timeout_selftest(static_cast<cudaStream_t>(stream), limit_clocks, dev_status);
}

int dsa_topk_pages_from_tokens(dsa_stream_t stream, const int32_t* topk, int T, int K, int ps, int max_pages,
                               int cap, int32_t* pages, int32_t* counts, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_topk_pages_from_tokens");
  if (T < 0 || K < 0 || ps < 1 || cap < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (max_pages < 1 || max_pages > topk_pages_max_pages()) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!pages || (K > 0 && !topk)) return DSA_ERR_INVALID_ARGUMENT;
  return run_topk_pages(static_cast<cudaStream_t>(stream), topk, T, K, ps, max_pages, cap, pages, counts,
                        dev_status);
}

int dsa_paged_write_back(dsa_stream_t stream, const uint16_t* rows, int src_stride, int D, uint16_t* cache,
                         int cache_stride, const int32_t* seq_lens, const int32_t* cu_q_lens,
                         const int32_t* cu_kv_lens, const int32_t* page_indices, int T, int S, int P, int PTW,
                         int ps, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_paged_write_back");
  return dsa_paged_write_back_pair(stream, rows, src_stride, D, cache, cache_stride, nullptr, 0, 0, nullptr, 0,
                                   seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps, dev_status);
}

static int write_back_target_check(const uint16_t* rows, int src_stride, int D, uint16_t* cache, int cache_stride) {
  if (D < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (D == 0) return DSA_OK;
  if (!rows || !cache) return DSA_ERR_INVALID_ARGUMENT;
  if (D % 8 || src_stride % 8 || cache_stride % 8 || D > src_stride || D > cache_stride) return DSA_ERR_UNSUPPORTED;
  if (!aligned16(rows) || !aligned16(cache)) return DSA_ERR_ALIGNMENT;
  return DSA_OK;
}

int dsa_paged_write_back_pair(dsa_stream_t stream, const uint16_t* rows0, int src_stride0, int D0, uint16_t* cache0,
                              int cache_stride0, const uint16_t* rows1, int src_stride1, int D1, uint16_t* cache1,
                              int cache_stride1, const int32_t* seq_lens, const int32_t* cu_q_lens,
                              const int32_t* cu_kv_lens, const int32_t* page_indices, int T, int S, int P, int PTW,
                              int ps, int32_t* dev_status) {
  if (T < 0 || S < 0 || P < 0 || PTW < 0) return DSA_ERR_INVALID_ARGUMENT;
  int rc = write_back_target_check(rows0, src_stride0, D0, cache0, cache_stride0);
  if (rc) return rc;
  if (rows1 || cache1 || D1) {
    rc = write_back_target_check(rows1, src_stride1, D1, cache1, cache_stride1);
    if (rc) return rc;
  }
  if (T == 0 || D0 == 0) {
    if (D1 == 0 || T == 0) return DSA_OK;
    // only the second cache: write it as the first
    rows0 = rows1, src_stride0 = src_stride1, D0 = D1, cache0 = cache1, cache_stride0 = cache_stride1;
    rows1 = nullptr, cache1 = nullptr, D1 = 0;
  }
  if (S < 1 || P < 1 || PTW < 1 || ps < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (!seq_lens || !cu_q_lens || !cu_kv_lens || !page_indices) return DSA_ERR_INVALID_ARGUMENT;
  return run_paged_write_back(static_cast<cudaStream_t>(stream), rows0, src_stride0, D0, cache0, cache_stride0, rows1,
                              src_stride1, D1, cache1, cache_stride1, seq_lens, cu_q_lens, cu_kv_lens, page_indices,
                              T, S, P, PTW, ps, dev_status);
}
long long dsa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int dsa_index_build_share_map(const int32_t* types, int num_layers, int skip_offset, int32_t* full_slot,
                              int32_t* src_slot, int32_t* num_full) {
  (void)skip_offset;  // accepted and unused, as in the reference map builder
  if (num_layers < 0 || !full_slot || !src_slot || !num_full) return DSA_ERR_INVALID_ARGUMENT;
  int last = -1, nfull = 0;
  for (int l = 0; l < num_layers; ++l) {
    const int ty = types ? types[l] : 0;
    if (ty == 0) {
      last = nfull++;
      full_slot[l] = last;
      src_slot[l] = last;
    } else if (ty == 1) {
      if (last < 0) return DSA_ERR_SHARED_BEFORE_FULL;
      full_slot[l] = -1;
      src_slot[l] = last;
    } else {
      return DSA_ERR_BAD_INDEXER_TYPE;
    }
  }
  *num_full = nfull;
  return DSA_OK;
}

size_t dsa_indexer_workspace_size(int T, int S, int max_kv, int ps) {
  if (T < 0 || S < 0 || max_kv < 1 || !ps_supported(ps)) return 0;
  return indexer_layout(T, S, max_kv, ps).total;
}

// workspace of the approximate top-k: the indexer's, then bin maxima and
// their positions [T, B], bin counts [T] and the selected bins [T, k]
static size_t approx_bins(int k, int over, int max_kv) {
  const long long kb = (long long)k * over;
  const size_t b = (size_t)(kb < max_kv ? kb : max_kv);
  return (b + 3) & ~(size_t)3;  // the row stride of the bin maxima: a multiple of four
}
static size_t approx_extra(int T, int k, int over, int max_kv) {
  const size_t B = approx_bins(k, over, max_kv);
  return 2 * align_up((size_t)T * B * 4, 256) + align_up((size_t)T * 4, 256) + align_up((size_t)T * k * 4, 256);
}

size_t dsa_indexer_topk_approx_workspace_size(int T, int S, int max_kv, int ps, int k, int over) {
  if (T < 0 || S < 0 || max_kv < 1 || !ps_supported(ps) || k < 1 || over < 1) return 0;
  return indexer_layout(T, S, max_kv, ps).total + approx_extra(T, k, over, max_kv);
}

int dsa_indexer_topk_approx(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                            const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                            const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di,
                            int max_kv, int k, int over, int32_t* topk, void* ws, size_t ws_bytes,
                            int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_indexer_topk_approx");
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  if (Hi != 32 || Di != 128) return DSA_ERR_UNSUPPORTED;
  if (!topk || k < 1 || over < 1 || max_kv < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (k > approx_max_k()) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!q || !w || !kcache) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(w) || !aligned16(kcache)) return DSA_ERR_ALIGNMENT;
  if (T >= (1 << 24) || S >= (1 << 24)) return DSA_ERR_UNSUPPORTED;
  const IndexerLayout L = indexer_layout(T, S, max_kv, ps);
  if (!ws || ws_bytes < L.total + approx_extra(T, k, over, max_kv) || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  IndexerMeta m{w, seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps, max_kv, dev_status, 0, 0};
  IndexerPlan pl;
  IndexerOut out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = run_indexer(st, m, q, kcache, ws, L, true, false, &pl, &out);
  if (rc) return rc;
  const size_t B = approx_bins(k, over, max_kv);
  uint8_t* x = static_cast<uint8_t*>(ws) + L.total;
  float* vals = reinterpret_cast<float*>(x);
  x += align_up((size_t)T * B * 4, 256);
  int* pos = reinterpret_cast<int*>(x);
  x += align_up((size_t)T * B * 4, 256);
  int* nb = reinterpret_cast<int*>(x);
  x += align_up((size_t)T * 4, 256);
  int32_t* cand = reinterpret_cast<int32_t*>(x);
  return run_topk_approx(st, out.tok_scores, out.ld_tok, pl.nvis, T, k, over, max_kv, vals, pos, nb, cand, topk);
}

int dsa_indexer_topk(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                     const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                     const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di, int max_kv,
                     int k, int32_t* topk, float* topk_scores, void* ws, size_t ws_bytes, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_indexer_topk");
  if (!topk) return DSA_ERR_INVALID_ARGUMENT;
  return indexer_common(static_cast<cudaStream_t>(stream), q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens,
                        page_indices, T, S, P, PTW, ps, Hi, Di, max_kv, 0, nullptr, k, topk, topk_scores, ws,
                        ws_bytes, dev_status);
}

int dsa_indexer_page_topk(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di,
                          int max_kv, int k_pages, int32_t* topk_pages, int k, int32_t* topk, float* topk_scores,
                          void* ws, size_t ws_bytes, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_indexer_page_topk");
  if (!topk_pages) return DSA_ERR_INVALID_ARGUMENT;
  return indexer_common(static_cast<cudaStream_t>(stream), q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens,
                        page_indices, T, S, P, PTW, ps, Hi, Di, max_kv, k_pages, topk_pages, k, topk, topk_scores,
                        ws, ws_bytes, dev_status);
}

int dsa_build_block_union(dsa_stream_t stream, const int32_t* topk_units, int T, int K, int QB, int u_max,
                          const int32_t* cu_q_lens, const int32_t* cu_kv_lens, int S, int ps, int PTW,
                          int32_t* units, uint32_t* member, int32_t* counts, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_build_block_union");
  if (T < 0 || K < 1 || QB < 32 || QB % 32 != 0 || QB > 1024 || PTW < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (cu_q_lens && (!cu_kv_lens || S < 1 || ps < 1)) return DSA_ERR_INVALID_ARGUMENT;
  if (u_max <= 0) u_max = (int)std::min<long long>((long long)QB * K, PTW);
  if (T == 0) return DSA_OK;
  if (!topk_units || !units || !member || !counts) return DSA_ERR_INVALID_ARGUMENT;
  return run_block_union(static_cast<cudaStream_t>(stream), topk_units, T, K, QB, u_max, cu_q_lens, cu_kv_lens, S,
                         ps, PTW, units, member, counts, dev_status);
}

size_t dsa_sparse_mla_decode_workspace_size(int T, int H, int Dv) {
  if (T <= 0 || H <= 0 || Dv != 512) return 0;
  const int z = attend_num_splits(T, H, 1 << 30, kModeToken);
  return attend_workspace_bytes(T, H, z);
}

int dsa_sparse_mla_decode(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, const int32_t* sel, int K, int unit, int T, int S, int P,
                          int PTW, int ps, int H, int Dk, int Dv, float sm_scale, uint16_t* o, float* lse,
                          void* ws, size_t ws_bytes, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_sparse_mla_decode");
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  rc = attend_check(q, kv, row_stride, T, H, Dk, Dv, o);
  if (rc) return rc;
  if (K < 1 || (T > 0 && !sel)) return DSA_ERR_INVALID_ARGUMENT;
  if (unit != 1 && unit != ps) return DSA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARGUMENT;
  if (T == 0 || H == 0) return DSA_OK;
  AttendParams prm{};
  prm.q = q;
  prm.kv = kv;
  prm.row_stride = row_stride;
  prm.seq_lens = seq_lens;
  prm.cu_q_lens = cu_q_lens;
  prm.cu_kv_lens = cu_kv_lens;
  prm.page_indices = page_indices;
  prm.T = T;
  prm.S = S;
  prm.P = P;
  prm.PTW = PTW;
  prm.ps = ps;
  prm.H = H;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  prm.mode = unit == 1 ? kModeToken : kModePage;
  prm.sel = sel;
  prm.K = K;
  prm.o = o;
  prm.lse = lse;
  prm.dev_status = dev_status;
  int z = attend_num_splits(T, H, K, prm.mode);
  if (z > 1 && (!ws || ws_bytes < attend_workspace_bytes(T, H, z) || !aligned16(ws))) z = 1;
  prm.nsplit = z;
  return run_attend(static_cast<cudaStream_t>(stream), prm, ws, ws_bytes);
}

int dsa_dense_mla(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride, const int32_t* seq_lens,
                  const int32_t* cu_q_lens, const int32_t* cu_kv_lens, const int32_t* page_indices, int max_kv,
                  int T, int S, int P, int PTW, int ps, int H, int Dk, int Dv, float sm_scale, int sliding_window,
                  float soft_cap, uint16_t* o, float* lse, void* ws, size_t ws_bytes, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_dense_mla");
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  rc = attend_check(q, kv, row_stride, T, H, Dk, Dv, o);
  if (rc) return rc;
  if (max_kv < 1 || sliding_window < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale) || !std::isfinite(soft_cap) || soft_cap < 0.f) return DSA_ERR_INVALID_ARGUMENT;
  if (T == 0 || H == 0) return DSA_OK;
  AttendParams prm{};
  prm.q = q;
  prm.kv = kv;
  prm.row_stride = row_stride;
  prm.seq_lens = seq_lens;
  prm.cu_q_lens = cu_q_lens;
  prm.cu_kv_lens = cu_kv_lens;
  prm.page_indices = page_indices;
  prm.T = T;
  prm.S = S;
  prm.P = P;
  prm.PTW = PTW;
  prm.ps = ps;
  prm.H = H;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  prm.mode = kModeDense;
  prm.window = sliding_window;
  if (soft_cap > 0.f) {
    prm.soft_cap_on = 1;
    prm.inv_cap_scale = sm_scale / soft_cap;
    prm.cap_log2 = soft_cap * 1.4426950408889634f;
  }
  prm.K = (max_kv + ps - 1) / ps;  // pages of the longest request: the split unit
  prm.o = o;
  prm.lse = lse;
  prm.dev_status = dev_status;
  int z = attend_num_splits(T, H, prm.K, prm.mode);
  if (z > 1 && (!ws || ws_bytes < attend_workspace_bytes(T, H, z) || !aligned16(ws))) z = 1;
  prm.nsplit = z;
  return run_attend(static_cast<cudaStream_t>(stream), prm, ws, ws_bytes);
}

// No-allocation variant of dsa_sparse_mla_decode: the same checks and split
// choice; the split scratch is the library's built-in device array instead of
// a caller workspace.
int dsa_sparse_mla_decode_noalloc(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                                  const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                  const int32_t* page_indices, const int32_t* sel, int K, int unit, int T, int S,
                                  int P, int PTW, int ps, int H, int Dk, int Dv, float sm_scale, uint16_t* o,
                                  float* lse, int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_sparse_mla_decode_noalloc");
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  rc = attend_check(q, kv, row_stride, T, H, Dk, Dv, o);
  if (rc) return rc;
  if (K < 1 || (T > 0 && !sel)) return DSA_ERR_INVALID_ARGUMENT;
  if (unit != 1 && unit != ps) return DSA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARGUMENT;
  if (T == 0 || H == 0) return DSA_OK;
  AttendParams prm{};
  prm.q = q;
  prm.kv = kv;
  prm.row_stride = row_stride;
  prm.seq_lens = seq_lens;
  prm.cu_q_lens = cu_q_lens;
  prm.cu_kv_lens = cu_kv_lens;
  prm.page_indices = page_indices;
  prm.T = T;
  prm.S = S;
  prm.P = P;
  prm.PTW = PTW;
  prm.ps = ps;
  prm.H = H;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  prm.mode = unit == 1 ? kModeToken : kModePage;
  prm.sel = sel;
  prm.K = K;
  prm.o = o;
  prm.lse = lse;
  prm.dev_status = dev_status;
  prm.nsplit = attend_num_splits(T, H, K, prm.mode);
  return run_attend_static_scratch(static_cast<cudaStream_t>(stream), prm);
}

static int qblock_common(cudaStream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                         const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                         const int32_t* page_indices, const int32_t* units, const uint32_t* member,
                         const int32_t* counts, int QB, int u_max, int T, int S, int P, int PTW, int ps, int H, int Dk,
                         int Dv, float sm_scale, int t_begin, int t_end, uint16_t* o, float* lse,
                         int32_t* dev_status) {
  int rc = check_meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices, T, S, P, PTW, ps);
  if (rc) return rc;
  rc = attend_check(q, kv, row_stride, T, H, Dk, Dv, o);
  if (rc) return rc;
  if (QB < 32 || QB % 32 != 0 || u_max < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (t_begin < 0 || t_end < t_begin || t_end > T) return DSA_ERR_INVALID_ARGUMENT;
  if (T > 0 && (!units || !member || !counts)) return DSA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARGUMENT;
  if (t_end == t_begin || H == 0) return DSA_OK;
  AttendParams prm{};
  prm.q = q;
  prm.kv = kv;
  prm.row_stride = row_stride;
  prm.seq_lens = seq_lens;
  prm.cu_q_lens = cu_q_lens;
  prm.cu_kv_lens = cu_kv_lens;
  prm.page_indices = page_indices;
  prm.T = T;
  prm.S = S;
  prm.P = P;
  prm.PTW = PTW;
  prm.ps = ps;
  prm.H = H;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  prm.mode = kModeQblock;
  prm.units = units;
  prm.member = member;
  prm.counts = counts;
  prm.QB = QB;
  prm.u_max = u_max;
  prm.K = 1;
  prm.nsplit = 1;
  prm.t0 = t_begin;
  prm.tn = t_end - t_begin;
  prm.o = o;
  prm.lse = lse;
  prm.dev_status = dev_status;
  return run_attend(stream, prm, nullptr, 0);
}

int dsa_sparse_mla_prefill_qblock(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                                  const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                  const int32_t* page_indices, const int32_t* units, const uint32_t* member,
                                  const int32_t* counts, int QB, int u_max, int T, int S, int P, int PTW, int ps,
                                  int H, int Dk, int Dv, float sm_scale, uint16_t* o, float* lse,
                                  int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_sparse_mla_prefill_qblock");
  return qblock_common(static_cast<cudaStream_t>(stream), q, kv, row_stride, seq_lens, cu_q_lens, cu_kv_lens,
                       page_indices, units, member, counts, QB, u_max, T, S, P, PTW, ps, H, Dk, Dv, sm_scale, 0,
                       T < 0 ? 0 : T, o, lse, dev_status);
}

int dsa_sparse_mla_prefill_qblock_range(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                                        const int32_t* seq_lens, const int32_t* cu_q_lens,
                                        const int32_t* cu_kv_lens, const int32_t* page_indices,
                                        const int32_t* units, const uint32_t* member, const int32_t* counts, int QB,
                                        int u_max, int T, int S, int P, int PTW, int ps, int H, int Dk, int Dv,
                                        float sm_scale, int t_begin, int t_end, uint16_t* o, float* lse,
                                        int32_t* dev_status) {
  NvtxRange nvtx_range("dsa_sparse_mla_prefill_qblock_range");
  return qblock_common(static_cast<cudaStream_t>(stream), q, kv, row_stride, seq_lens, cu_q_lens, cu_kv_lens,
                       page_indices, units, member, counts, QB, u_max, T, S, P, PTW, ps, H, Dk, Dv, sm_scale,
                       t_begin, t_end, o, lse, dev_status);
}

}  // extern "C"
