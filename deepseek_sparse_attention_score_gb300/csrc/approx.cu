// Approximate token top-k (ref.py, streamindex_topk_ref's fast path uses
// approx_max_k with a recall target; this is a two-stage GPU form of the
// same trade): a row of n visible scores is folded into B = min(n, over * k)
// bins (bin b holds positions b, b + B, b + 2B, ...), each bin keeps its
// maximum (lowest position on ties), and the exact top-k of the B bin maxima
// (ties to the lower bin) is the approximate selection, written in ascending
// position order and -1 padded. A true top-k position is missed only when a
// higher score shares its bin, so the recall grows with `over`; B >= n makes
// it exact.
//
// Stage 1 is one coalesced pass over the row (consecutive bins are
// consecutive positions), stage 2 reuses the exact radix select on the
// over * k bin maxima instead of the whole row, stage 3 sorts the k winning
// positions (bitonic, in shared memory).
#include "common.cuh"
#include "indexer.cuh"

namespace dsa {

namespace {
constexpr int kBinThreads = 256;
constexpr int kFinThreads = 512;

__global__ void __launch_bounds__(kBinThreads) approx_bins_kernel(const float* __restrict__ scores, long long ld,
                                                                  const int* __restrict__ nvis, int kb,
                                                                  float* __restrict__ vals, int* __restrict__ pos,
                                                                  int* __restrict__ nb, long long ldb) {
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x;
  const int n = nvis[t];
  const int B = min(n, kb);
  if (blockIdx.y == 0 && threadIdx.x == 0) nb[t] = B;
  const int b = blockIdx.y * kBinThreads + threadIdx.x;
  if (b >= B) return;
  const float* row = scores + (size_t)t * ld;
  float best = __ldg(row + b);
  int bj = b;
  for (int j = b + B; j < n; j += B) {
    const float v = __ldg(row + j);
    if (v > best) {  // strictly greater: the lowest position wins ties
      best = v;
      bj = j;
    }
  }
  vals[(size_t)t * ldb + b] = best;
  pos[(size_t)t * ldb + b] = bj;
}

__global__ void __launch_bounds__(kFinThreads) approx_finish_kernel(const int32_t* __restrict__ cand, int k,
                                                                    const int* __restrict__ pos, long long ldb,
                                                                    int32_t* __restrict__ out, int n_pow2) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int a[];
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < n_pow2; i += kFinThreads) {
    const int b = i < k ? __ldg(cand + (size_t)t * k + i) : -1;
    a[i] = b >= 0 ? __ldg(pos + (size_t)t * ldb + b) : 0x7fffffff;
  }
  __syncthreads();
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2 / 2; i += kFinThreads) {
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
  for (int i = threadIdx.x; i < k; i += kFinThreads) out[(size_t)t * k + i] = a[i] == 0x7fffffff ? -1 : a[i];
}
}  // namespace

int approx_max_k() { return 16384; }

int run_topk_approx(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int k, int over,
                    int max_kv, float* vals, int* pos, int* nb, int32_t* cand, int32_t* out) {
  if (T == 0) return DSA_OK;
  const long long kb = (long long)k * over;
  const int bmax = (int)(kb < max_kv ? kb : max_kv);
  const int ldb = (bmax + 3) & ~3;  // bin rows start 16-byte aligned (the top-k reads them as float4)
  dim3 g1(T, (bmax + kBinThreads - 1) / kBinThreads);
  DSA_LAUNCH_PDL(approx_bins_kernel, dim3(g1), dim3(kBinThreads), 0, stream, scores, ld, nvis,
                 (int)(kb < (1LL << 30) ? kb : (1LL << 30)),
                                                     vals, pos, nb, ldb);
  int rc = run_topk(stream, vals, ldb, nb, T, 1, k, cand, nullptr, bmax);
  if (rc) return rc;
  int n_pow2 = 1;
  while (n_pow2 < k) n_pow2 <<= 1;
  set_smem_attr_once(reinterpret_cast<const void*>(approx_finish_kernel), approx_max_k() * 4);
  DSA_LAUNCH_PDL(approx_finish_kernel, dim3(T), dim3(kFinThreads), (size_t)n_pow2 * 4, stream, cand, k, pos, ldb,
                 out, n_pow2);
  return DSA_OK;
}

}  // namespace dsa
