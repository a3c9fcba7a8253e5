// Per-query-block union + membership (sparse_mla_prefill_qblock.py,
// build_block_unit_tables, with the ragged-mode lift of
// sparse_mla_attention_qblock).
//
// One CTA per block of QB queries. The block's QB*K lifted unit ids are
// marked in a shared-memory bitmap over [min id, max id] (in windows of 256K
// ids, so any id range works); a block scan of per-word popcounts turns the
// bitmap into the ascending unique list, and the same prefix gives every id
// its union slot directly, so membership bits are set without a sort or a
// search. The pages build the same tables by sort + broadcast-compare, their
// TPU-friendly form.
#include "common.cuh"

namespace dsa {

constexpr int kUnionThreads = 1024;
constexpr int kWindowWords = 8192;  // 256K unit ids per bitmap window
constexpr int kWordsPerThread = kWindowWords / kUnionThreads;

__device__ __forceinline__ int lifted_unit(const int32_t* topk_units, const int32_t* cu_q_lens,
                                           const int32_t* cu_kv_lens, int S, int ps, int K, int t, int c) {
  const int p = __ldg(topk_units + (size_t)t * K + c);
  if (p < 0) return -1;
  if (!cu_q_lens) return p;
  const int s = seq_of_token(cu_q_lens, S, t);
  return __ldg(cu_kv_lens + s) / ps + p;
}

__global__ void __launch_bounds__(kUnionThreads) block_union_kernel(const int32_t* __restrict__ topk_units, int T,
                                                                    int K, int QB, int u_max,
                                                                    const int32_t* __restrict__ cu_q_lens,
                                                                    const int32_t* __restrict__ cu_kv_lens, int S,
                                                                    int ps, int PTW, int32_t* __restrict__ units,
                                                                    uint32_t* __restrict__ member,
                                                                    int32_t* __restrict__ counts,
                                                                    int32_t* dev_status) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ uint32_t bits[kWindowWords];
  __shared__ int s_base[kUnionThreads];
  __shared__ int s_warp[32];
  __shared__ int s_min, s_max;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const int t0 = b * QB, nq = min(QB, T - t0);
  const int words_q = QB / 32;
  const int nent = nq * K;
  uint32_t* mem_b = member + (size_t)b * u_max * words_q;
  int32_t* units_b = units + (size_t)b * u_max;
  for (size_t i = tid; i < (size_t)u_max * words_q; i += kUnionThreads) mem_b[i] = 0u;
  if (tid == 0) {
    s_min = 0x7fffffff;
    s_max = -1;
  }
  __syncthreads();
  int lmin = 0x7fffffff, lmax = -1;
  for (int e = tid; e < nent; e += kUnionThreads) {
    const int g = lifted_unit(topk_units, cu_q_lens, cu_kv_lens, S, ps, K, t0 + e / K, e % K);
    if (g < 0) continue;
    if (g >= PTW) {
      set_status(dev_status, DSA_STATUS_BAD_INDEX);
      continue;
    }
    lmin = min(lmin, g);
    lmax = max(lmax, g);
  }
  atomicMin(&s_min, lmin);
  atomicMax(&s_max, lmax);
  __syncthreads();
  const int gmin = s_min, gmax = s_max;
  int count = 0;  // uniques emitted by earlier windows
  if (gmax >= 0) {
    for (long long w0 = gmin; w0 <= gmax; w0 += (long long)kWindowWords * 32) {
      const long long w1 = w0 + (long long)kWindowWords * 32;
      for (int i = tid; i < kWindowWords; i += kUnionThreads) bits[i] = 0u;
      __syncthreads();
      for (int e = tid; e < nent; e += kUnionThreads) {
        const int g = lifted_unit(topk_units, cu_q_lens, cu_kv_lens, S, ps, K, t0 + e / K, e % K);
        if (g < 0 || g >= PTW || g < w0 || g >= w1) continue;
        const int off = (int)(g - w0);
        atomicOr(bits + (off >> 5), 1u << (off & 31));
      }
      __syncthreads();
      // block exclusive scan of the per-thread popcounts (8 words per thread)
      int local = 0;
#pragma unroll
      for (int j = 0; j < kWordsPerThread; ++j) local += __popc(bits[tid * kWordsPerThread + j]);
      int x = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) s_warp[wp] = x;
      __syncthreads();
      if (wp == 0) {
        int y = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int z = __shfl_up_sync(0xffffffffu, y, o);
          if (lane >= o) y += z;
        }
        s_warp[lane] = y;
      }
      __syncthreads();
      const int excl = x - local + (wp > 0 ? s_warp[wp - 1] : 0);
      const int tot = s_warp[31];
      s_base[tid] = count + excl;
      // ascending unique ids: thread order == id order
      int slot = count + excl;
#pragma unroll
      for (int j = 0; j < kWordsPerThread; ++j) {
        uint32_t word = bits[tid * kWordsPerThread + j];
        const long long idbase = w0 + (long long)(tid * kWordsPerThread + j) * 32;
        while (word) {
          const int bit = __ffs(word) - 1;
          if (slot < u_max) units_b[slot] = (int)(idbase + bit);
          ++slot;
          word &= word - 1u;
        }
      }
      __syncthreads();
      // membership: slot(g) = base(owner thread) + popcounts of the owner's
      // words below g's word + popcount of the bits below g in its word
      for (int e = tid; e < nent; e += kUnionThreads) {
        const int q = e / K;
        const int g = lifted_unit(topk_units, cu_q_lens, cu_kv_lens, S, ps, K, t0 + q, e % K);
        if (g < 0 || g >= PTW || g < w0 || g >= w1) continue;
        const int off = (int)(g - w0), wd = off >> 5, owner = wd / kWordsPerThread;
        int s = s_base[owner];
        for (int j = owner * kWordsPerThread; j < wd; ++j) s += __popc(bits[j]);
        s += __popc(bits[wd] & ((1u << (off & 31)) - 1u));
        if (s < u_max) atomicOr(mem_b + (size_t)s * words_q + (q >> 5), 1u << (q & 31));
      }
      count += tot;
      __syncthreads();
    }
  }
  if (tid == 0) {
    counts[b] = count;
    if (count > u_max) set_status(dev_status, DSA_STATUS_UNION_TRUNCATED);
  }
  for (int s = count + tid; s < u_max; s += kUnionThreads) units_b[s] = -1;
}

int run_block_union(cudaStream_t stream, const int32_t* topk_units, int T, int K, int QB, int u_max,
                    const int32_t* cu_q_lens, const int32_t* cu_kv_lens, int S, int ps, int PTW, int32_t* units,
                    uint32_t* member, int32_t* counts, int32_t* dev_status) {
  const int nqb = (T + QB - 1) / QB;
  if (nqb == 0) return DSA_OK;
  DSA_LAUNCH_PDL(block_union_kernel, dim3(nqb), dim3(kUnionThreads), 0, stream, topk_units, T, K, QB, u_max,
                 cu_q_lens, cu_kv_lens, S, ps, PTW, units, member, counts, dev_status);
  return DSA_OK;
}

}  // namespace dsa
