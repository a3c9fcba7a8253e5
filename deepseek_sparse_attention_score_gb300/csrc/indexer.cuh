// Indexer internals shared by the indexer, top-k and API translation units.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>

namespace dsa {

constexpr int kChunkDecode = 512;      // keys per work item of one-token tiles (at least)
constexpr int kChunkDecodeMax = 4096;  // ... and at most
constexpr int kChunkPrefill = 2048;    // keys per work item of 8-token tiles

struct IndexerMeta {
  const float* w;
  const int32_t* seq_lens;
  const int32_t* cu_q_lens;
  const int32_t* cu_kv_lens;
  const int32_t* page_indices;
  int T, S, P, PTW, ps, max_kv;
  int32_t* dev_status;
  // one-token launches without a planner: item ii is token ii / direct_nch,
  // keys [c, c + 1) * direct_ch of it with c = ii % direct_nch (0: planned)
  int direct_nch, direct_ch;
};

struct IndexerPlan {
  int* counts;        // [0] decode items, [1] prefill items
  int* nvis;          // [T] visible prefix per token
  int2* seq_tile_off; // [S]
  int4* dec_tiles;
  int4* pre_tiles;
  int4* dec_items;    // {t0, ntok<<24 | seq, key_begin, key_end}
  int4* pre_items;
};

struct IndexerOut {
  float* tok_scores;   // [T, ld_tok] or null
  float* gran_scores;  // [T, ld_gr] or null: the maximum score of every 32-key granule
  long long ld_tok, ld_gr;
};

// page_scores [T, ld_pg]: page maxima folded from the granules, only for page
// rows longer than the page top-k can fold while it reads them
struct IndexerLayout {
  size_t counts, nvis, seq_tile_off, dec_tiles, pre_tiles, dec_items, pre_items, tok_scores, gran_scores, page_scores;
  size_t ld_tok, ld_gr, ld_pg, total;
};

IndexerLayout indexer_layout(int T, int S, int max_kv, int ps);
int run_indexer(cudaStream_t stream, const IndexerMeta& m, const uint16_t* q, const uint16_t* kcache, void* ws,
                const IndexerLayout& L, bool want_tok, bool want_page, IndexerPlan* plan_out, IndexerOut* out_out);

// Approximate token top-k over the score rows (approx.cu).
int approx_max_k();
int run_topk_approx(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int k, int over,
                    int max_kv, float* vals, int* pos, int* nb, int32_t* cand, int32_t* out);
// Exact per-row top-k over a score buffer (token or page scores).
int run_topk(cudaStream_t stream, const float* scores, long long ld, const int* nvis, int T, int div, int k,
             int32_t* out_idx, float* out_val, int max_len);
// Exact page top-k from 32-key granule maxima: a page's score is the maximum
// of its ps / 32 visible granules. page_buf [T, ld_pg] is used only when the
// rows are too long to fold while reading.
int run_page_topk(cudaStream_t stream, const float* gran, long long ld_gr, const int* nvis, int T, int ps, int k_pages,
                  int32_t* out_idx, float* page_buf, long long ld_pg, int max_pages);

}  // namespace dsa
