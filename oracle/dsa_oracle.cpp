// CPU oracle for the DSA sparse-attention hot path. TEST INFRASTRUCTURE ONLY:
// the tests, the smoke check and the benchmark's CPU-baseline leg load it; the
// CUDA library never does, and this file shares no code, header or constant
// with it.
//
// The plain, slow, obviously correct definition of every step, written from
// the sglang-jax DSA pages:
//   * "ref.py" (jnp reference implementations, which the page calls the
//     correctness oracles of its kernels): build_index_share_map,
//     streamindex_topk_ref, streamindex_page_topk_ref, sparse_mla_ref;
//   * "sparse_mla_prefill_qblock.py": build_block_unit_tables, _qblock_kernel,
//     sparse_mla_attention_qblock, prefill_write_and_attend_ragged_qblock,
//     paged_write_back;
//   * "dsa_sparse_backend.py": the IndexShare dispatch, the prefill page
//     budget, _scatter_paged, compute_topk_pages and the dense route.
//
// Plain C++17, OpenMP over query rows only (each row is computed by one
// thread, in the order written here, so the result does not depend on the
// thread count). Arithmetic in double: bf16 and fp32 inputs widen exactly;
// the indexer score is rounded once to fp32, as the pages keep scores in
// fp32; the attention (logits, softmax, weighted sum) stays in double. The
// pages' approximate top-k (approx_max_k) is replaced by the exact top-k,
// ties to the lower index.
//
// Readings taken where the pages are silent:
//   * selected sets are emitted in ascending index order, -1 padded (the
//     pages emit score order; every consumer is order-invariant);
//   * the attention masks every key by both j < kv_len and j <= pos (the jnp
//     reference applies only the first, the qblock kernel both; they coincide
//     on indices produced by the indexer);
//   * a row with no visible key outputs 0 (the pages' masked softmax does the
//     same);
//   * the dense route's sliding window W keeps positions pos-W < j <= pos and
//     its logit cap c maps a scaled logit l to c*tanh(l/c);
//   * compute_topk_pages (imported, not shown) is the sorted unique pages of
//     the selected tokens, the first `cap` of them;
//   * the approximate top-k is the two-stage form written out in
//     orc_approx_topk_row.
//
// Every function is pinned by tests/test_oracle_pins.py against values and
// properties fixed outside this file; none is "parity unpinned".
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <utility>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

typedef long long i64;

// Input element types accepted for tensors: fp32, fp64, or bf16 bit patterns.
enum { kF32 = 0, kF64 = 1, kBF16 = 2 };

// Exact widening of element i of an array of the given type.
inline double widen_at(const void* p, int dtype, i64 i) {
  if (dtype == kF32) return (double)static_cast<const float*>(p)[i];
  if (dtype == kF64) return static_cast<const double*>(p)[i];
  const uint32_t bits = (uint32_t)static_cast<const uint16_t*>(p)[i] << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

inline void widen_row(const void* p, int dtype, i64 off, i64 n, double* out) {
  for (i64 i = 0; i < n; ++i) out[i] = widen_at(p, dtype, off + i);
}

const double kNegInf = -std::numeric_limits<double>::infinity();

// ---------------------------------------------------------------- metadata
// Request of token t: the s with cu_q_lens[s] <= t < cu_q_lens[s+1], i.e. the
// searchsorted(cu_q_lens[1:], t, side="right") of
// prefill_write_and_attend_ragged_qblock.
i64 seq_of(const i64* cu_q_lens, i64 S, i64 t) {
  i64 s = 0;
  while (s < S && cu_q_lens[s + 1] <= t) ++s;
  return s;
}

struct Geom {
  i64 seq, pos, nvis;
};

// ref.py, streamindex_topk_ref: abs_q = kv_len - (q_end - q_start) + (t - q_start);
// visible keys j < kv_len and j <= abs_q, i.e. the prefix [0, nvis).
Geom geom_of(const i64* seq_lens, const i64* cu_q_lens, i64 S, i64 t) {
  Geom g;
  g.seq = seq_of(cu_q_lens, S, t);
  const i64 q0 = cu_q_lens[g.seq], q1 = cu_q_lens[g.seq + 1];
  const i64 kv = seq_lens[g.seq];
  g.pos = kv - (q1 - q0) + (t - q0);
  g.nvis = std::max<i64>(0, std::min(kv, g.pos + 1));
  return g;
}

// Flat physical row page*ps + offset of position j of request s (ref.py:
// seq_pages = page_indices[cu_kv_lens[s]//ps : ...]).
i64 physical_row(const i64* cu_kv_lens, const i64* page_indices, i64 ps, i64 s, i64 j) {
  const i64 base = cu_kv_lens[s] / ps;
  return page_indices[base + j / ps] * ps + j % ps;
}

// --------------------------------------------------------------- a1: score
// s_j = sum_h relu(q[h,:] . k_j) * w[h] (ref.py, streamindex_topk_ref: an
// einsum over D, relu, an einsum with the head weights), summed in double and
// rounded once to fp32. No extra scale factor: the pages' score has none.
float score_one(const double* q, const double* w, const double* key, i64 H, i64 D) {
  double s = 0.0;
  for (i64 h = 0; h < H; ++h) {
    double dot = 0.0;
    for (i64 d = 0; d < D; ++d) dot += q[h * D + d] * key[d];
    s += std::max(dot, 0.0) * w[h];
  }
  return (float)s;
}

// --------------------------------------------------------------- a2: top-k
// Exact top-k of one row: the finite entries ordered by (score desc, index
// asc), the first min(k, n_finite) kept and emitted ascending, -1 padded.
void topk_row(const float* s, i64 n, i64 k, i64* out) {
  std::vector<i64> idx;
  for (i64 j = 0; j < n; ++j)
    if (std::isfinite(s[j])) idx.push_back(j);
  std::sort(idx.begin(), idx.end(), [&](i64 a, i64 b) {
    if (s[a] != s[b]) return s[a] > s[b];
    return a < b;
  });
  const i64 m = std::min<i64>(k, (i64)idx.size());
  std::vector<i64> chosen(idx.begin(), idx.begin() + m);
  std::sort(chosen.begin(), chosen.end());
  for (i64 i = 0; i < k; ++i) out[i] = i < m ? chosen[i] : -1;
}

// --------------------------------------------------------- a3: page scores
// streamindex_page_topk_ref: scores.reshape(.., pages, ps).max(-1); only the
// row's (visible) entries enter the max.
void page_scores_row(const float* s, i64 n, i64 ps, float* out) {
  const i64 npg = (n + ps - 1) / ps;
  for (i64 p = 0; p < npg; ++p) {
    float m = -std::numeric_limits<float>::infinity();
    for (i64 r = p * ps; r < std::min(n, (p + 1) * ps); ++r) m = std::max(m, s[r]);
    out[p] = m;
  }
}

// ----------------------------------------------------- a5/a6: attention
// Masked softmax attention of one query (H heads) over the given key rows,
// in double: logits l = sm_scale * q . k, o = sum_j e^(l_j - max) v_j /
// sum_j e^(l_j - max), lse = max + log(sum). No key: o = 0, lse = -inf
// (sparse_mla_ref: p = where(valid, softmax, 0)).
void attend_rows(const double* q, i64 H, i64 Dk, const std::vector<std::vector<double>>& rows, i64 Dv,
                 double sm_scale, double* o, double* lse) {
  const i64 n = (i64)rows.size();
  if (n == 0) {
    for (i64 i = 0; i < H * Dv; ++i) o[i] = 0.0;
    for (i64 h = 0; h < H; ++h) lse[h] = kNegInf;
    return;
  }
  std::vector<double> logit(n);
  for (i64 h = 0; h < H; ++h) {
    const double* qh = q + h * Dk;
    double mx = kNegInf;
    for (i64 j = 0; j < n; ++j) {
      double dot = 0.0;
      for (i64 d = 0; d < Dk; ++d) dot += qh[d] * rows[j][d];
      logit[j] = sm_scale * dot;
      mx = std::max(mx, logit[j]);
    }
    double l = 0.0;
    double* oh = o + h * Dv;
    for (i64 d = 0; d < Dv; ++d) oh[d] = 0.0;
    for (i64 j = 0; j < n; ++j) {
      const double e = std::exp(logit[j] - mx);
      l += e;
      for (i64 d = 0; d < Dv; ++d) oh[d] += e * rows[j][d];
    }
    for (i64 d = 0; d < Dv; ++d) oh[d] /= l;
    lse[h] = mx + std::log(l);
  }
}

}  // namespace

extern "C" {

// Threads the OpenMP loops below use.
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Exact fp64 values of n elements of the given type.
void orc_widen(const void* src, int dtype, i64 n, double* out) { widen_row(src, dtype, 0, n, out); }

// Request of each of T token rows (rows at or past cu_q_lens[S] get S, as the
// searchsorted does).
void orc_token_seq(const i64* cu_q_lens, i64 S, i64 T, i64* seq) {
  for (i64 t = 0; t < T; ++t) seq[t] = seq_of(cu_q_lens, S, t);
}

// Per token: request, absolute position and visible prefix length.
void orc_token_geometry(const i64* seq_lens, const i64* cu_q_lens, i64 S, i64 T, i64* seq, i64* pos, i64* nvis) {
  for (i64 t = 0; t < T; ++t) {
    const Geom g = geom_of(seq_lens, cu_q_lens, S, t);
    seq[t] = g.seq;
    pos[t] = g.pos;
    nvis[t] = g.nvis;
  }
}

void orc_physical_rows(const i64* cu_kv_lens, const i64* page_indices, i64 ps, i64 s, const i64* positions, i64 n,
                       i64* out) {
  for (i64 i = 0; i < n; ++i) out[i] = physical_row(cu_kv_lens, page_indices, ps, s, positions[i]);
}

// ref.py, build_index_share_map: a full layer (0) opens a new slot, a shared
// layer (1) consumes the nearest preceding full layer's slot. Returns 0, or
// 1 = wrong length, 2 = shared before any full layer, 3 = unknown type.
// types == NULL: every layer is full. skip_offset is not used, as on the page.
int orc_share_map(const int* types, i64 n_types, i64 num_layers, i64* full_slot, i64* src_slot, i64* num_full) {
  if (types && n_types != num_layers) return 1;
  i64 last = -1, nfull = 0;
  for (i64 l = 0; l < num_layers; ++l) {
    const int ty = types ? types[l] : 0;
    if (ty == 0) {
      last = nfull++;
      full_slot[l] = last;
      src_slot[l] = last;
    } else if (ty == 1) {
      if (last < 0) return 2;
      full_slot[l] = -1;
      src_slot[l] = last;
    } else {
      return 3;
    }
  }
  *num_full = nfull;
  return 0;
}

// One score row: q [H, D], w [H], keys [n, D] (any accepted types).
void orc_score_row(const void* q, int q_dt, const void* w, int w_dt, const void* keys, int k_dt, i64 H, i64 D,
                   i64 n, float* out) {
  std::vector<double> qd(H * D), wd(H), kd(D);
  widen_row(q, q_dt, 0, H * D, qd.data());
  widen_row(w, w_dt, 0, H, wd.data());
  for (i64 j = 0; j < n; ++j) {
    widen_row(keys, k_dt, j * D, D, kd.data());
    out[j] = score_one(qd.data(), wd.data(), kd.data(), H, D);
  }
}

// Score rows of the tokens `tokens[0..n)`: q [n, H, D] and w [n, H] hold
// those tokens' rows in order; the cache is [P, ps, D]. Row i gets the scores
// of the visible prefix [0, nvis(t)) at out[i*ld ..]; lens[i] = nvis(t).
// Masked positions (-inf) are simply absent from a row.
void orc_indexer_scores(const void* q, int q_dt, const void* w, int w_dt, const void* kcache, int k_dt, i64 ps,
                        i64 H, i64 D, const i64* seq_lens, const i64* cu_q_lens, const i64* cu_kv_lens,
                        const i64* page_indices, i64 S, const i64* tokens, i64 n, i64 ld, float* out, i64* lens) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) {
    const Geom g = geom_of(seq_lens, cu_q_lens, S, tokens[i]);
    std::vector<double> qd(H * D), wd(H), kd(D);
    widen_row(q, q_dt, i * H * D, H * D, qd.data());
    widen_row(w, w_dt, i * H, H, wd.data());
    const i64 m = std::min(g.nvis, ld);
    for (i64 j = 0; j < m; ++j) {
      const i64 r = physical_row(cu_kv_lens, page_indices, ps, g.seq, j);
      widen_row(kcache, k_dt, r * D, D, kd.data());
      out[i * ld + j] = score_one(qd.data(), wd.data(), kd.data(), H, D);
    }
    lens[i] = m;
  }
}

// Exact top-k of each of n rows (row i: s[i*ld ..], lens[i] entries).
void orc_topk_rows(const float* s, i64 ld, const i64* lens, i64 n, i64 k, i64* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) topk_row(s + i * ld, lens[i], k, out + i * k);
}

// Page max-pool of each row, then the exact top-k_pages pages (pages with
// score -inf are dropped): streamindex_page_topk_ref.
void orc_page_topk_rows(const float* s, i64 ld, const i64* lens, i64 n, i64 ps, i64 k_pages, i64* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) {
    std::vector<float> pm((lens[i] + ps - 1) / ps);
    page_scores_row(s + i * ld, lens[i], ps, pm.data());
    topk_row(pm.data(), (i64)pm.size(), k_pages, out + i * k_pages);
  }
}

void orc_page_scores_row(const float* s, i64 n, i64 ps, float* out) { page_scores_row(s, n, ps, out); }

// sparse_mla_attention_qblock (ragged mode): g = cu_kv_lens[seq(t)]//ps + p
// for p >= 0, else -1.
void orc_lift_units(const i64* tk, i64 T, i64 K, const i64* cu_q_lens, i64 S, const i64* cu_kv_lens, i64 ps,
                    i64* out) {
  for (i64 t = 0; t < T; ++t) {
    const i64 base = cu_kv_lens[seq_of(cu_q_lens, S, t)] / ps;
    for (i64 c = 0; c < K; ++c) out[t * K + c] = tk[t * K + c] >= 0 ? tk[t * K + c] + base : -1;
  }
}

// build_block_unit_tables: T padded to a multiple of QB with -1 rows; per
// block the ascending unique selected ids (first u_max kept, -1 padded), the
// uncapped count, and member[b][q][u] = 1 iff query q of block b selected
// units[b][u].
void orc_block_union(const i64* g, i64 T, i64 K, i64 QB, i64 u_max, int* units, signed char* member, int* counts) {
  const i64 nqb = (T + QB - 1) / QB;
  for (i64 b = 0; b < nqb; ++b) {
    std::vector<i64> ids;
    const i64 t1 = std::min(T, (b + 1) * QB);
    for (i64 t = b * QB; t < t1; ++t)
      for (i64 c = 0; c < K; ++c)
        if (g[t * K + c] >= 0) ids.push_back(g[t * K + c]);
    std::sort(ids.begin(), ids.end());
    ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
    counts[b] = (int)ids.size();
    const i64 kept = std::min<i64>(u_max, (i64)ids.size());
    for (i64 u = 0; u < u_max; ++u) units[b * u_max + u] = u < kept ? (int)ids[u] : -1;
    for (i64 q = 0; q < QB; ++q) {
      const i64 t = b * QB + q;
      for (i64 u = 0; u < u_max; ++u) {
        signed char m = 0;
        if (t < T && u < kept)
          for (i64 c = 0; c < K; ++c)
            if (g[t * K + c] == ids[u]) m = 1;
        member[(b * QB + q) * u_max + u] = m;
      }
    }
  }
}

// Key positions named by one selection row: token ids (unit 1) or whole
// pages expanded to p*unit .. p*unit+unit-1; -1 entries ignored, duplicates
// kept as given. Returns the count written to out (capacity K*unit).
i64 orc_selected_positions(const i64* sel, i64 K, i64 unit, i64* out) {
  i64 n = 0;
  for (i64 c = 0; c < K; ++c) {
    if (sel[c] < 0) continue;
    if (unit == 1) {
      out[n++] = sel[c];
    } else {
      for (i64 r = 0; r < unit; ++r) out[n++] = sel[c] * unit + r;
    }
  }
  return n;
}

// sparse_mla_ref for the tokens tokens[0..n): q [n, H, Dk] their query rows,
// sel [n, K] their selection rows (unit 1: token ids; unit ps: page ids);
// kv cache [P, ps, W] with the key in columns [0, Dk) and the value in
// [0, Dv) of the same row. Masked softmax of sm_scale * q . k over the
// selected positions j with 0 <= j < kv_len and j <= pos(t); o [n, H, Dv]
// and lse [n, H] in double.
void orc_sparse_mla(const void* q, int q_dt, const void* kv, int kv_dt, i64 ps, i64 W, i64 H, i64 Dk, i64 Dv,
                    const i64* seq_lens, const i64* cu_q_lens, const i64* cu_kv_lens, const i64* page_indices, i64 S,
                    const i64* tokens, i64 n, const i64* sel, i64 K, i64 unit, double sm_scale, double* o,
                    double* lse) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) {
    const Geom g = geom_of(seq_lens, cu_q_lens, S, tokens[i]);
    std::vector<i64> pos(K * unit);
    const i64 np = orc_selected_positions(sel + i * K, K, unit, pos.data());
    std::vector<std::vector<double>> rows;
    for (i64 c = 0; c < np; ++c) {
      const i64 j = pos[c];
      if (j < 0 || j >= g.nvis) continue;
      const i64 r = physical_row(cu_kv_lens, page_indices, ps, g.seq, j);
      std::vector<double> row(std::max(Dk, Dv));
      widen_row(kv, kv_dt, r * W, (i64)row.size(), row.data());
      rows.push_back(std::move(row));
    }
    std::vector<double> qd(H * Dk);
    widen_row(q, q_dt, i * H * Dk, H * Dk, qd.data());
    attend_rows(qd.data(), H, Dk, rows, Dv, sm_scale, o + i * H * Dv, lse + i * H);
  }
}

// _qblock_kernel semantics for the tokens tokens[0..n): query t of block
// b = t / QB walks the block's union slots u < min(counts[b], u_max) in
// order; unit g = units[b][u] is physical page page_indices[g], whose row r
// is key position kp = g*ps + r - (cu_kv_lens[seq(t)]/ps)*ps; the key is
// visible iff member[b][t % QB][u] and kp <= pos(t) and kp < kv_len(t).
// Masked softmax over the visible keys, as orc_sparse_mla.
void orc_qblock_attend(const void* q, int q_dt, const void* kv, int kv_dt, i64 ps, i64 W, i64 H, i64 Dk, i64 Dv,
                       const i64* seq_lens, const i64* cu_q_lens, const i64* cu_kv_lens, const i64* page_indices,
                       i64 S, const i64* tokens, i64 n, const i64* units, const signed char* member,
                       const i64* counts, i64 QB, i64 u_max, double sm_scale, double* o, double* lse) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) {
    const i64 t = tokens[i];
    const Geom g = geom_of(seq_lens, cu_q_lens, S, t);
    const i64 b = t / QB, qq = t % QB;
    const i64 base_tok = (cu_kv_lens[g.seq] / ps) * ps;
    const i64 kv_len = seq_lens[g.seq];
    std::vector<std::vector<double>> rows;
    for (i64 u = 0; u < std::min(counts[b], u_max); ++u) {
      if (!member[(b * QB + qq) * u_max + u]) continue;
      const i64 unit = units[b * u_max + u];
      for (i64 r = 0; r < ps; ++r) {
        const i64 kp = unit * ps + r - base_tok;
        if (kp > g.pos || kp >= kv_len) continue;
        std::vector<double> row(std::max(Dk, Dv));
        widen_row(kv, kv_dt, (page_indices[unit] * ps + r) * W, (i64)row.size(), row.data());
        rows.push_back(std::move(row));
      }
    }
    std::vector<double> qd(H * Dk);
    widen_row(q, q_dt, i * H * Dk, H * Dk, qd.data());
    attend_rows(qd.data(), H, Dk, rows, Dv, sm_scale, o + i * H * Dv, lse + i * H);
  }
}

// Dense causal absorbed MLA (the route the backend falls back to), written
// independently of the sparse path: every visible position, one at a time,
// with a two-pass max / sum softmax per head. window > 0 keeps the `window`
// most recent positions pos-window < j <= pos; cap > 0 maps each scaled
// logit l to cap*tanh(l/cap) first. o [n, H, Dv].
void orc_dense_mla(const void* q, int q_dt, const void* kv, int kv_dt, i64 ps, i64 W, i64 H, i64 Dk, i64 Dv,
                   const i64* seq_lens, const i64* cu_q_lens, const i64* cu_kv_lens, const i64* page_indices, i64 S,
                   const i64* tokens, i64 n, double sm_scale, i64 window, double cap, double* o) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 i = 0; i < n; ++i) {
    const Geom g = geom_of(seq_lens, cu_q_lens, S, tokens[i]);
    std::vector<double> qd(H * Dk);
    widen_row(q, q_dt, i * H * Dk, H * Dk, qd.data());
    double* oi = o + i * H * Dv;
    const i64 last = g.nvis - 1;  // the query's own position when it is visible
    const i64 lo = window > 0 ? std::max<i64>(0, last - window + 1) : 0;
    if (g.nvis - lo <= 0) {
      for (i64 e = 0; e < H * Dv; ++e) oi[e] = 0.0;
      continue;
    }
    const i64 m = g.nvis - lo;
    std::vector<double> logit(m * H), vals(m * Dv), row(std::max(Dk, Dv));
    for (i64 j = lo; j < g.nvis; ++j) {
      const i64 r = page_indices[cu_kv_lens[g.seq] / ps + j / ps] * ps + j % ps;
      widen_row(kv, kv_dt, r * W, (i64)row.size(), row.data());
      for (i64 d = 0; d < Dv; ++d) vals[(j - lo) * Dv + d] = row[d];
      for (i64 h = 0; h < H; ++h) {
        double l = 0.0;
        for (i64 d = 0; d < Dk; ++d) l += qd[h * Dk + d] * row[d];
        l *= sm_scale;
        logit[(j - lo) * H + h] = cap > 0.0 ? cap * std::tanh(l / cap) : l;
      }
    }
    std::vector<double> wgt(m);
    for (i64 h = 0; h < H; ++h) {
      double mx = kNegInf;
      for (i64 j = 0; j < m; ++j) mx = std::max(mx, logit[j * H + h]);
      double tot = 0.0;
      for (i64 j = 0; j < m; ++j) {
        wgt[j] = std::exp(logit[j * H + h] - mx);
        tot += wgt[j];
      }
      for (i64 d = 0; d < Dv; ++d) {
        double acc = 0.0;
        for (i64 j = 0; j < m; ++j) acc += wgt[j] * vals[j * Dv + d];
        oi[h * Dv + d] = acc / tot;
      }
    }
  }
}

// dsa_sparse_backend.py, _scatter_paged: token t of request s lands at
// absolute position pos = kv_len - q_len + (t - q_start), i.e. row pos % ps of
// physical page page_indices[cu_kv_lens[s]//ps + pos//ps]; the first D
// columns of that cache row are overwritten with the token's row. The cache
// is [P, ps, W] elements of `elem` bytes; rows [T, D] of the same type.
void orc_paged_write_back(unsigned char* cache, i64 elem, i64 ps, i64 W, const unsigned char* rows, i64 D,
                          const i64* seq_lens, const i64* cu_q_lens, const i64* cu_kv_lens, const i64* page_indices,
                          i64 S, i64 T) {
  for (i64 t = 0; t < T; ++t) {
    const Geom g = geom_of(seq_lens, cu_q_lens, S, t);
    const i64 entry = cu_kv_lens[g.seq] / ps + g.pos / ps;
    const i64 r = page_indices[entry] * ps + g.pos % ps;
    std::memcpy(cache + r * W * elem, rows + t * D * elem, (size_t)(D * elem));
  }
}

// compute_topk_pages (dsa_sparse_backend.py imports it; its module is not
// shown): the ascending unique pages position // ps of one query's selected
// tokens, the first `cap` of them, -1 padded; returns the uncapped count.
i64 orc_topk_pages_of_tokens(const i64* row, i64 K, i64 ps, i64 cap, i64* out) {
  std::vector<i64> pages;
  for (i64 c = 0; c < K; ++c)
    if (row[c] >= 0) pages.push_back(row[c] / ps);
  std::sort(pages.begin(), pages.end());
  pages.erase(std::unique(pages.begin(), pages.end()), pages.end());
  for (i64 i = 0; i < cap; ++i) out[i] = i < (i64)pages.size() ? pages[i] : -1;
  return (i64)pages.size();
}

// Approximate top-k of one row, the two-stage form written out (the pages'
// fast path calls approx_max_k with a recall target): fold the n scores into
// B = min(n, over*k) bins (bin b holds positions b, b+B, b+2B, ...), keep
// each bin's largest score (lowest position on ties), take the exact top-k of
// the B bin maxima (ties to the lower bin) and return their positions in
// ascending order, -1 padded.
void orc_approx_topk_row(const float* s, i64 n, i64 k, i64 over, i64* out) {
  for (i64 i = 0; i < k; ++i) out[i] = -1;
  if (n == 0) return;
  const i64 B = std::min(n, over * k);
  std::vector<i64> best_pos(B);
  std::vector<float> best_val(B);
  for (i64 b = 0; b < B; ++b) {
    i64 j = b;
    for (i64 x = b + B; x < n; x += B)
      if (s[x] > s[j]) j = x;
    best_pos[b] = j;
    best_val[b] = s[j];
  }
  std::vector<i64> bins(k);
  topk_row(best_val.data(), B, k, bins.data());
  std::vector<i64> sel;
  for (i64 i = 0; i < k; ++i)
    if (bins[i] >= 0) sel.push_back(best_pos[bins[i]]);
  std::sort(sel.begin(), sel.end());
  for (i64 i = 0; i < (i64)sel.size(); ++i) out[i] = sel[i];
}

}  // extern "C"
