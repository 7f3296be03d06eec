/*
 * mla_oracle.c -- plain fp64 CPU oracle for absorbed-MLA decode attention
 * under decode context parallelism (DCP).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Every function is the plain definition written out, in double precision,
 * with no blocking, fusion or reordering.  bf16 inputs are widened exactly.
 * Sources (page title, then section):
 *   [P1] "[Attention] add DCP support for FLASH_ATTN_MLA backend" -- review
 *        thread: the per-rank seqlen_k example and the mask tables
 *        "Normal", "DCP Rank 0", "DCP Rank 1".
 *   [P2] "[Attention][DCP] Support DCP with query length > 1 (MTP) with FA3"
 *        -- Purpose: varlen queries, pass the cp world size and rank.
 *   [P3] "vllm.v1.attention.backends.mla.flashattn_mla" --
 *        FlashAttnMLAImpl._forward_decode: q split into (q_nope, q_pe),
 *        cache split into kv_c (first kv_lora_rank) and k_pe, call with
 *        q=q_pe, k=k_pe, v=kv_c, q_v=q_nope, causal, softmax_scale, LSE.
 *   [P4] "[Attention] DCP sparse MLA output-merge optimizations" -- summary:
 *        LSE-weighted merge, W_UV projection commuting with it, per-row
 *        valid counts, sparse MLA.
 *
 * Parity pins (tests/test_oracle_*.py) check this file against the mask
 * tables of [P1], closed forms, brute force and invariants; see those tests.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define KV_LORA_RANK 512 /* width of kv_c, from [P3] kv_c_cache slice */
#define ROPE_DIM 64      /* width of k_pe */
#define ROW_WIDTH (KV_LORA_RANK + ROPE_DIM)

/* bf16 -> double is exact: a bf16 is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------- masks -- */

/* [P1] tables: shard r of D holds the global tokens p with p mod D == r, its
 * j-th local token being the j-th such p (so p = j*D + r).  The number of
 * tokens of a request of global length L held by shard r is counted here by
 * enumeration, which is the definition itself. */
int64_t mla_oracle_local_len(int64_t L, int64_t D, int64_t r) {
  int64_t n = 0;
  for (int64_t p = 0; p < L; ++p)
    if (p % D == r) ++n;
  return n;
}

/* [P1] "DCP Rank" tables: query token at global position P (new tokens are
 * the last q_len of the sequence, so P = seq_len - q_len + i) may see local
 * key j on shard r iff j*D + r <= P. */
int mla_oracle_key_visible(int64_t P, int64_t D, int64_t r, int64_t j) {
  return j * D + r <= P;
}

/* Number of local keys of shard r that the query at global position P sees,
 * for a request of global length L, counted by enumeration of the local keys. */
int64_t mla_oracle_visible_count(int64_t P, int64_t L, int64_t D, int64_t r) {
  int64_t n = 0, Lr = mla_oracle_local_len(L, D, r);
  for (int64_t j = 0; j < Lr; ++j)
    if (mla_oracle_key_visible(P, D, r, j)) ++n;
  return n;
}

/* ------------------------------------------------------- one query row -- */

/* Softmax attention of one (query token, head) row over an explicit list of
 * key rows.  [P3]: score = scale * (q_nope . kv_c + q_pe . k_pe); output =
 * sum softmax * kv_c; lse = natural log of sum exp(score) (scale included).
 * An empty list gives lse = -inf and a zero output. */
static void attend_row(const uint16_t *qn, const uint16_t *qp,
                       const uint16_t *const *keys, int64_t nkeys, double scale,
                       double *s /* scratch [nkeys] */, double *out,
                       double *lse) {
  for (int d = 0; d < KV_LORA_RANK; ++d) out[d] = 0.0;
  if (nkeys == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t k = 0; k < nkeys; ++k) {
    const uint16_t *row = keys[k];
    double acc = 0.0;
    for (int d = 0; d < KV_LORA_RANK; ++d)
      acc += bf16_to_double(qn[d]) * bf16_to_double(row[d]);
    for (int e = 0; e < ROPE_DIM; ++e)
      acc += bf16_to_double(qp[e]) * bf16_to_double(row[KV_LORA_RANK + e]);
    s[k] = scale * acc;
    if (s[k] > m) m = s[k];
  }
  double z = 0.0;
  for (int64_t k = 0; k < nkeys; ++k) z += exp(s[k] - m);
  double l = m + log(z);
  for (int64_t k = 0; k < nkeys; ++k) {
    double p = exp(s[k] - l);
    const uint16_t *row = keys[k];
    for (int d = 0; d < KV_LORA_RANK; ++d) out[d] += p * bf16_to_double(row[d]);
  }
  *lse = l;
}

/* Cache row of local token j of request b, read through the block table
 * ([P3] block_table argument; pages of page_size rows of ROW_WIDTH). */
static const uint16_t *paged_row(const uint16_t *kv_cache, int64_t page_size,
                                 const int32_t *block_table, int64_t bt_stride,
                                 int64_t b, int64_t j) {
  int64_t page = block_table[b * bt_stride + j / page_size];
  return kv_cache + (page * page_size + j % page_size) * ROW_WIDTH;
}

/* Request that owns query token t. */
static int64_t request_of(const int32_t *qsl, int64_t B, int64_t t) {
  for (int64_t b = 0; b < B; ++b)
    if (t >= qsl[b] && t < qsl[b + 1]) return b;
  return -1;
}

/* --------------------------------------------- dense, unsharded, causal -- */

/* Unsharded causal MLA over a logical (unpaged) KV sequence per request:
 * kv rows of request b are kv[kv_start[b] .. kv_start[b]+seq_lens[b]).  Query
 * token i of request b sits at P = L - q_len + i and sees keys p <= P ([P1]
 * "Normal" table; [P3] causal=True).  Tokens [t_lo, t_hi) are computed;
 * out [t_hi - t_lo, H, 512] and lse [t_hi - t_lo, H] hold them in order. */
void mla_oracle_causal_dense(const uint16_t *q_nope, const uint16_t *q_pe,
                             const uint16_t *kv, const int64_t *kv_start,
                             const int32_t *seq_lens, const int32_t *qsl,
                             int64_t B, int64_t H, double scale, int64_t t_lo,
                             int64_t t_hi, double *out, double *lse,
                             const uint16_t **key_scratch, double *s_scratch) {
  for (int64_t t = t_lo; t < t_hi; ++t) {
    int64_t b = request_of(qsl, B, t);
    int64_t L = seq_lens[b], q_len = qsl[b + 1] - qsl[b];
    int64_t P = L - q_len + (t - qsl[b]);
    int64_t n = 0;
    for (int64_t p = 0; p < L; ++p)
      if (p <= P) key_scratch[n++] = kv + (kv_start[b] + p) * ROW_WIDTH;
    for (int64_t h = 0; h < H; ++h)
      attend_row(q_nope + (t * H + h) * KV_LORA_RANK,
                 q_pe + (t * H + h) * ROPE_DIM, key_scratch, n, scale,
                 s_scratch, out + ((t - t_lo) * H + h) * KV_LORA_RANK,
                 lse + (t - t_lo) * H + h);
  }
}

/* ------------------------------------------------- dense, one DCP shard -- */

/* Shard r of D: its cache slice holds the local tokens of every request,
 * paged through its own block table.  Seq_lens are GLOBAL lengths (new
 * tokens included); the shard-local length and the per-row visible count
 * come from the [P1] rule.  row_counts[t - t_lo] = number of keys token t
 * sees.  Tokens [t_lo, t_hi) are computed; outputs are indexed from t_lo. */
void mla_oracle_dcp_decode(const uint16_t *q_nope, const uint16_t *q_pe,
                           const uint16_t *kv_cache, int64_t page_size,
                           const int32_t *block_table, int64_t bt_stride,
                           const int32_t *seq_lens, const int32_t *qsl,
                           int64_t B, int64_t H, int64_t D, int64_t r,
                           double scale, int64_t t_lo, int64_t t_hi,
                           double *out, double *lse, int32_t *row_counts,
                           const uint16_t **key_scratch, double *s_scratch) {
  for (int64_t t = t_lo; t < t_hi; ++t) {
    int64_t b = request_of(qsl, B, t);
    int64_t L = seq_lens[b], q_len = qsl[b + 1] - qsl[b];
    int64_t P = L - q_len + (t - qsl[b]);
    int64_t Lr = mla_oracle_local_len(L, D, r);
    int64_t n = 0;
    for (int64_t j = 0; j < Lr; ++j)
      if (mla_oracle_key_visible(P, D, r, j))
        key_scratch[n++] =
            paged_row(kv_cache, page_size, block_table, bt_stride, b, j);
    row_counts[t - t_lo] = (int32_t)n;
    for (int64_t h = 0; h < H; ++h)
      attend_row(q_nope + (t * H + h) * KV_LORA_RANK,
                 q_pe + (t * H + h) * ROPE_DIM, key_scratch, n, scale,
                 s_scratch, out + ((t - t_lo) * H + h) * KV_LORA_RANK,
                 lse + (t - t_lo) * H + h);
  }
}

/* ------------------------------------- dense, one DCP shard, FP8 cache -- */

/* FP8 latent cache (an extension: the [P3] backend rejects an FP8 cache).
 * Reading taken: every value of a cache row (kv_c and k_pe) is stored as one
 * OCP FP8 E4M3 code -- 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals at exponent 0, no infinities, S.1111.111 is NaN -- and
 * the whole tensor shares one dequantisation scale: the value is
 * kv_scale * decode(code).  The decode below is that definition, exact in
 * double. */
double mla_oracle_e4m3_to_double(uint8_t code) {
  int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);              /* m/8 * 2^(1-7) */
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);      /* 1.m * 2^(e-7) */
  return sign ? -v : v;
}

/* attend_row with FP8 key rows: each value is kv_scale * decode(code). */
static void attend_row_kv8(const uint16_t *qn, const uint16_t *qp,
                           const uint8_t *const *keys, int64_t nkeys,
                           double kv_scale, double scale, double *s,
                           double *out, double *lse) {
  for (int d = 0; d < KV_LORA_RANK; ++d) out[d] = 0.0;
  if (nkeys == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t k = 0; k < nkeys; ++k) {
    const uint8_t *row = keys[k];
    double acc = 0.0;
    for (int d = 0; d < KV_LORA_RANK; ++d)
      acc += bf16_to_double(qn[d]) * (kv_scale * mla_oracle_e4m3_to_double(row[d]));
    for (int e = 0; e < ROPE_DIM; ++e)
      acc += bf16_to_double(qp[e]) *
             (kv_scale * mla_oracle_e4m3_to_double(row[KV_LORA_RANK + e]));
    s[k] = scale * acc;
    if (s[k] > m) m = s[k];
  }
  double z = 0.0;
  for (int64_t k = 0; k < nkeys; ++k) z += exp(s[k] - m);
  double l = m + log(z);
  for (int64_t k = 0; k < nkeys; ++k) {
    double p = exp(s[k] - l);
    const uint8_t *row = keys[k];
    for (int d = 0; d < KV_LORA_RANK; ++d)
      out[d] += p * (kv_scale * mla_oracle_e4m3_to_double(row[d]));
  }
  *lse = l;
}

/* mla_oracle_dcp_decode over an FP8 cache slice [pages][page_size][576]
 * bytes with dequantisation scale kv_scale. */
void mla_oracle_dcp_decode_kv8(const uint16_t *q_nope, const uint16_t *q_pe,
                               const uint8_t *kv_cache, double kv_scale,
                               int64_t page_size, const int32_t *block_table,
                               int64_t bt_stride, const int32_t *seq_lens,
                               const int32_t *qsl, int64_t B, int64_t H,
                               int64_t D, int64_t r, double scale,
                               int64_t t_lo, int64_t t_hi, double *out,
                               double *lse, int32_t *row_counts,
                               const uint8_t **key_scratch,
                               double *s_scratch) {
  for (int64_t t = t_lo; t < t_hi; ++t) {
    int64_t b = request_of(qsl, B, t);
    int64_t L = seq_lens[b], q_len = qsl[b + 1] - qsl[b];
    int64_t P = L - q_len + (t - qsl[b]);
    int64_t Lr = mla_oracle_local_len(L, D, r);
    int64_t n = 0;
    for (int64_t j = 0; j < Lr; ++j)
      if (mla_oracle_key_visible(P, D, r, j)) {
        int64_t page = block_table[b * bt_stride + j / page_size];
        key_scratch[n++] = kv_cache + (page * page_size + j % page_size) * ROW_WIDTH;
      }
    row_counts[t - t_lo] = (int32_t)n;
    for (int64_t h = 0; h < H; ++h)
      attend_row_kv8(q_nope + (t * H + h) * KV_LORA_RANK,
                     q_pe + (t * H + h) * ROPE_DIM, key_scratch, n, kv_scale,
                     scale, s_scratch,
                     out + ((t - t_lo) * H + h) * KV_LORA_RANK,
                     lse + (t - t_lo) * H + h);
  }
}

/* ------------------------------------------------ sparse, one DCP shard -- */

/* [P4] sparse MLA: query token t attends to the keys listed in
 * topk[t, 0 .. valid[t]) (global positions of its request).  An entry is
 * used iff 0 <= idx <= P (padding is -1; keys past the query position are
 * never visible).  Shard r keeps the entries with idx mod D == r, at local
 * position idx div D.  local_counts[t - t_lo] = entries kept by shard r.
 * Outputs are indexed from t_lo. */
void mla_oracle_sparse_dcp_decode(
    const uint16_t *q_nope, const uint16_t *q_pe, const uint16_t *kv_cache,
    int64_t page_size, const int32_t *block_table, int64_t bt_stride,
    const int32_t *seq_lens, const int32_t *qsl, int64_t B, int64_t H,
    const int32_t *topk, int64_t K, const int32_t *valid, int64_t D, int64_t r,
    double scale, int64_t t_lo, int64_t t_hi, double *out, double *lse,
    int32_t *local_counts, const uint16_t **key_scratch, double *s_scratch) {
  for (int64_t t = t_lo; t < t_hi; ++t) {
    int64_t b = request_of(qsl, B, t);
    int64_t L = seq_lens[b], q_len = qsl[b + 1] - qsl[b];
    int64_t P = L - q_len + (t - qsl[b]);
    int64_t n = 0;
    for (int64_t e = 0; e < valid[t] && e < K; ++e) {
      int64_t p = topk[t * K + e];
      if (p < 0 || p > P) continue;
      if (p % D != r) continue;
      key_scratch[n++] =
          paged_row(kv_cache, page_size, block_table, bt_stride, b, p / D);
    }
    local_counts[t - t_lo] = (int32_t)n;
    for (int64_t h = 0; h < H; ++h)
      attend_row(q_nope + (t * H + h) * KV_LORA_RANK,
                 q_pe + (t * H + h) * ROPE_DIM, key_scratch, n, scale,
                 s_scratch, out + ((t - t_lo) * H + h) * KV_LORA_RANK,
                 lse + (t - t_lo) * H + h);
  }
}

/* ---------------------------------------------------------- DCP merge -- */

/* [P4] LSE-weighted merge of D partial results per (token, head) row:
 * LSE = log sum_r exp(lse_r), out = sum_r exp(lse_r - LSE) * o_r, over the
 * shards that hold keys for the row.  With valid_counts [D, T] given, shard r
 * takes part iff valid_counts[r, t] > 0 and its partial is not read
 * otherwise; without them, shard r takes part iff lse_r > -inf.  No shard
 * taking part gives out = 0 and LSE = -inf.  partials [D, T, H, width]. */
void mla_oracle_lse_merge(const double *partials, const double *lses,
                          const int32_t *valid_counts, int64_t D, int64_t T,
                          int64_t H, int64_t width, double *out,
                          double *lse_out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double *o = out + (t * H + h) * width;
      for (int64_t d = 0; d < width; ++d) o[d] = 0.0;
      double m = -INFINITY;
      int any = 0;
      for (int64_t r = 0; r < D; ++r) {
        int part = valid_counts ? valid_counts[r * T + t] > 0
                                : lses[(r * T + t) * H + h] > -INFINITY;
        if (!part) continue;
        double l = lses[(r * T + t) * H + h];
        if (!any || l > m) m = l;
        any = 1;
      }
      if (!any || m == -INFINITY) {
        lse_out[t * H + h] = -INFINITY;
        continue;
      }
      double z = 0.0;
      for (int64_t r = 0; r < D; ++r) {
        int part = valid_counts ? valid_counts[r * T + t] > 0
                                : lses[(r * T + t) * H + h] > -INFINITY;
        if (part) z += exp(lses[(r * T + t) * H + h] - m);
      }
      double L = m + log(z);
      for (int64_t r = 0; r < D; ++r) {
        int part = valid_counts ? valid_counts[r * T + t] > 0
                                : lses[(r * T + t) * H + h] > -INFINITY;
        if (!part) continue;
        double w = exp(lses[(r * T + t) * H + h] - L);
        const double *p = partials + ((r * T + t) * H + h) * width;
        for (int64_t d = 0; d < width; ++d) o[d] += w * p[d];
      }
      lse_out[t * H + h] = L;
    }
}

/* ------------------------------------------------------------- W_UV -- */

/* [P4] per-head up-projection y[t, h, :] = o[t, h, :] . W_UV[h] with W_UV
 * [H, 512, V] (bf16, widened exactly).  rows = T*H rows of width 512. */
void mla_oracle_wuv_project(const double *o, const uint16_t *w_uv, int64_t T,
                            int64_t H, int64_t V, double *y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      const double *x = o + (t * H + h) * KV_LORA_RANK;
      const uint16_t *w = w_uv + h * KV_LORA_RANK * V;
      double *out = y + (t * H + h) * V;
      for (int64_t v = 0; v < V; ++v) {
        double acc = 0.0;
        for (int64_t d = 0; d < KV_LORA_RANK; ++d)
          acc += x[d] * bf16_to_double(w[d * V + v]);
        out[v] = acc;
      }
    }
}
