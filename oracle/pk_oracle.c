/*
 * pk_oracle.c -- plain, slow, fp64 CPU oracle for packed variable-length
 * attention with the HunyuanImage-3.0 "generalized causal" mask.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code with the CUDA library.
 *
 * What it computes (the plain definition, no tiling, no fusion):
 *
 *   Packing.  Requests are packed back to back into one token stream; the
 *   sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]).  No attention
 *   crosses sequences and nothing is padded.
 *     -- "[RFC]: HunyuanImage 3.0 deployment", Proposed Change, P0
 *        "Packed Attention for Multi-Request Batching": contiguous packing
 *        with cu_seqlens replaces batch duplication, padding and the
 *        explicit (bsz,1,seqlen,seqlen) mask (Motivation, item (1)).
 *
 *   Mask.  Inside a sequence of length L, query row i sees key j iff
 *        j <= i                                  (text tokens are causal)
 *     or seg(i) is an IMAGE segment and seg(j) == seg(i)
 *                                  (image tokens see their whole own segment)
 *     -- same page, P0 bullet "Attention mask challenge" (generalized causal
 *        attention: text causal, image bidirectional) and "Model structure",
 *        item 1 (image patches attend to each other simultaneously).
 *     The dense L x L mask is materialised per sequence, exactly as the
 *     replaced path would.
 *
 *   Heads.  Query head h reads key/value head g = h / (Hq / Hkv)
 *     (grouped-query attention, contiguous groups).
 *
 *   Scores, LSE, output (fp64 throughout, from the bf16 input values):
 *        s_ij  = scale * sum_c q[i,h,c] * k[j,g,c]
 *        lse_i = ln sum_{j visible} exp(s_ij)      (max-subtracted)
 *        o_i   = sum_{j visible} exp(s_ij - lse_i) * v[j,g,:]
 *
 * Layouts: q [T][Hq][d], k and v [T][Hkv][d] as raw bf16 bit patterns
 * (uint16); out [rows][Hq][d] fp64; lse [Hq][rows] fp64, where rows is T for
 * the full call or n_rows for the sampled call.  Segments are int32 triples
 * {start (global token index), len, type (0 = text, 1 = image)}.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define PKO_TEXT 0
#define PKO_IMAGE 1

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
double pko_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Descriptor check: cu_seqlens starts at 0 and never decreases; segments are
 * in order, non-empty, typed 0/1, and tile every sequence exactly.
 * Returns 0 when valid, a positive code otherwise. */
int pko_validate(const int32_t* cu, int32_t num_seqs, const int32_t* segs,
                 int32_t num_segs) {
  if (num_seqs < 0 || num_segs < 0) return 1;
  if (cu[0] != 0) return 2;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return 3;
  int32_t g = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t pos = cu[s];
    while (pos < cu[s + 1]) {
      if (g >= num_segs) return 4;
      const int32_t* sg = segs + 3 * g;
      if (sg[0] != pos || sg[1] <= 0) return 5;
      if (sg[2] != PKO_TEXT && sg[2] != PKO_IMAGE) return 6;
      if (sg[0] + sg[1] > cu[s + 1]) return 7;
      pos += sg[1];
      ++g;
    }
  }
  if (g != num_segs) return 8;
  return 0;
}

/* Segment index of every token of the pack (explicit lookup table). */
static int32_t* segment_of_tokens(int32_t T, const int32_t* segs,
                                  int32_t num_segs) {
  int32_t* seg_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  for (int32_t g = 0; g < num_segs; ++g)
    for (int32_t t = segs[3 * g]; t < segs[3 * g] + segs[3 * g + 1]; ++t)
      seg_of[t] = g;
  return seg_of;
}

/* One row of the dense mask of sequence s: row_out[j] = 1 iff the i-th token
 * of s (0-based inside s) sees the j-th token of s. */
static void mask_row(int32_t b, int32_t L, int32_t i, const int32_t* seg_of,
                     const int32_t* segs, uint8_t* row_out) {
  int32_t gi = seg_of[b + i];
  int is_image = segs[3 * gi + 2] == PKO_IMAGE;
  for (int32_t j = 0; j < L; ++j) {
    int causal = j <= i;
    int own_image_segment = is_image && seg_of[b + j] == gi;
    row_out[j] = (uint8_t)(causal || own_image_segment);
  }
}

/* Dense bool mask of sequence s, M[i*L + j], L = cu[s+1]-cu[s]. */
int pko_mask_dense(const int32_t* cu, int32_t num_seqs, const int32_t* segs,
                   int32_t num_segs, int32_t s, uint8_t* M) {
  int rc = pko_validate(cu, num_seqs, segs, num_segs);
  if (rc) return rc;
  if (s < 0 || s >= num_seqs) return 9;
  int32_t T = cu[num_seqs];
  int32_t* seg_of = segment_of_tokens(T, segs, num_segs);
  int32_t b = cu[s], L = cu[s + 1] - cu[s];
  for (int32_t i = 0; i < L; ++i) mask_row(b, L, i, seg_of, segs, M + (size_t)i * L);
  free(seg_of);
  return 0;
}

/* Number of visible (query, key) pairs of the whole pack, per head, counted
 * from the dense mask rule. */
int64_t pko_visible_pairs(const int32_t* cu, int32_t num_seqs,
                          const int32_t* segs, int32_t num_segs) {
  if (pko_validate(cu, num_seqs, segs, num_segs)) return -1;
  int32_t T = cu[num_seqs];
  int32_t* seg_of = segment_of_tokens(T, segs, num_segs);
  int64_t total = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t b = cu[s], L = cu[s + 1] - cu[s];
    uint8_t* row = (uint8_t*)malloc((size_t)(L > 0 ? L : 1));
    for (int32_t i = 0; i < L; ++i) {
      mask_row(b, L, i, seg_of, segs, row);
      for (int32_t j = 0; j < L; ++j) total += row[j];
    }
    free(row);
  }
  free(seg_of);
  return total;
}

/* Visible keys of every query row of the pack (row sums of the dense mask),
 * out[T]; returns 0, or -1 for invalid descriptors. */
int pko_row_keys(const int32_t* cu, int32_t num_seqs, const int32_t* segs,
                 int32_t num_segs, int64_t* out) {
  if (pko_validate(cu, num_seqs, segs, num_segs)) return -1;
  int32_t T = cu[num_seqs];
  int32_t* seg_of = segment_of_tokens(T, segs, num_segs);
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t b = cu[s], L = cu[s + 1] - cu[s];
    uint8_t* row = (uint8_t*)malloc((size_t)(L > 0 ? L : 1));
    for (int32_t i = 0; i < L; ++i) {
      mask_row(b, L, i, seg_of, segs, row);
      int64_t n = 0;
      for (int32_t j = 0; j < L; ++j) n += row[j];
      out[b + i] = n;
    }
    free(row);
  }
  free(seg_of);
  return 0;
}

/* Attention of one query row (all query heads) over its sequence, given the
 * row of the dense mask.  q_row points at q[i][0][0]; k_seq / v_seq at the
 * first token of the sequence.  Writes out_row[Hq][d] and lse[h*lse_stride]. */
static void attend_row(const uint16_t* q_row, const uint16_t* k_seq,
                       const uint16_t* v_seq, const uint8_t* mrow, int32_t L,
                       int32_t Hq, int32_t Hkv, int32_t d, double scale,
                       double* out_row, double* lse, int64_t lse_stride,
                       double* s_buf, double* qd) {
  int32_t group = Hq / Hkv;
  for (int32_t h = 0; h < Hq; ++h) {
    int32_t g = h / group;
    for (int32_t c = 0; c < d; ++c)
      qd[c] = pko_bf16_to_double(q_row[(size_t)h * d + c]);
    double m = -INFINITY;
    for (int32_t j = 0; j < L; ++j) {
      if (!mrow[j]) continue;
      const uint16_t* kj = k_seq + ((size_t)j * Hkv + g) * d;
      double acc = 0.0;
      for (int32_t c = 0; c < d; ++c) acc += qd[c] * pko_bf16_to_double(kj[c]);
      s_buf[j] = scale * acc;
      if (s_buf[j] > m) m = s_buf[j];
    }
    double denom = 0.0;
    for (int32_t j = 0; j < L; ++j)
      if (mrow[j]) denom += exp(s_buf[j] - m);
    double lse_h = m + log(denom);
    lse[(int64_t)h * lse_stride] = lse_h;
    double* o = out_row + (size_t)h * d;
    for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int32_t j = 0; j < L; ++j) {
      if (!mrow[j]) continue;
      double p = exp(s_buf[j] - lse_h);
      const uint16_t* vj = v_seq + ((size_t)j * Hkv + g) * d;
      for (int32_t c = 0; c < d; ++c) o[c] += p * pko_bf16_to_double(vj[c]);
    }
  }
}

/*
 * Packed masked attention.
 *   rows == NULL : every token; out [T][Hq][d], lse [Hq][T].  The dense mask
 *                  of each sequence is built in full before its rows run.
 *   rows != NULL : only the listed global token indices (any order);
 *                  out [n_rows][Hq][d], lse [Hq][n_rows].  Each listed row
 *                  builds its own row of the dense mask.
 * nthreads <= 0 uses the OpenMP default.  Returns 0 or a validation code.
 */
int pko_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const int32_t* cu, int32_t num_seqs, const int32_t* segs,
                  int32_t num_segs, int32_t Hq, int32_t Hkv, int32_t d,
                  double scale, const int32_t* rows, int32_t n_rows,
                  double* out, double* lse, int32_t nthreads) {
  int rc = pko_validate(cu, num_seqs, segs, num_segs);
  if (rc) return rc;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 10;
  int32_t T = cu[num_seqs];
  int32_t* seg_of = segment_of_tokens(T, segs, num_segs);
  int32_t Lmax = 0;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] - cu[s] > Lmax) Lmax = cu[s + 1] - cu[s];
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  if (rows == NULL) {
    for (int32_t s = 0; s < num_seqs; ++s) {
      int32_t b = cu[s], L = cu[s + 1] - cu[s];
      if (L == 0) continue;
      uint8_t* M = (uint8_t*)malloc((size_t)L * L);
      for (int32_t i = 0; i < L; ++i) mask_row(b, L, i, seg_of, segs, M + (size_t)i * L);
#pragma omp parallel
      {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)L);
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int32_t i = 0; i < L; ++i) {
          int32_t t = b + i;
          attend_row(q + (size_t)t * Hq * d, k + (size_t)b * Hkv * d,
                     v + (size_t)b * Hkv * d, M + (size_t)i * L, L, Hq, Hkv, d,
                     scale, out + (size_t)t * Hq * d, lse + t, T, s_buf, qd);
        }
        free(s_buf);
        free(qd);
      }
      free(M);
    }
  } else {
    for (int32_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= T) { free(seg_of); return 11; }
#pragma omp parallel
    {
      double* s_buf = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
      double* qd = (double*)malloc(sizeof(double) * (size_t)d);
      uint8_t* mrow = (uint8_t*)malloc((size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for schedule(dynamic, 1)
      for (int32_t r = 0; r < n_rows; ++r) {
        int32_t t = rows[r];
        int32_t s = 0;
        while (cu[s + 1] <= t) ++s;
        int32_t b = cu[s], L = cu[s + 1] - cu[s];
        mask_row(b, L, t - b, seg_of, segs, mrow);
        attend_row(q + (size_t)t * Hq * d, k + (size_t)b * Hkv * d,
                   v + (size_t)b * Hkv * d, mrow, L, Hq, Hkv, d, scale,
                   out + (size_t)r * Hq * d, lse + r, n_rows, s_buf, qd);
      }
      free(s_buf);
      free(qd);
      free(mrow);
    }
  }
  free(seg_of);
  return 0;
}

/* Threads the OpenMP runtime would use (reported with the CPU baseline). */
int32_t pko_max_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * General form, for queries and keys that are position ranges of their
 * sequences (the cached-prefix hand-over of "[RFC]: HunyuanImage 3.0
 * deployment", Proposed Change, P0 "KV Cache Transfer Integration for DiT":
 * image queries attend to a text prefix whose keys/values come from the AR
 * stage; and key chunks of one sequence, as a ring of devices holds them).
 *
 *   seg_seq/seg_start/seg_len/seg_type [G]: segments of every sequence in its
 *       own position space, ordered, tiling [0, L_s) of each sequence.
 *   cu_q [S+1]: packed query rows; query i of sequence s has position
 *       q_pos0[s] + i.
 *   cu_k [S+1]: key rows per sequence; key j of sequence s has position
 *       k_pos0[s] + j and lives at packed row cu_k[s] + j, or, when
 *       block_table is given, at pool row
 *       block_table[s*blocks_per_seq + p/block] * block + p % block with
 *       p = k_pos0[s] + j.
 *   Query position pq sees key position pk iff the dense mask of the whole
 *   sequence has (pq, pk) set.  A query that sees no key of the range gets
 *   out = 0 and lse = -inf.
 * q: [Tq][Hq][d], k/v: [rows][Hkv][d] bf16 bits; out [Tq][Hq][d], lse [Hq][Tq].
 */
int pko_attention_general(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* cu_q, const int32_t* cu_k, const int32_t* q_pos0,
                          const int32_t* k_pos0, int32_t num_seqs, const int32_t* seg_seq,
                          const int32_t* seg_start, const int32_t* seg_len,
                          const int32_t* seg_type, int32_t num_segs,
                          const int32_t* block_table, int32_t blocks_per_seq, int32_t block,
                          int32_t Hq, int32_t Hkv, int32_t d, double scale, double* out,
                          double* lse, int32_t nthreads) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0) return 10;
  if (cu_q[0] != 0 || cu_k[0] != 0) return 2;
  int32_t* L = (int32_t*)calloc((size_t)(num_seqs > 0 ? num_seqs : 1), sizeof(int32_t));
  int32_t* first_seg = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_seqs + 1));
  for (int32_t s = 0; s <= num_seqs; ++s) first_seg[s] = num_segs;
  for (int32_t g = 0; g < num_segs; ++g) {
    int32_t s = seg_seq[g];
    if (s < 0 || s >= num_seqs || seg_len[g] <= 0 || seg_start[g] != L[s] ||
        (seg_type[g] != PKO_TEXT && seg_type[g] != PKO_IMAGE) ||
        (g > 0 && seg_seq[g - 1] > s)) {
      free(L); free(first_seg); return 5;
    }
    if (first_seg[s] == num_segs) first_seg[s] = g;
    L[s] += seg_len[g];
  }
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t nq = cu_q[s + 1] - cu_q[s], nk = cu_k[s + 1] - cu_k[s];
    if (nq < 0 || nk < 0 || q_pos0[s] < 0 || k_pos0[s] < 0 || q_pos0[s] + nq > L[s] ||
        k_pos0[s] + nk > L[s]) {
      free(L); free(first_seg); return 3;
    }
  }
  const int32_t Tq = cu_q[num_seqs];
  const int32_t group = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t Ls = L[s], nq = cu_q[s + 1] - cu_q[s], nk = cu_k[s + 1] - cu_k[s];
    if (nq == 0) continue;
    /* segment index of every position, then the dense mask rows of the queries */
    int32_t* seg_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(Ls > 0 ? Ls : 1));
    for (int32_t g = first_seg[s]; g < num_segs && seg_seq[g] == s; ++g)
      for (int32_t p = seg_start[g]; p < seg_start[g] + seg_len[g]; ++p) seg_of[p] = g;
#pragma omp parallel
    {
      uint8_t* mrow = (uint8_t*)malloc((size_t)(Ls > 0 ? Ls : 1));
      double* sbuf = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
      double* qd = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
      for (int32_t i = 0; i < nq; ++i) {
        const int32_t pq = q_pos0[s] + i, t = cu_q[s] + i;
        const int32_t gi = seg_of[pq];
        const int is_image = seg_type[gi] == PKO_IMAGE;
        for (int32_t pk = 0; pk < Ls; ++pk)
          mrow[pk] = (uint8_t)(pk <= pq || (is_image && seg_of[pk] == gi));
        for (int32_t h = 0; h < Hq; ++h) {
          const int32_t g = h / group;
          for (int32_t c = 0; c < d; ++c) qd[c] = pko_bf16_to_double(q[((size_t)t * Hq + h) * d + c]);
          double m = -INFINITY;
          for (int32_t j = 0; j < nk; ++j) {
            const int32_t pk = k_pos0[s] + j;
            if (!mrow[pk]) continue;
            size_t row = block_table
                ? (size_t)block_table[(size_t)s * blocks_per_seq + pk / block] * block + pk % block
                : (size_t)(cu_k[s] + j);
            const uint16_t* kj = k + (row * Hkv + g) * d;
            double acc = 0.0;
            for (int32_t c = 0; c < d; ++c) acc += qd[c] * pko_bf16_to_double(kj[c]);
            sbuf[j] = scale * acc;
            if (sbuf[j] > m) m = sbuf[j];
          }
          double* o = out + ((size_t)t * Hq + h) * d;
          for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
          if (m == -INFINITY) {
            lse[(size_t)h * Tq + t] = -INFINITY;
            continue;
          }
          double den = 0.0;
          for (int32_t j = 0; j < nk; ++j)
            if (mrow[k_pos0[s] + j]) den += exp(sbuf[j] - m);
          const double l = m + log(den);
          lse[(size_t)h * Tq + t] = l;
          for (int32_t j = 0; j < nk; ++j) {
            const int32_t pk = k_pos0[s] + j;
            if (!mrow[pk]) continue;
            size_t row = block_table
                ? (size_t)block_table[(size_t)s * blocks_per_seq + pk / block] * block + pk % block
                : (size_t)(cu_k[s] + j);
            const uint16_t* vj = v + (row * Hkv + g) * d;
            const double pw = exp(sbuf[j] - l);
            for (int32_t c = 0; c < d; ++c) o[c] += pw * pko_bf16_to_double(vj[c]);
          }
        }
      }
      free(mrow);
      free(sbuf);
      free(qd);
    }
    free(seg_of);
  }
  free(L);
  free(first_seg);
  return 0;
}

/*
 * Merge of partial attentions over disjoint key sets of the same queries
 * (the combination a ring of devices performs, "Parallelism Acceleration
 * Guide", Ring Attention): with per-part log-sum-exps lse_c and normalised
 * outputs o_c,
 *     lse = ln sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) o_c.
 * Parts with lse_c = -inf contribute nothing; if every part is -inf the
 * result is o = 0, lse = -inf.  o_parts [C][T][H][d], lse_parts [C][H][T]
 * (fp64); out [T][H][d], lse [H][T].
 */
void pko_lse_merge(const double* o_parts, const double* lse_parts, int32_t C, int32_t T,
                   int32_t H, int32_t d, double* out, double* lse) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t h = 0; h < H; ++h) {
      double m = -INFINITY;
      for (int32_t c = 0; c < C; ++c) {
        const double lc = lse_parts[((size_t)c * H + h) * T + t];
        if (lc > m) m = lc;
      }
      double* o = out + ((size_t)t * H + h) * d;
      for (int32_t x = 0; x < d; ++x) o[x] = 0.0;
      if (m == -INFINITY) {
        lse[(size_t)h * T + t] = -INFINITY;
        continue;
      }
      double den = 0.0;
      for (int32_t c = 0; c < C; ++c) den += exp(lse_parts[((size_t)c * H + h) * T + t] - m);
      const double L = m + log(den);
      lse[(size_t)h * T + t] = L;
      for (int32_t c = 0; c < C; ++c) {
        const double w = exp(lse_parts[((size_t)c * H + h) * T + t] - L);
        if (w == 0.0) continue;
        const double* oc = o_parts + (((size_t)c * T + t) * H + h) * d;
        for (int32_t x = 0; x < d; ++x) o[x] += w * oc[x];
      }
    }
}

/* ------------------------------------------------------------------------
 * FP8 queries and keys.  The pages quantise linear layers to FP8 (e.g.
 * "HunyuanImage-3.0-Instruct ...", FP8 checkpoints; "MiniMax H3-Image on Vera
 * Rubin", MXFP8 GEMMs); this entry is the attention of the same packed
 * sequences when q and k arrive as FP8 E4M3 codes with one scale each.
 *
 * E4M3 (the OCP 8-bit floating point format): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m/8 * 2^-6; there are no infinities, and S.1111.111 is NaN.
 */
double pko_e4m3_to_double(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* One query row over its sequence: q value = e4m3(q8) * q_scale, k value =
 * e4m3(k8) * k_scale, v bf16 (v8_seq NULL) or e4m3(v8) * v_scale; the same
 * score, LSE and output definitions as the bf16 entry.  A row with no
 * visible key gets o = 0, lse = -inf. */
static void attend_row_e4m3(const uint8_t* q_row, double q_scale, const uint8_t* k_seq,
                            double k_scale, const uint16_t* v_seq, const uint8_t* v8_seq,
                            double v_scale, const uint8_t* mrow,
                            int32_t L, int32_t Hq, int32_t Hkv, int32_t d, double scale,
                            double* out_row, double* lse, int64_t lse_stride, double* s_buf) {
  const int32_t group = Hq / Hkv;
  for (int32_t h = 0; h < Hq; ++h) {
    const int32_t g = h / group;
    double mx = -INFINITY;
    for (int32_t j = 0; j < L; ++j) {
      if (!mrow[j]) continue;
      double dot = 0.0;
      for (int32_t c = 0; c < d; ++c)
        dot += (pko_e4m3_to_double(q_row[(size_t)h * d + c]) * q_scale) *
               (pko_e4m3_to_double(k_seq[((size_t)j * Hkv + g) * d + c]) * k_scale);
      s_buf[j] = scale * dot;
      if (s_buf[j] > mx) mx = s_buf[j];
    }
    double* o = out_row + (size_t)h * d;
    for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
    if (mx == -INFINITY) {
      lse[(size_t)h * lse_stride] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int32_t j = 0; j < L; ++j)
      if (mrow[j]) z += exp(s_buf[j] - mx);
    const double l = mx + log(z);
    lse[(size_t)h * lse_stride] = l;
    for (int32_t j = 0; j < L; ++j) {
      if (!mrow[j]) continue;
      const double w = exp(s_buf[j] - l);
      const size_t vo = ((size_t)j * Hkv + g) * d;
      if (v8_seq)
        for (int32_t c = 0; c < d; ++c) o[c] += w * (pko_e4m3_to_double(v8_seq[vo + c]) * v_scale);
      else
        for (int32_t c = 0; c < d; ++c) o[c] += w * pko_bf16_to_double(v_seq[vo + c]);
    }
  }
}

/* Packed attention with E4M3 q [T][Hq][d] and k [T][Hkv][d] (codes) and
 * their scales; v bf16 (v8 NULL) or E4M3 codes v8 [T][Hkv][d] with v_scale.
 * rows == NULL: every row, out [T][Hq][d], lse [Hq][T]; else the n_rows
 * listed rows, out [n_rows][Hq][d], lse [Hq][n_rows]. */
static int attention_e4m3(const uint8_t* q8, double q_scale, const uint8_t* k8, double k_scale,
                          const uint16_t* v, const uint8_t* v8, double v_scale,
                          const int32_t* cu, int32_t num_seqs,
                          const int32_t* segs, int32_t num_segs, int32_t Hq, int32_t Hkv,
                          int32_t d, double scale, const int32_t* rows, int32_t n_rows,
                          double* out, double* lse, int32_t nthreads) {
  int rc = pko_validate(cu, num_seqs, segs, num_segs);
  if (rc) return rc;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 10;
  const int32_t T = cu[num_seqs];
  const int32_t n = rows ? n_rows : T;
  for (int32_t r = 0; rows && r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return 11;
  int32_t* seg_of = segment_of_tokens(T, segs, num_segs);
  int32_t Lmax = 1;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] - cu[s] > Lmax) Lmax = cu[s + 1] - cu[s];
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)Lmax);
    uint8_t* mrow = (uint8_t*)malloc((size_t)Lmax);
#pragma omp for schedule(dynamic, 1)
    for (int32_t r = 0; r < n; ++r) {
      const int32_t t = rows ? rows[r] : r;
      int32_t s = 0;
      while (cu[s + 1] <= t) ++s;
      const int32_t b = cu[s], L = cu[s + 1] - cu[s];
      mask_row(b, L, t - b, seg_of, segs, mrow);
      attend_row_e4m3(q8 + (size_t)t * Hq * d, q_scale, k8 + (size_t)b * Hkv * d, k_scale,
                      v8 ? NULL : v + (size_t)b * Hkv * d, v8 ? v8 + (size_t)b * Hkv * d : NULL,
                      v_scale, mrow, L, Hq, Hkv, d, scale,
                      out + (size_t)r * Hq * d, lse + r, n, s_buf);
    }
    free(s_buf);
    free(mrow);
  }
  free(seg_of);
  return 0;
}

int pko_attention_e4m3(const uint8_t* q8, double q_scale, const uint8_t* k8, double k_scale,
                       const uint16_t* v, const int32_t* cu, int32_t num_seqs,
                       const int32_t* segs, int32_t num_segs, int32_t Hq, int32_t Hkv,
                       int32_t d, double scale, const int32_t* rows, int32_t n_rows,
                       double* out, double* lse, int32_t nthreads) {
  return attention_e4m3(q8, q_scale, k8, k_scale, v, NULL, 1.0, cu, num_seqs, segs, num_segs,
                        Hq, Hkv, d, scale, rows, n_rows, out, lse, nthreads);
}

/* The same with E4M3 values too: v8 [T][Hkv][d] codes, value e4m3(v8) * v_scale. */
int pko_attention_e4m3_v8(const uint8_t* q8, double q_scale, const uint8_t* k8, double k_scale,
                          const uint8_t* v8, double v_scale, const int32_t* cu, int32_t num_seqs,
                          const int32_t* segs, int32_t num_segs, int32_t Hq, int32_t Hkv,
                          int32_t d, double scale, const int32_t* rows, int32_t n_rows,
                          double* out, double* lse, int32_t nthreads) {
  if (v8 == NULL) return 10;
  return attention_e4m3(q8, q_scale, k8, k_scale, NULL, v8, v_scale, cu, num_seqs, segs,
                        num_segs, Hq, Hkv, d, scale, rows, n_rows, out, lse, nthreads);
}
