/*
 * kpool_oracle.c -- plain CPU oracle for KPool DSA indexer selection.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no code, header or constant with the CUDA
 * library, and it is written to be read against the pages by eye: no
 * blocking, no fusion, no reordering beyond what the definition states.
 *
 * What it computes (one function per step, each citing where it comes from):
 *   1. pool    -- kpool consecutive index keys of a sequence form one pool
 *                 ("spark_model/layers/glm5next_dsa/tp.rs", module docs,
 *                 "Why the indexer is REPLICATED": n_pools = seq / kpool).
 *                 The pages never name the pooling operator; this oracle
 *                 takes the MEAN (an explicit assumption): an fp32 sum in
 *                 increasing key order, one IEEE fp32 division by kpool, then
 *                 round-to-nearest-even to the input dtype (bf16 inputs give
 *                 bf16 pooled keys, fp32 inputs stay fp32).
 *   2. score   -- s[t,p] = sum_h w[t,h] * relu(scale * q[t,h,:] . kpool[p,:]),
 *                 a plain head sum taken before any top-k (same page, same
 *                 section: index_scores accumulates weights[h] *
 *                 relu(scale . dot) over heads). Computed in fp64 from the
 *                 exact input values.
 *   3. select  -- row t (sequence-local) may use the complete pools whose last
 *                 token is <= t: p < e_t = floor((t+1)/kpool). It keeps the
 *                 first budget = index_topk/kpool of them under the order
 *                 "higher score first, then smaller pool index" (tp.rs module
 *                 docs: the deterministic tiebreak pinned because torch.topk's
 *                 tie order is undefined). Unused slots hold -1. Rows are
 *                 independent of one another ("NVIDIA/Megatron-LM pull request
 *                 #8299", section "Mechanism").
 *   4. expand  -- pool expansion, tail append and mask filtering (Megatron-LM
 *                 #8299, section "Change"): slot j*kpool+r holds
 *                 pool_ids[j]*kpool + r; the tail slots index_topk + r hold
 *                 e_t*kpool + r for r < (t+1) mod kpool (the row's own
 *                 incomplete trailing pool); any token id beyond the row or
 *                 the sequence becomes -1.
 *
 * Indices are sequence-local (pool ids count from the sequence's first pool,
 * token ids from the sequence's first token); sequences come packed (THD)
 * with cumulative lengths cu_seqlens (Megatron-LM #8299, "Test plan": packed
 * THD with cu_seqlens_kv and varlen bounds).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (fp-contract off so
 * that the fp32 pooling sum is the plain sequence of IEEE additions).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_F32 1

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* ---- element access -------------------------------------------------- */

static float bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round an fp32 value to the nearest bf16, ties to even (IEEE RNE on the
   upper 16 bits). Inputs here are finite. */
static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lower = u & 0xFFFFu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

static float load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == ORACLE_BF16) return bf16_to_float(((const uint16_t*)base)[i]);
  return ((const float*)base)[i];
}

/* ---- step 1: pooling -------------------------------------------------- */

/* Pool offsets: pool_off[b] = sum_{j<b} floor(L_j / kpool). */
int kpool_oracle_pool_offsets(const int32_t* cu_seqlens, int num_seqs, int kpool,
                              int64_t* pool_off) {
  if (num_seqs < 0 || kpool < 1) return ORACLE_BAD_ARG;
  pool_off[0] = 0;
  for (int b = 0; b < num_seqs; ++b) {
    int64_t len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
    if (len < 0) return ORACLE_BAD_ARG;
    pool_off[b + 1] = pool_off[b] + len / kpool;
  }
  return ORACLE_OK;
}

/* Mean-pooled keys, as float values already rounded to the input dtype.
   k is [T, d] in dtype; out_kp is [P, d] with P = pool_off[num_seqs]. */
int kpool_oracle_pool(const void* k, int dtype, const int32_t* cu_seqlens, int num_seqs,
                      int head_dim, int kpool, float* out_kp) {
  if (kpool < 1 || head_dim < 1) return ORACLE_BAD_ARG;
  int64_t out_row = 0;
  for (int b = 0; b < num_seqs; ++b) {
    int64_t start = cu_seqlens[b];
    int64_t len = (int64_t)cu_seqlens[b + 1] - start;
    int64_t n_pools = len / kpool;
    for (int64_t p = 0; p < n_pools; ++p, ++out_row) {
      for (int c = 0; c < head_dim; ++c) {
        float sum = 0.0f;
        for (int j = 0; j < kpool; ++j)
          sum += load_elem(k, dtype, (start + p * kpool + j) * head_dim + c);
        float mean = sum / (float)kpool;
        if (dtype == ORACLE_BF16) mean = bf16_to_float(float_to_bf16_rne(mean));
        out_kp[out_row * head_dim + c] = mean;
      }
    }
  }
  return ORACLE_OK;
}

/* Gated pooling: a second pooling operator, a stated reading of parameters the
   pages name without a formula. The GLM-5.3 DSA shard plan lists
   indexer.index_kpool_compress_gate, shaped [index_head_dim, hidden] (one gate
   score per token and key channel), and indexer.index_kpool_compress_ape,
   shaped [kpool, index_head_dim] (one vector per position inside a pool)
   ("spark_model/layers/glm5next_dsa/tp.rs", the indexer parameter list), and
   the Megatron change passes "gate scores" to the fused top-k ("NVIDIA/Megatron-
   LM pull request #8299", section "Mechanism"). Read as gated compression: per
   pool and channel, a softmax over the pool's kpool positions of the tokens'
   gate scores weights the keys plus their position embedding,
       kp[p,c] = sum_j softmax_j(gate[t_j,c]) * (k[t_j,c] + ape[j,c]),
   t_j = start + p*kpool + j. Computed in fp64 (max-subtracted softmax), then
   rounded to fp32 and, for bf16 inputs, to bf16 (round to nearest even).
   gate is [T, d] fp32, ape is [kpool, d] fp32. */
int kpool_oracle_pool_gated(const void* k, int dtype, const float* gate, const float* ape,
                            const int32_t* cu_seqlens, int num_seqs, int head_dim, int kpool,
                            float* out_kp) {
  if (kpool < 1 || head_dim < 1) return ORACLE_BAD_ARG;
  int64_t out_row = 0;
  for (int b = 0; b < num_seqs; ++b) {
    int64_t start = cu_seqlens[b];
    int64_t len = (int64_t)cu_seqlens[b + 1] - start;
    int64_t n_pools = len / kpool;
    for (int64_t p = 0; p < n_pools; ++p, ++out_row) {
      for (int c = 0; c < head_dim; ++c) {
        int64_t t0 = start + p * kpool;
        double m = -INFINITY;
        for (int j = 0; j < kpool; ++j) {
          double g = gate[(t0 + j) * head_dim + c];
          if (g > m) m = g;
        }
        double den = 0.0;
        for (int j = 0; j < kpool; ++j) den += exp((double)gate[(t0 + j) * head_dim + c] - m);
        double v = 0.0;
        for (int j = 0; j < kpool; ++j) {
          double wj = exp((double)gate[(t0 + j) * head_dim + c] - m) / den;
          v += wj * ((double)load_elem(k, dtype, (t0 + j) * head_dim + c) + (double)ape[(int64_t)j * head_dim + c]);
        }
        float f = (float)v;
        if (dtype == ORACLE_BF16) f = bf16_to_float(float_to_bf16_rne(f));
        out_kp[out_row * head_dim + c] = f;
      }
    }
  }
  return ORACLE_OK;
}

/* ---- step 2: score ------------------------------------------------------ */

/* s = sum_h w[h] * max(0, scale * (q[h,:] . kp[:])), all in fp64.
   q_row is [H, d] in dtype, w_row is [H] fp32, kp_row is [d]. */
double kpool_oracle_score(const void* q_row, int dtype, const float* w_row,
                          const float* kp_row, int heads, int head_dim, float scale) {
  double s = 0.0;
  for (int h = 0; h < heads; ++h) {
    double dot = 0.0;
    for (int c = 0; c < head_dim; ++c)
      dot += (double)load_elem(q_row, dtype, (int64_t)h * head_dim + c) * (double)kp_row[c];
    double v = (double)scale * dot;
    if (v < 0.0) v = 0.0;
    s += (double)w_row[h] * v;
  }
  return s;
}

/* ---- step 3: select ----------------------------------------------------- */

typedef struct {
  double score;
  int64_t pool;
} scored_pool;

/* Higher score first; equal scores: smaller pool index first. */
static int by_score_then_index(const void* a, const void* b) {
  const scored_pool* x = (const scored_pool*)a;
  const scored_pool* y = (const scored_pool*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  if (x->pool < y->pool) return -1;
  if (x->pool > y->pool) return 1;
  return 0;
}

/* Sequence that holds global token row `row`; cu_seqlens is nondecreasing and
   0 <= row < cu_seqlens[num_seqs], so empty sequences are stepped over. */
static int seq_of_row(const int32_t* cu_seqlens, int num_seqs, int64_t row) {
  int b = 0;
  while (b + 1 < num_seqs && row >= cu_seqlens[b + 1]) ++b;
  return b;
}

/*
 * Selection for a list of global token rows.
 *   q_rows   [nrows, H, d] dtype   -- the query of each listed row
 *   w_rows   [nrows, H]    fp32    -- the head weights of each listed row
 *   kp       [P, d]        fp32    -- pooled keys from kpool_oracle_pool
 *   rows     [nrows]               -- global token index of each row
 * Outputs (each row-major per listed row):
 *   out_pool_ids  [nrows, B] int32, -1 padded
 *   out_token_ids [nrows, index_topk + kpool] int32, -1 padded
 *   out_scores    [nrows, B] fp64 (NaN where the pool id is -1); may be NULL
 *   out_eligible  [nrows] int64 (e_t); may be NULL
 */
int kpool_oracle_select(const void* q_rows, const float* w_rows, const float* kp,
                        const int32_t* cu_seqlens, int num_seqs, int heads, int head_dim,
                        int dtype, int kpool, int index_topk, float scale,
                        const int64_t* rows, int64_t nrows, int32_t* out_pool_ids,
                        int32_t* out_token_ids, double* out_scores, int64_t* out_eligible) {
  if (kpool < 1 || index_topk < 0 || index_topk % kpool != 0 || heads < 1 || head_dim < 1)
    return ORACLE_BAD_ARG;
  if (dtype != ORACLE_BF16 && dtype != ORACLE_F32) return ORACLE_BAD_ARG;
  const int64_t budget = index_topk / kpool;
  const int64_t width = (int64_t)index_topk + kpool;
  const int64_t total = num_seqs > 0 ? cu_seqlens[num_seqs] : 0;

  int64_t* pool_off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
  if (!pool_off) return ORACLE_BAD_ARG;
  if (kpool_oracle_pool_offsets(cu_seqlens, num_seqs, kpool, pool_off) != ORACLE_OK) {
    free(pool_off);
    return ORACLE_BAD_ARG;
  }
  for (int64_t i = 0; i < nrows; ++i)
    if (rows[i] < 0 || rows[i] >= total) {
      free(pool_off);
      return ORACLE_BAD_ARG;
    }

  const size_t q_row_elems = (size_t)heads * (size_t)head_dim;
  const size_t elem_bytes = dtype == ORACLE_BF16 ? 2 : 4;
  int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t row = rows[i];
    const int b = seq_of_row(cu_seqlens, num_seqs, row);
    const int64_t start = cu_seqlens[b];
    const int64_t len = (int64_t)cu_seqlens[b + 1] - start;
    const int64_t t = row - start;          /* sequence-local row */
    const int64_t eligible = (t + 1) / kpool; /* complete pools ending at or before t */
    const void* q_row = (const char*)q_rows + (size_t)i * q_row_elems * elem_bytes;
    const float* w_row = w_rows + (size_t)i * (size_t)heads;

    scored_pool* cand = NULL;
    if (eligible > 0) {
      cand = (scored_pool*)malloc(sizeof(scored_pool) * (size_t)eligible);
      if (!cand) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
    }
    for (int64_t p = 0; p < eligible; ++p) {
      cand[p].pool = p;
      cand[p].score = kpool_oracle_score(q_row, dtype, w_row,
                                         kp + (size_t)(pool_off[b] + p) * (size_t)head_dim,
                                         heads, head_dim, scale);
    }
    if (eligible > 1) qsort(cand, (size_t)eligible, sizeof(scored_pool), by_score_then_index);

    const int64_t kept = eligible < budget ? eligible : budget;
    int32_t* ids = out_pool_ids + (size_t)i * (size_t)budget;
    for (int64_t j = 0; j < budget; ++j) ids[j] = j < kept ? (int32_t)cand[j].pool : -1;
    if (out_scores) {
      double* sc = out_scores + (size_t)i * (size_t)budget;
      for (int64_t j = 0; j < budget; ++j) sc[j] = j < kept ? cand[j].score : NAN;
    }
    if (out_eligible) out_eligible[i] = eligible;

    /* step 4: expansion, tail append, mask filtering */
    int32_t* tok = out_token_ids + (size_t)i * (size_t)width;
    for (int64_t j = 0; j < budget; ++j)
      for (int r = 0; r < kpool; ++r)
        tok[j * kpool + r] = ids[j] >= 0 ? (int32_t)((int64_t)ids[j] * kpool + r) : -1;
    const int64_t tail_len = (t + 1) % kpool;
    for (int r = 0; r < kpool; ++r)
      tok[budget * kpool + r] = r < tail_len ? (int32_t)(eligible * kpool + r) : -1;
    for (int64_t s = 0; s < width; ++s)
      if (tok[s] > t || tok[s] >= len) tok[s] = -1;

    free(cand);
  }
  free(pool_off);
  return failed ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* Threads the OpenMP runtime will use (for reporting the CPU baseline). */
int kpool_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
