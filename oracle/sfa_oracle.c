/*
 * sfa_oracle.c -- fp64 CPU oracle for sparse MLA decode (SFA) and the
 * decode-context-parallel (out, lse) merge.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA kernels are checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * What is computed (one query token t = b*Q + i, one head h):
 *
 *   L      = seq_lens[b] - (Q - 1 - i)                 causal length of token t
 *   J      = { j : 0 <= topk_idx[t, j] < L }           kept in list order (multiset)
 *   slot_j = block_table[b, p_j / bs] * bs + p_j % bs  paged latent-cache row
 *   K_j    = kv[slot_j, 0:D]      V_j = kv[slot_j, 0:DV]   (V = latent part of the row)
 *   s_j    = scale * sum_d q[t, h, d] * K_j[d]
 *   m      = max_j s_j,  l = sum_j exp(s_j - m)
 *   out    = sum_j exp(s_j - m) V_j / l,   lse = m + ln l  (natural log)
 *   J empty  ->  out = 0, lse = -inf
 *
 * Sources (page title, section):
 *  - "RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1: the MLA latent
 *    cache is [N_blk, block_size, kv_lora_rank + qk_rope_head_dim] with one
 *    latent row per token and a block_table [requests, max_blk_per_seq].
 *  - same page, symbol table in 2.1.4: Q = 1 + num_spec_tokens query tokens per
 *    step, h_kv = 1 for MLA, D = kv_lora_rank + qk_rope_head_dim.
 *  - same page, 2.1.4.2 and 2.1.4.4: the attention op returns the output and an
 *    fp32 log-sum-exp [B*Q, heads] (softmax_lse_flag=True).
 *  - same page, 1.1 and 2.1.1: DCP shards the KV along the sequence, each rank
 *    runs attention on its own shard, and the partial (out, lse) are rebuilt by
 *    an online-softmax merge; 2.1.4.3: both are upcast to fp32 first.
 *  - "vllm-ascend PR #18870 解读", 4.3 and 4.5: QK^T -> softmax -> .V is one fused
 *    step, the low-rank latent KV is shared by all heads, and sparse attention
 *    only visits the top-2048 entries chosen by the indexer.
 *  - "RFC: Context Parallel Modeling for DeepSeek-Style Attention", 3.6: the SFA
 *    operator's inputs are bf16.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - V is the first DV columns of the latent row (latent first, rope last).
 *  - lse includes the scale and uses the natural log.
 *  - Indices are logical token positions; anything outside [0, L) is padding.
 *  - Query token i of Q sees positions [0, seq_lens[b] - (Q-1-i)).
 *  - Shard r of n covers positions [r*c, (r+1)*c) of the sequence's cache with
 *    c = ceil(seq_lens[b] / n), intersected with the token's causal range.  With an
 *    interleave size g > 0 ("cp_kv_cache_interleave_size", same page 2.1.4.1: tokens
 *    are dealt to the DCP ranks g at a time), shard r instead holds the positions p
 *    of the causal range with (p / g) mod n = r.
 *  - The block table has one row per sequence, or (flattened for speculative
 *    decoding, same page 2.1.4.1) one row per query token.
 *  - Duplicate indices count once per list entry.
 *
 * Arithmetic: bf16 inputs are widened exactly to double; every sum is a plain
 * left-to-right fp64 loop.  Threads only split the (token, head) pairs; each
 * pair is computed by exactly one thread in the same order, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_NOMEM -2

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t *q, *kv;
  const int32_t *block_table, *seq_lens, *topk_idx;
  int B, Q, h, top_k, num_blocks, block_size, max_blocks_per_seq, D, DV;
  double scale;
  int interleave;     /* > 0: shard r holds positions p with (p / interleave) % n == r */
  int bt_per_token;   /* block_table has one row per query token instead of per sequence */
} problem_t;

static int check_problem(const problem_t *p) {
  if (!p->q || !p->kv || !p->block_table || !p->seq_lens || !p->topk_idx) return ORACLE_ERR_ARG;
  if (p->B < 0 || p->Q < 1 || p->h < 1 || p->top_k < 0 || p->num_blocks < 0 || p->block_size < 1 ||
      p->max_blocks_per_seq < 0 || p->D < 1 || p->DV < 1 || p->DV > p->D)
    return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Causal length of query token t (reading: token i of Q sees one more position than token i-1). */
static long causal_len(const problem_t *p, int t) {
  int b = t / p->Q, i = t % p->Q;
  return (long)p->seq_lens[b] - (long)(p->Q - 1 - i);
}

/* Physical cache row of logical position pos through block-table row `row`, or -1
 * when the table does not hold a valid block for it. */
static long slot_of(const problem_t *p, int row, long pos) {
  long blk = pos / p->block_size;
  if (blk < 0 || blk >= p->max_blocks_per_seq) return -1;
  long phys = p->block_table[(long)row * p->max_blocks_per_seq + blk];
  if (phys < 0 || phys >= p->num_blocks) return -1;
  return phys * p->block_size + pos % p->block_size;
}

/* Whether list entry pos belongs to the unit: inside [lo, hi) and, for shard r of n
 * with interleaving, dealt to shard r. */
static int in_unit(const problem_t *p, long pos, long lo, long hi, int n, int r) {
  if (pos < lo || pos >= hi) return 0;
  if (p->interleave > 0 && n > 1 && r >= 0) return (pos / p->interleave) % n == r;
  return 1;
}

/*
 * Attention of token t, head hh over the selected positions that fall in
 * [lo, hi) (already clipped to the causal range by the caller) and, with
 * interleaving, in shard r of n_sh.
 * out_row receives DV doubles; *lse_out the log-sum-exp.  Returns the number
 * of list entries used, or -1 if an entry points at a block the table lacks.
 */
static long attend(const problem_t *p, int t, int hh, long lo, long hi, int n_sh, int r, double *scores,
                   double *out_row, double *lse_out) {
  int b = p->bt_per_token ? t : t / p->Q;   /* block-table row */
  const uint16_t *qrow = p->q + ((size_t)t * p->h + hh) * p->D;
  const int32_t *idx = p->topk_idx + (size_t)t * p->top_k;
  long n = 0;
  double m = -INFINITY;
  /* scores s_j = scale * <q, K_j> for every kept entry, in list order */
  for (int j = 0; j < p->top_k; ++j) {
    long pos = idx[j];
    if (!in_unit(p, pos, lo, hi, n_sh, r)) continue;
    long slot = slot_of(p, b, pos);
    if (slot < 0) return -1;
    const uint16_t *krow = p->kv + (size_t)slot * p->D;
    double dot = 0.0;
    for (int d = 0; d < p->D; ++d) dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
    double s = p->scale * dot;
    scores[n++] = s;
    if (s > m) m = s;
  }
  for (int c = 0; c < p->DV; ++c) out_row[c] = 0.0;
  if (n == 0) {
    *lse_out = -INFINITY;
    return 0;
  }
  /* l = sum exp(s_j - m);  out = sum exp(s_j - m) V_j / l */
  double l = 0.0;
  long k = 0;
  for (int j = 0; j < p->top_k; ++j) {
    long pos = idx[j];
    if (!in_unit(p, pos, lo, hi, n_sh, r)) continue;
    long slot = slot_of(p, b, pos);
    double w = exp(scores[k++] - m);
    l += w;
    const uint16_t *vrow = p->kv + (size_t)slot * p->D;
    for (int c = 0; c < p->DV; ++c) out_row[c] += w * bf16_to_double(vrow[c]);
  }
  for (int c = 0; c < p->DV; ++c) out_row[c] /= l;
  *lse_out = m + log(l);
  return n;
}

/* ---- threading: a static split of a work list over worker threads ---- */

typedef struct {
  const problem_t *p;
  int n_splits;      /* 0 = unsplit */
  long n_items;      /* work items */
  const int32_t *item_t, *item_h, *item_r; /* optional explicit (t, h, r) lists */
  double *out, *lse; /* destinations */
  long first, last;  /* item range of this worker */
  int status;
} job_t;

static void run_item(job_t *jb, long it, double *scores) {
  const problem_t *p = jb->p;
  int t, hh, r;
  double *orow, *lrow;
  if (jb->item_t) {
    t = jb->item_t[it];
    hh = jb->item_h[it];
    r = jb->item_r ? jb->item_r[it] : -1;
    orow = jb->out + (size_t)it * p->DV;
    lrow = jb->lse + it;
  } else {
    long T = (long)p->B * p->Q;
    long per_split = T * p->h;
    r = jb->n_splits > 0 ? (int)(it / per_split) : -1;
    long rem = it % per_split;
    t = (int)(rem / p->h);
    hh = (int)(rem % p->h);
    orow = jb->out + (size_t)it * p->DV;
    lrow = jb->lse + it;
  }
  long L = causal_len(p, t);
  long lo = 0, hi = L;
  int n = jb->n_splits > 0 ? jb->n_splits : 1;
  if (r >= 0 && p->interleave <= 0) {
    /* shard r of n_splits over the sequence's cache, clipped to the causal range */
    int b = t / p->Q;
    long S = p->seq_lens[b];
    long c = S > 0 ? (S + n - 1) / n : 0;
    lo = (long)r * c;
    hi = (long)(r + 1) * c;
    if (hi > L) hi = L;
  }
  if (attend(p, t, hh, lo, hi, n, r, scores, orow, lrow) < 0) jb->status = ORACLE_ERR_ARG;
}

static void *worker(void *arg) {
  job_t *jb = (job_t *)arg;
  double *scores = (double *)malloc(sizeof(double) * (size_t)(jb->p->top_k > 0 ? jb->p->top_k : 1));
  if (!scores) {
    jb->status = ORACLE_ERR_NOMEM;
    return NULL;
  }
  for (long it = jb->first; it < jb->last; ++it) run_item(jb, it, scores);
  free(scores);
  return NULL;
}

static int run_jobs(const job_t *proto, int nthreads) {
  if (nthreads <= 0) {
    long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = ncpu > 0 ? (int)ncpu : 1;
  }
  if (nthreads > proto->n_items) nthreads = proto->n_items > 0 ? (int)proto->n_items : 1;
  job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return ORACLE_ERR_NOMEM;
  }
  long per = (proto->n_items + nthreads - 1) / nthreads;
  for (int w = 0; w < nthreads; ++w) {
    jobs[w] = *proto;
    jobs[w].first = (long)w * per;
    jobs[w].last = jobs[w].first + per < proto->n_items ? jobs[w].first + per : proto->n_items;
    if (jobs[w].first > jobs[w].last) jobs[w].first = jobs[w].last;
    jobs[w].status = ORACLE_OK;
  }
  int status = ORACLE_OK;
  int started = 0;
  for (int w = 1; w < nthreads; ++w) {
    if (pthread_create(&th[w], NULL, worker, &jobs[w]) != 0) break;
    started = w;
  }
  worker(&jobs[0]);
  for (int w = 1; w <= started; ++w) pthread_join(th[w], NULL);
  /* any worker that could not be started runs here */
  for (int w = started + 1; w < nthreads; ++w) worker(&jobs[w]);
  for (int w = 0; w < nthreads; ++w)
    if (jobs[w].status != ORACLE_OK) status = jobs[w].status;
  free(jobs);
  free(th);
  return status;
}

static problem_t make_problem(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                              const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                              int top_k, int num_blocks, int block_size, int max_blocks_per_seq, int D,
                              int DV, double scale, int interleave, int bt_per_token) {
  problem_t p;
  p.q = q;
  p.kv = kv;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.topk_idx = topk_idx;
  p.B = B;
  p.Q = Q;
  p.h = h;
  p.top_k = top_k;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.D = D;
  p.DV = DV;
  p.scale = scale;
  p.interleave = interleave;
  p.bt_per_token = bt_per_token;
  return p;
}

/*
 * Unsplit decode: out [B*Q, h, DV], lse [B*Q, h].
 */
int sfa_oracle_decode(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                      const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h, int top_k,
                      int num_blocks, int block_size, int max_blocks_per_seq, int D, int DV,
                      double scale, double *out, double *lse, int nthreads) {
  problem_t p = make_problem(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                             block_size, max_blocks_per_seq, D, DV, scale, 0, 0);
  if (check_problem(&p) != ORACLE_OK || !out || !lse) return ORACLE_ERR_ARG;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.p = &p;
  jb.n_splits = 0;
  jb.n_items = (long)B * Q * h;
  jb.out = out;
  jb.lse = lse;
  return run_jobs(&jb, nthreads);
}

/*
 * Per-shard partials (DCP emulation): out_part [n_splits, B*Q, h, DV],
 * lse_part [n_splits, B*Q, h].  Each shard is attended on its own, as each
 * DCP rank would on its slice of the sequence.
 */
int sfa_oracle_decode_splits(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                             int top_k, int num_blocks, int block_size, int max_blocks_per_seq, int D,
                             int DV, double scale, int n_splits, double *out_part, double *lse_part,
                             int nthreads) {
  problem_t p = make_problem(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                             block_size, max_blocks_per_seq, D, DV, scale, 0, 0);
  if (check_problem(&p) != ORACLE_OK || n_splits < 1 || !out_part || !lse_part) return ORACLE_ERR_ARG;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.p = &p;
  jb.n_splits = n_splits;
  jb.n_items = (long)n_splits * B * Q * h;
  jb.out = out_part;
  jb.lse = lse_part;
  return run_jobs(&jb, nthreads);
}

/*
 * The two entry points above with the layout options: per-shard partials with shards
 * interleaved `interleave` positions at a time (0 = contiguous shards), and a block
 * table with one row per query token (bt_per_token != 0).  n_splits = 1 gives the
 * unsplit result in out_part / lse_part.
 */
int sfa_oracle_decode_ex(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                         const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h, int top_k,
                         int num_blocks, int block_size, int max_blocks_per_seq, int D, int DV, double scale,
                         int n_splits, int interleave, int bt_per_token, double *out_part, double *lse_part,
                         int nthreads) {
  problem_t p = make_problem(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                             block_size, max_blocks_per_seq, D, DV, scale, interleave, bt_per_token);
  if (check_problem(&p) != ORACLE_OK || n_splits < 1 || interleave < 0 || !out_part || !lse_part)
    return ORACLE_ERR_ARG;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.p = &p;
  jb.n_splits = n_splits > 1 ? n_splits : 0;
  jb.n_items = (long)n_splits * B * Q * h;
  jb.out = out_part;
  jb.lse = lse_part;
  return run_jobs(&jb, nthreads);
}

/*
 * Selected (token, head[, shard]) pairs only, for spot checks of full-size
 * workloads.  split_r may be NULL (unsplit) or give a shard per sample, in
 * which case n_splits must be the shard count.  out [n, DV], lse [n].
 */
int sfa_oracle_decode_sampled_ex(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                                 const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                                 int top_k, int num_blocks, int block_size, int max_blocks_per_seq, int D,
                                 int DV, double scale, int n_splits, int interleave, int bt_per_token,
                                 long n_samples, const int32_t *sample_t, const int32_t *sample_h,
                                 const int32_t *sample_r, double *out, double *lse, int nthreads);

int sfa_oracle_decode_sampled(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                              const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                              int top_k, int num_blocks, int block_size, int max_blocks_per_seq, int D,
                              int DV, double scale, int n_splits, long n_samples,
                              const int32_t *sample_t, const int32_t *sample_h,
                              const int32_t *sample_r, double *out, double *lse, int nthreads) {
  return sfa_oracle_decode_sampled_ex(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                                      block_size, max_blocks_per_seq, D, DV, scale, n_splits, 0, 0, n_samples,
                                      sample_t, sample_h, sample_r, out, lse, nthreads);
}

/* The sampled entry point with the layout options of sfa_oracle_decode_ex. */
int sfa_oracle_decode_sampled_ex(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                                 const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                                 int top_k, int num_blocks, int block_size, int max_blocks_per_seq, int D,
                                 int DV, double scale, int n_splits, int interleave, int bt_per_token,
                                 long n_samples, const int32_t *sample_t, const int32_t *sample_h,
                                 const int32_t *sample_r, double *out, double *lse, int nthreads) {
  problem_t p = make_problem(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                             block_size, max_blocks_per_seq, D, DV, scale, interleave, bt_per_token);
  if (check_problem(&p) != ORACLE_OK || n_samples < 0 || interleave < 0 || !sample_t || !sample_h || !out ||
      !lse)
    return ORACLE_ERR_ARG;
  long T = (long)B * Q;
  for (long s = 0; s < n_samples; ++s) {
    if (sample_t[s] < 0 || sample_t[s] >= T || sample_h[s] < 0 || sample_h[s] >= h) return ORACLE_ERR_ARG;
    if (sample_r && (n_splits < 1 || sample_r[s] < 0 || sample_r[s] >= n_splits)) return ORACLE_ERR_ARG;
  }
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.p = &p;
  jb.n_splits = sample_r ? n_splits : 0;
  jb.n_items = n_samples;
  jb.item_t = sample_t;
  jb.item_h = sample_h;
  jb.item_r = sample_r;
  jb.out = out;
  jb.lse = lse;
  return run_jobs(&jb, nthreads);
}

/*
 * Online-softmax merge of n partial (out_r, lse_r) into (out, lse), the local
 * step after the all-to-all in "RFC: MsModeling 支持 Decode Context Parallel 仿真"
 * (1.1, 2.1.1, 2.1.4.3):
 *   M = max_r lse_r;  lse = M + ln sum_r exp(lse_r - M);
 *   out = sum_r exp(lse_r - lse) * out_r;
 *   every lse_r = -inf  ->  out = 0, lse = -inf.
 * out_part [n, rows, DV], lse_part [n, rows]; out [rows, DV], lse [rows].
 */
int sfa_oracle_merge(const double *out_part, const double *lse_part, int n, long rows, int DV,
                     double *out, double *lse) {
  if (!out_part || !lse_part || !out || !lse || n < 1 || rows < 0 || DV < 1) return ORACLE_ERR_ARG;
  for (long x = 0; x < rows; ++x) {
    double M = -INFINITY;
    for (int r = 0; r < n; ++r)
      if (lse_part[(size_t)r * rows + x] > M) M = lse_part[(size_t)r * rows + x];
    double *orow = out + (size_t)x * DV;
    for (int c = 0; c < DV; ++c) orow[c] = 0.0;
    if (M == -INFINITY) {
      lse[x] = -INFINITY;
      continue;
    }
    double Z = 0.0;
    for (int r = 0; r < n; ++r) Z += exp(lse_part[(size_t)r * rows + x] - M);
    double L = M + log(Z);
    lse[x] = L;
    for (int r = 0; r < n; ++r) {
      double w = exp(lse_part[(size_t)r * rows + x] - L);
      if (w == 0.0) continue;
      const double *prow = out_part + ((size_t)r * rows + x) * DV;
      for (int c = 0; c < DV; ++c) orow[c] += w * prow[c];
    }
  }
  return ORACLE_OK;
}

/*
 * Latent-cache write: the slot_mapping scatter by which the fused pre-attention op
 * stores each new token's latent row ("RFC: MsModeling 支持 Decode Context Parallel
 * 仿真", 2.1.4.1: slot_mapping is [total_num_tokens] int32, one physical cache slot
 * per new token; 1.3: the fused RMSNorm + QKV proj + RoPE + KV-write op writes the
 * local cache).
 *
 *   for each new token t:  slot = slot_mapping[t]
 *     slot < 0            ->  padding, nothing is written
 *     0 <= slot < slots   ->  kv[slot, 0:D] = rows[t, 0:D]   (bit copy)
 *
 * kv is the cache seen as [num_slots, D] rows (num_slots = N_blk * block_size).
 * Returns ORACLE_ERR_ARG, writing nothing, when a slot is >= num_slots or when two
 * tokens name the same slot (the write order would then decide the result).
 */
int sfa_oracle_kv_write(uint16_t *kv, long num_slots, const int32_t *slot_mapping, const uint16_t *rows,
                        long T, int D) {
  if (!kv || !slot_mapping || (!rows && T > 0) || num_slots < 0 || T < 0 || D < 1) return ORACLE_ERR_ARG;
  for (long t = 0; t < T; ++t) {
    const long s = slot_mapping[t];
    if (s >= num_slots) return ORACLE_ERR_ARG;
    if (s < 0) continue;
    for (long u = 0; u < t; ++u)
      if (slot_mapping[u] == slot_mapping[t]) return ORACLE_ERR_ARG;
  }
  for (long t = 0; t < T; ++t) {
    const long s = slot_mapping[t];
    if (s < 0) continue;
    for (int d = 0; d < D; ++d) kv[(size_t)s * D + d] = rows[(size_t)t * D + d];
  }
  return ORACLE_OK;
}

/*
 * Indexer top-k selection: the list of positions each query token attends to.
 * "vllm-ascend PR #18870 解读", 4.5: sparse attention visits only the top-2048
 * positions the indexer chose instead of the whole history.  The pages give no
 * formula for the indexer's scores, so the scores are an input here:
 *
 *   token t = b*Q + i:  L = min(S, seq_lens[b] - (Q-1-i))   (L = S without seq_lens)
 *   candidates        = positions 0 <= p < L with scores[t, p]
 *   order             = score under IEEE 754 totalOrder, larger first; equal bit
 *                       patterns: lower position first
 *   out[t, 0:n]       = the first n = min(k, L) candidates in that order, written in
 *                       ascending position;  out[t, n:k] = -1
 *
 * The tie rule and the output order are readings (the pages leave both open).
 * scores is [T, row_stride] fp32 as raw bit patterns; out is [T, k].
 */
typedef struct {
  uint32_t bits;
  int32_t pos;
} cand_t;

/* IEEE 754 totalOrder on binary32 bit patterns: the sign decides first (negatives
 * below positives, so -0 < +0); among positives a larger magnitude field is larger,
 * among negatives a larger magnitude field is smaller.  NaNs take their place by the
 * same rule: +NaN above +inf, -NaN below -inf.  Returns <0, 0, >0. */
static int total_order_cmp(uint32_t a, uint32_t b) {
  const int neg_a = (int)(a >> 31), neg_b = (int)(b >> 31);
  if (neg_a != neg_b) return neg_a ? -1 : 1;
  const uint32_t ma = a & 0x7FFFFFFFu, mb = b & 0x7FFFFFFFu;
  if (ma == mb) return 0;
  if (!neg_a) return ma < mb ? -1 : 1;
  return ma > mb ? -1 : 1;
}

/* qsort order of the candidates: larger score first, then lower position first */
static int cand_before(const void *x, const void *y) {
  const cand_t *a = (const cand_t *)x, *b = (const cand_t *)y;
  const int c = total_order_cmp(a->bits, b->bits);
  if (c != 0) return c > 0 ? -1 : 1;
  return a->pos < b->pos ? -1 : (a->pos > b->pos ? 1 : 0);
}

static int pos_ascending(const void *x, const void *y) {
  const int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
  return a < b ? -1 : (a > b ? 1 : 0);
}

typedef struct {
  const uint32_t *scores;
  long row_stride;
  const int32_t *seq_lens;
  int Q, S, k;
  int32_t *out;
  long t0, t1;
  int status;
} topk_job_t;

static void *topk_rows(void *arg) {
  topk_job_t *jb = (topk_job_t *)arg;
  cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(jb->S > 0 ? jb->S : 1));
  int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)(jb->k > 0 ? jb->k : 1));
  if (!c || !sel) {
    jb->status = ORACLE_ERR_ARG;
    free(c);
    free(sel);
    return NULL;
  }
  for (long t = jb->t0; t < jb->t1; ++t) {
    long L = jb->S;
    if (jb->seq_lens) {
      const long b = t / jb->Q, i = t % jb->Q;
      const long causal = (long)jb->seq_lens[b] - (long)(jb->Q - 1 - i);
      if (causal < L) L = causal;
    }
    if (L < 0) L = 0;
    for (long p = 0; p < L; ++p) {
      c[p].bits = jb->scores[(size_t)t * jb->row_stride + p];
      c[p].pos = (int32_t)p;
    }
    qsort(c, (size_t)L, sizeof(cand_t), cand_before);
    const long n = L < jb->k ? L : jb->k;
    for (long j = 0; j < n; ++j) sel[j] = c[j].pos;
    qsort(sel, (size_t)n, sizeof(int32_t), pos_ascending);
    int32_t *row = jb->out + (size_t)t * jb->k;
    for (long j = 0; j < jb->k; ++j) row[j] = j < n ? sel[j] : -1;
  }
  free(c);
  free(sel);
  return NULL;
}

int sfa_oracle_topk(const uint32_t *scores, long row_stride, const int32_t *seq_lens, int B, int Q, int S, int k,
                    int32_t *out, int nthreads) {
  if (!scores || !out || B < 0 || Q < 1 || S < 0 || k < 1 || row_stride < S) return ORACLE_ERR_ARG;
  const long T = (long)B * Q;
  if (T == 0) return ORACLE_OK;
  if (nthreads <= 0) {
    long nc = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = nc > 0 ? (int)nc : 1;
  }
  if (nthreads > T) nthreads = (int)T;
  if (nthreads > 256) nthreads = 256;
  topk_job_t jobs[256];
  pthread_t th[256];
  int started[256];
  for (int w = 0; w < nthreads; ++w) {
    jobs[w].scores = scores;
    jobs[w].row_stride = row_stride;
    jobs[w].seq_lens = seq_lens;
    jobs[w].Q = Q;
    jobs[w].S = S;
    jobs[w].k = k;
    jobs[w].out = out;
    jobs[w].t0 = T * w / nthreads;
    jobs[w].t1 = T * (w + 1) / nthreads;
    jobs[w].status = ORACLE_OK;
    started[w] = pthread_create(&th[w], NULL, topk_rows, &jobs[w]) == 0;
    if (!started[w]) topk_rows(&jobs[w]);
  }
  int st = ORACLE_OK;
  for (int w = 0; w < nthreads; ++w) {
    if (started[w]) pthread_join(th[w], NULL);
    if (jobs[w].status != ORACLE_OK) st = jobs[w].status;
  }
  return st;
}
