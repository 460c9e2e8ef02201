/*
 * sfa.h -- C ABI of the GB300 (sm_103a) sparse MLA decode library (libsfa.so).
 *
 * One decode step of DeepSeek-style sparse attention (SFA) over a paged MLA
 * latent KV cache, plus the online-softmax merge of per-shard (out, lse)
 * partials used by decode context parallelism (DCP).
 *
 * Conventions for every call:
 *  - Pointers marked "device" must point to memory of the current CUDA device;
 *    pointers marked "host" to host memory (pinned memory gives asynchronous
 *    copies).  The caller allocates and owns every buffer; the library never
 *    allocates, frees or keeps a pointer after a call returns, with three stated
 *    exceptions: an sfa_host_plan keeps the pointers it was created with,
 *    sfa_decode_noalloc works in a fixed device array of the library's own, and
 *    sfa_decode_host creates its helper streams and events once per device.
 *  - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 *    default stream).  Calls only enqueue work on it and return without
 *    synchronising, except sfa_last_device_status() and the host-buffer entry
 *    point's error path, which say so.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns an error code and launches nothing.  Problems only the
 *    device can see (a block-table entry outside [0, num_blocks) for a selected
 *    position, a bounded wait that ran out) are recorded in a per-device status
 *    word read by sfa_last_device_status().  The offending row is skipped,
 *    never dereferenced.
 *  - Layouts are dense, row-major, with no padding between rows.
 */
#ifndef SFA_H
#define SFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SFA_OK = 0,
  SFA_ERR_INVALID_ARG = -1,    /* null pointer, negative size, misaligned buffer, bad value   */
  SFA_ERR_UNSUPPORTED = -2,    /* valid but outside what the kernels implement (e.g. h > 128)  */
  SFA_ERR_WORKSPACE = -3,      /* workspace / staging buffer missing or too small              */
  SFA_ERR_CUDA = -4,           /* a CUDA runtime call failed (launch error, copy error)        */
  SFA_ERR_DEVICE_TIMEOUT = -5, /* a bounded device-side wait gave up (device status only)      */
  SFA_ERR_DEVICE_BAD_BLOCK = -6 /* a selected position mapped to an invalid block (device)     */
} sfa_status;

typedef void *sfa_stream; /* a cudaStream_t */

#define SFA_D_QK 576     /* kv_lora_rank (512) + qk_rope_head_dim (64) */
#define SFA_D_V 512      /* kv_lora_rank: V is the latent part of the row */
#define SFA_MAX_HEADS 128
#define SFA_MAX_SPLITS 64

/*
 * sfa_decode -- sparse attention of each query token over its selected latent
 * cache rows.
 *
 * Defined by: "RFC: MsModeling 支持 Decode Context Parallel 仿真" 2.1.4.1 (paged MLA
 * latent cache [N_blk, block_size, kv_lora_rank + qk_rope_head_dim] and block
 * table), 2.1.4.2 / 2.1.4.4 (attention output plus fp32 lse [B*Q, heads]), 1.1 and
 * 2.1.1 (KV sharded along the sequence, partial (out, lse) per shard);
 * "vllm-ascend PR #18870 解读" 4.3 / 4.5 (fused QK^T -> softmax -> .V over the
 * top-2048 selected entries, latent shared by all heads); "RFC: Context Parallel
 * Modeling for DeepSeek-Style Attention" 3.6 (bf16 SFA inputs).
 *
 * For query token t = b*Q + i (0 <= i < Q) and head hh:
 *   L_t   = seq_lens[b] - (Q - 1 - i)              (token i sees one more position than i-1)
 *   entry j is used iff 0 <= topk_idx[t, j] < L_t   (anything else, e.g. -1, is padding)
 *   row   = block_table[b, p / block_size] * block_size + p % block_size
 *   s_j   = scale * dot(q[t, hh, 0:576], kv[row, 0:576])
 *   out   = softmax(s) . kv[rows, 0:512],   lse = ln sum_j exp(s_j)   (natural log)
 *   no entry used -> out = 0, lse = -inf
 * Duplicate entries count once per list entry.
 *
 * Shards (n_splits > 1, decode context parallelism on one GPU): shard r covers
 * positions [r*c, (r+1)*c) of sequence b with c = ceil(seq_lens[b] / n_splits),
 * intersected with the token's causal range; each shard is attended on its own
 * into out_part[r], lse_part[r] (empty shard -> 0, -inf).
 *
 * Arguments:
 *   q           device, bf16 [B*Q, h, 576]
 *   kv          device, bf16 [num_blocks, block_size, 576]; V = columns 0..511
 *   block_table device, int32 [B, max_blocks_per_seq]; entries for blocks a sequence
 *               does not own are never read (any value)
 *   seq_lens    device, int32 [B]: cache length of each sequence (includes the Q new tokens)
 *   topk_idx    device, int32 [B*Q, top_k]: logical positions, -1 = padding
 *   B >= 0, Q >= 1, 1 <= h <= 128, top_k >= 0, num_blocks >= 1, block_size >= 1,
 *   max_blocks_per_seq >= 1, scale finite, 1 <= n_splits <= 64
 *   out, lse    device, fp32 [B*Q, h, 512] and [B*Q, h]: the final result.  Required
 *               when n_splits == 1.  When n_splits > 1 they may be NULL (only the
 *               partials are produced); if given, the partials are also merged
 *               into them on the same stream (as sfa_lse_merge does).
 *   out_part, lse_part  device, fp32 [n_splits, B*Q, h, 512] and [n_splits, B*Q, h];
 *               required when n_splits > 1, ignored otherwise.
 *   workspace   optional device scratch, 256-byte aligned.  With at least
 *               sfa_decode_workspace_bytes(...) bytes the kernel for 33-64 heads
 *               spreads the work of more (token, shard) units than SMs evenly over
 *               the SMs; with less (or NULL) the call runs all the same, one unit per
 *               SM at a time.  Contents need no initialisation and are undefined
 *               afterwards; calls that overlap on the GPU must not share it.
 *   All float/bf16 buffers must be 16-byte aligned.
 * Returns SFA_OK, or an error code with nothing launched.
 */
sfa_status sfa_decode(const void *q, const void *kv, const int32_t *block_table,
                      const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                      int top_k, int num_blocks, int block_size, int max_blocks_per_seq,
                      float scale, int n_splits, float *out, float *lse, float *out_part,
                      float *lse_part, void *workspace, size_t workspace_bytes,
                      sfa_stream stream);

/*
 * sfa_decode_workspace_bytes -- device scratch that lets sfa_decode balance this
 * shape over the SMs of the current device (see `workspace` above).  Nonzero only
 * when 33 <= h <= 64 and B*Q*n_splits exceeds the SM count: then 2 partial
 * results (64 x 512 fp32 and 64 (max, sum) pairs) per SM, plus one counter per
 * (token, shard) unit, each part rounded up to 256 bytes.  0 otherwise, and 0
 * while sfa_set_kernel_path selects a fixed kernel.
 */
size_t sfa_decode_workspace_bytes(int B, int Q, int h, int top_k, int n_splits);

/*
 * sfa_lse_merge -- online-softmax merge of n_splits partial results.
 *
 * Defined by: "RFC: MsModeling 支持 Decode Context Parallel 仿真" 1.1 and 2.1.1 (the
 * local online-softmax merge after the all-to-all of output and lse) and 2.1.4.3
 * (both exchanged in fp32).  For each row x:
 *   M = max_r lse_part[r, x];  lse[x] = M + ln sum_r exp(lse_part[r, x] - M)
 *   out[x, :] = sum_r exp(lse_part[r, x] - lse[x]) * out_part[r, x, :]
 *   every lse_part[r, x] = -inf  ->  out[x, :] = 0, lse[x] = -inf
 *
 *   out_part device fp32 [n_splits, rows, dv], lse_part device fp32 [n_splits, rows]
 *   out      device fp32 [rows, dv],           lse      device fp32 [rows]
 *   (for decode partials rows = B*Q*h: the (token, head) pairs are merged alike, so
 *   they are passed flattened rather than as separate token and head counts)
 *   1 <= n_splits <= 64, rows >= 0, dv >= 1; float buffers 16-byte aligned.
 *   out/lse must not overlap out_part/lse_part.
 */
sfa_status sfa_lse_merge(const float *out_part, const float *lse_part, int n_splits, int rows,
                         int dv, float *out, float *lse, sfa_stream stream);

/*
 * sfa_decode_ex -- sfa_decode with the two layout options of decode context
 * parallelism ("RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1):
 *
 *   interleave_size  0: shard r of n_splits is the contiguous range [r*c, (r+1)*c) of
 *                    the sequence's cache, c = ceil(seq_lens[b] / n_splits) (as in
 *                    sfa_decode).  g > 0: the sequence's positions are dealt to the
 *                    shards g at a time, as cp_kv_cache_interleave_size deals them to
 *                    the DCP ranks: shard r holds the positions p with (p / g) % n_splits
 *                    == r.  Either way each shard is clipped to the token's causal range
 *                    and the merged result is the same (up to rounding).
 *   flags            SFA_BLOCK_TABLE_PER_TOKEN: block_table is [B*Q, max_blocks_per_seq],
 *                    one row per query token (the table flattened for speculative
 *                    decoding); otherwise [B, max_blocks_per_seq], one row per sequence.
 *
 * Every other argument, and the return codes, as in sfa_decode.  interleave_size < 0 or
 * an unknown flag bit returns SFA_ERR_INVALID_ARG.
 */
#define SFA_BLOCK_TABLE_PER_TOKEN 1
sfa_status sfa_decode_ex(const void *q, const void *kv, const int32_t *block_table, const int32_t *seq_lens,
                         const int32_t *topk_idx, int B, int Q, int h, int top_k, int num_blocks, int block_size,
                         int max_blocks_per_seq, float scale, int n_splits, int interleave_size, int flags,
                         float *out, float *lse, float *out_part, float *lse_part, void *workspace,
                         size_t workspace_bytes, sfa_stream stream);

/*
 * sfa_topk -- the indexer's top-k selection: for each query token, the positions of the
 * k largest indexer scores, the list sparse attention then visits ("vllm-ascend PR
 * #18870 解读", 4.5: only the top-2048 positions chosen by the indexer are attended).
 * The pages give no formula for the scores themselves; they are an input here.
 *
 *   scores      device fp32 [B*Q, row_stride]: row t holds the scores of positions 0..S-1
 *               of token t's sequence (columns S..row_stride-1 are never read);
 *               16-byte aligned, row_stride >= S and a multiple of 4
 *   seq_lens    device int32 [B] or NULL: token t = b*Q + i chooses among the positions
 *               [0, min(S, seq_lens[b] - (Q-1-i))) (the causal range sfa_decode uses);
 *               NULL: among [0, S)
 *   topk_idx    device int32 [B*Q, k], written: the chosen positions in ascending order,
 *               then -1 where fewer than k positions are candidates -- the layout
 *               sfa_decode reads
 *
 * The positions chosen are those of the k largest scores under IEEE 754 totalOrder
 * (-0 below +0; a NaN with the sign bit clear above +inf); among equal scores the lower
 * positions are chosen first.  1 <= k; 0 <= S <= SFA_TOPK_MAX_S.
 * Returns SFA_OK, SFA_ERR_INVALID_ARG (bad sizes, stride, alignment or NULL buffers) or
 * SFA_ERR_UNSUPPORTED (S above SFA_TOPK_MAX_S); nothing is launched on an error.
 */
#define SFA_TOPK_MAX_S 262144
sfa_status sfa_topk(const float *scores, long long row_stride, const int32_t *seq_lens, int B, int Q, int S, int k,
                    int32_t *topk_idx, sfa_stream stream);

/*
 * sfa_kv_write -- the latent-cache write that precedes attention: each new token's
 * latent row (kv_lora_rank + qk_rope_head_dim = 576 bf16) is stored at the cache slot
 * slot_mapping[t] ("RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1:
 * slot_mapping [total_num_tokens] int32; 1.3: the fused pre-attention op writes the
 * KV).  A slot is block * block_size + offset, i.e. a row of the cache seen as
 * [num_blocks * block_size, 576].
 *
 *   kv            device bf16 [num_blocks, block_size, 576] (num_slots rows), written in place
 *   slot_mapping  device int32 [T]: the slot of each new token; < 0 = padding (skipped)
 *   rows          device bf16 [T, 576]: the new latent rows
 *   T >= 0, num_slots >= 0; kv and rows 16-byte aligned.
 * Two tokens naming the same slot write it concurrently: the slot ends up holding parts
 * of their rows, which parts is not defined (a slot mapping names each slot once).  A
 * slot >= num_slots writes nothing and sets SFA_ERR_DEVICE_BAD_BLOCK in
 * the device status word.  Returns SFA_OK or a host-side argument error, nothing launched.
 */
sfa_status sfa_kv_write(void *kv, long long num_slots, const int32_t *slot_mapping, const void *rows, int T,
                        sfa_stream stream);

/*
 * sfa_uv_proj -- the W_UV up-projection that follows attention in the latent space:
 *   y[t, h, v] = sum_{c < 512} out[t, h, c] * w_uv[h, c, v],   v < 128
 * (MLA attends over the 512-wide latent; W_UV, derived from kv_b_proj, takes each head's
 * output to its 128-wide value space: "RFC: Context Parallel Modeling for
 * DeepSeek-Style Attention", 3.5).  A tcgen05 contraction per (head, 64 tokens).
 *
 *   out   device fp32 [T, h, 512] (sfa_decode's out); rounded to bf16 for the tensor cores
 *   w_uv  device bf16 [h, 512, 128]
 *   y     device bf16 [T, h, 128]
 *   T >= 0, 1 <= h <= 65535; out and w_uv 16-byte aligned, y 2-byte aligned.
 * Accuracy: |y - exact| <= 2^-8 * sum_c |out[c] * w[c, v]| + 2^-8 * |exact| (bf16 inputs,
 * fp32 accumulation, bf16 result).  A bounded wait that gives up sets
 * SFA_ERR_DEVICE_TIMEOUT in the device status word.  Returns SFA_OK or a host-side error.
 */
sfa_status sfa_uv_proj(const float *out, const void *w_uv, void *y, int T, int h, sfa_stream stream);

/*
 * sfa_decode_host -- one decode step whose per-step inputs and outputs live in
 * host memory, with the latent cache resident on the device (the form a serving
 * loop that keeps its cache in HBM uses).  Enqueues on `stream`: host->device
 * copies of q, block_table, seq_lens and topk_idx into `staging`, sfa_decode,
 * and device->host copies of out and lse.  The caller synchronises the stream
 * before reading out_host / lse_host.
 *
 *   q_host, block_table_host, seq_lens_host, topk_idx_host: host, layouts as in sfa_decode
 *   kv           device, as in sfa_decode
 *   out_host, lse_host: host fp32 [B*Q, h, 512] and [B*Q, h] (the merged result)
 *   staging      device scratch of at least sfa_decode_host_staging_bytes(...) bytes,
 *                256-byte aligned; holds the device copies, partials and workspace.
 * Host buffers must stay valid until the stream reaches the end of the copies.
 *
 * A batch whose out is at least 4 MiB is processed as up to 4 groups of whole
 * sequences.  Each group runs on a helper stream that the library creates once per
 * device, forked from `stream` by an event and joined back into it, so the call stays
 * ordered on `stream`.  A group's result copies overlap later groups' input copies
 * and kernels.  Calls from several host threads take turns at enqueueing (a mutex),
 * and their groups share the helper streams.  If an error is returned after some
 * groups were enqueued, that work may still run.
 */
size_t sfa_decode_host_staging_bytes(int B, int Q, int h, int top_k, int max_blocks_per_seq,
                                     int n_splits);
sfa_status sfa_decode_host(const void *q_host, const void *kv, const int32_t *block_table_host,
                           const int32_t *seq_lens_host, const int32_t *topk_idx_host, int B,
                           int Q, int h, int top_k, int num_blocks, int block_size,
                           int max_blocks_per_seq, float scale, int n_splits, float *out_host,
                           float *lse_host, void *staging, size_t staging_bytes,
                           sfa_stream stream);

/*
 * sfa_host_plan -- one sfa_decode_host step captured as a CUDA graph, for a serving loop
 * that calls it with the same buffers every step: the ~20 copies, launches and stream
 * joins of a step then cost one graph launch on the host instead of being enqueued one
 * by one (the host side of a step otherwise takes longer than the copy engines need).
 *
 *   sfa_host_plan_create  records the step exactly as sfa_decode_host with the same
 *                         arguments would enqueue it (same checks and return codes; nothing
 *                         runs).  The host buffers must be page-locked (pinned); a failed
 *                         capture returns SFA_ERR_CUDA and a NULL `plan` SFA_ERR_INVALID_ARG;
 *                         *plan is NULL unless SFA_OK.  The plan keeps the pointers: every launch copies q,
 *                         block_table, seq_lens and topk_idx in from those host buffers as
 *                         they are at that moment and writes out and lse back to theirs, so
 *                         the caller refills the inputs between launches.  The buffers must
 *                         outlive the plan; staging must not be used by anything else while
 *                         a launch may be in flight.
 *   sfa_host_plan_launch  enqueues one step on `stream` (asynchronous, like sfa_decode_host).
 *   sfa_host_plan_destroy releases the plan (NULL is ignored); no launch may be in flight.
 */
typedef struct sfa_host_plan_s *sfa_host_plan;
sfa_status sfa_host_plan_create(const void *q_host, const void *kv, const int32_t *block_table_host,
                                const int32_t *seq_lens_host, const int32_t *topk_idx_host, int B, int Q, int h,
                                int top_k, int num_blocks, int block_size, int max_blocks_per_seq, float scale,
                                int n_splits, float *out_host, float *lse_host, void *staging,
                                size_t staging_bytes, sfa_host_plan *plan);
sfa_status sfa_host_plan_launch(sfa_host_plan plan, sfa_stream stream);
void sfa_host_plan_destroy(sfa_host_plan plan);

/*
 * sfa_last_device_status -- synchronises `stream`, then returns and clears the
 * current device's status word: SFA_OK, SFA_ERR_DEVICE_TIMEOUT (a bounded wait
 * inside a kernel gave up; that kernel's outputs are undefined) or
 * SFA_ERR_DEVICE_BAD_BLOCK (a selected position's block-table entry was outside
 * [0, num_blocks); that row was skipped).  SFA_ERR_CUDA if the stream itself failed.
 */
sfa_status sfa_last_device_status(sfa_stream stream);

/*
 * sfa_decode_noalloc -- sfa_decode followed by the shard merge, for callers that
 * cannot allocate device memory.  No passage of the source pages corresponds to
 * it: it exists for deployments, not for the method.
 *
 * Some callers have no allocator: an engine that hands all free HBM to its cache
 * pool at start-up, a plugin host that passes a library only its inputs and
 * outputs, or a decode loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.  This entry point takes only the inputs and the final out/lse
 * (layouts, alignment and argument rules as in sfa_decode; out and lse are
 * required for every n_splits) and keeps the shard partials and any workspace in
 * a fixed device array of SFA_NOALLOC_SCRATCH_BYTES that the library owns.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Limit: a call whose partials (n_splits > 1: n_splits*B*Q*h*513 floats, each
 *    part rounded up to 256 bytes) plus workspace exceed SFA_NOALLOC_SCRATCH_BYTES
 *    returns SFA_ERR_WORKSPACE and launches nothing.
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The first call on each device looks the array's address up (with that
 *    device current); make that first call before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (other streams,
 *    other threads) race.  Each call writes all the scratch it reads, so no
 *    clearing between calls is needed.
 *  - A call with n_splits == 1 uses no scratch and does not look the array up.
 *  - The looked-up address is cached per device for the life of the process; it is
 *    not valid after a device reset (cudaDeviceReset), so no call may follow one.
 *  - out or lse NULL returns SFA_ERR_INVALID_ARG before any other check.
 */
#define SFA_NOALLOC_SCRATCH_BYTES (72u << 20)
sfa_status sfa_decode_noalloc(const void *q, const void *kv, const int32_t *block_table,
                              const int32_t *seq_lens, const int32_t *topk_idx, int B, int Q, int h,
                              int top_k, int num_blocks, int block_size, int max_blocks_per_seq,
                              float scale, int n_splits, float *out, float *lse, sfa_stream stream);

/*
 * sfa_decode_launches -- how many kernels one sfa_decode call with these
 * arguments enqueues (merge != 0: out/lse given with n_splits > 1), and through
 * *tensor_core_path which kernel serves it: 2 = the small-head tcgen05 kernel
 * (h <= 32), 3 = the stacked-half tcgen05 kernel (33 <= h <= 64), 1 = the CTA-pair
 * tcgen05 kernel, 0 = the CUDA-core kernel.
 * tensor_core_path may be NULL.  Returns -1 for invalid arguments.
 */
int sfa_decode_launches(int B, int Q, int h, int top_k, int block_size, int n_splits, int merge,
                        int *tensor_core_path);

/*
 * sfa_set_kernel_path -- kernel family for sfa_decode calls made afterwards in
 * this process: 0 = automatic (the small-head tcgen05 kernel for h <= 32, the
 * stacked-half tcgen05 kernel for 33 <= h <= 64, the CTA-pair tcgen05 kernel
 * above), 1 = the CUDA-core kernel for every shape, 2 = the
 * CTA-pair tcgen05 kernel for every shape.  Paths 1 and 2 exist to cross-check the
 * kernels against each other.  Returns the previous setting, or -1 (and changes
 * nothing) for another value.
 */
int sfa_set_kernel_path(int path);

/* sfa_status_string -- static, human-readable name of a status code. */
const char *sfa_status_string(sfa_status s);

/*
 * sfa_set_wait_limit -- test hook for the failure path: sets the iteration cap
 * of every bounded device-side wait in kernels launched afterwards from this
 * process (0 restores the default).  With a tiny cap a wait gives up early and
 * the kernel reports SFA_ERR_DEVICE_TIMEOUT through sfa_last_device_status()
 * instead of hanging.  Returns the previous cap.
 */
long long sfa_set_wait_limit(long long iterations);

/*
 * sfa_set_stall_injection -- test hook for the failure path: with on != 0, the
 * kernels with bounded waits (the tcgen05 decode kernel and sfa_uv_proj) launched
 * afterwards from this process first wait on a barrier that nothing ever completes.
 * That wait runs out after the wait limit (sfa_set_wait_limit), the kernel records
 * SFA_ERR_DEVICE_TIMEOUT, drains its own copies and matrix operations and returns:
 * nothing faults, traps or hangs, and the context stays usable.  Returns the
 * previous setting.
 */
int sfa_set_stall_injection(int on);

#ifdef __cplusplus
}
#endif
#endif /* SFA_H */
