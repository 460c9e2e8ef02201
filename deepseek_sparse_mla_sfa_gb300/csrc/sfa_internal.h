// sfa_internal.h -- declarations shared by the translation units of libsfa.so.
// Not part of the public ABI (that is include/sfa.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sfa {

constexpr int kDQK = 576;  // kv_lora_rank + qk_rope_head_dim
constexpr int kDV = 512;   // kv_lora_rank
constexpr int kMaxHeads = 128;
constexpr int kMaxSplits = 64;
constexpr int kTopkChunkMax = 32768;                  // candidate positions one top-k CTA holds
constexpr int kTopkMaxS = 8 * kTopkChunkMax;          // a cluster of at most 8 CTAs per token

// Device status codes (mirror sfa_status values).
constexpr int kStatusTimeout = -5;
constexpr int kStatusBadBlock = -6;

// One decode problem as the kernels see it.  Pointers are device pointers.
struct DecodeParams {
  const __nv_bfloat16* q;    // [T, h, 576]
  const __nv_bfloat16* kv;   // [num_blocks, block_size, 576]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* seq_lens;     // [B]
  const int32_t* topk_idx;     // [T, top_k]
  int B, Q, h, top_k, num_blocks, block_size, max_blocks;
  float scale;
  int n_splits;
  float* out;  // n_splits == 1: [T, h, 512]; else partials [n_splits, T, h, 512]
  float* lse;  // n_splits == 1: [T, h];      else partials [n_splits, T, h]
  void* workspace;
  size_t workspace_bytes;
  int* status;            // per-device status word
  long long wait_limit;   // iteration cap of every bounded device wait
  int interleave;         // > 0: shard r holds positions p with (p / interleave) % n_splits == r
  int bt_per_token;       // block_table has one row per query token (else one per sequence)
  int stall;              // test hook: first wait on a barrier that nothing completes
};

// Record the first device-side error in the status word (never traps).
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Shard bounds of sequence `seq_len` for shard r of n (n == 1: the whole cache),
// intersected with the causal range [0, L).
__host__ __device__ __forceinline__ void shard_bounds(int seq_len, int L, int r, int n, int& lo,
                                                      int& hi) {
  if (n <= 1) {
    lo = 0;
    hi = L;
    return;
  }
  int c = seq_len > 0 ? (seq_len + n - 1) / n : 0;
  long long l = (long long)r * c, u = (long long)(r + 1) * c;
  if (u > L) u = L;
  lo = (int)(l > 0x7fffffff ? 0x7fffffff : l);
  hi = (int)(u < lo ? lo : u);
}

// The positions one work unit (token t, shard r) attends to.  Contiguous shards:
// [lo, hi) = shard r of the sequence's cache clipped to the causal range.  Interleaved
// shards (interleave = g > 0, as DCP deals a sequence's tokens to its ranks g at a
// time): the whole causal range [0, L), keeping the positions p with (p / g) % n == r.
struct ShardSel {
  int lo, hi, g, n, r;
  __host__ __device__ __forceinline__ bool has(int pos) const {
    return pos >= lo && pos < hi && (g <= 0 || (pos / g) % n == r);
  }
  // the same test with the layout fixed at compile time (kInterleaved == (g > 0)), for
  // loops that branch on the layout once instead of once per entry
  template <bool kInterleaved>
  __host__ __device__ __forceinline__ bool has_fixed(int pos) const {
    return pos >= lo && pos < hi && (!kInterleaved || (pos / g) % n == r);
  }
};
__host__ __device__ __forceinline__ ShardSel shard_sel(int seq_len, int L, int r, int n, int interleave) {
  ShardSel s;
  s.n = n;
  s.r = r;
  s.g = n > 1 ? interleave : 0;
  if (s.g > 0) {
    s.lo = 0;
    s.hi = L > 0 ? L : 0;
  } else {
    shard_bounds(seq_len, L, r, n, s.lo, s.hi);
  }
  return s;
}

// Launchers (return the launch error, if any).
cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream);
// One-time per-device kernel attributes (shared-memory size), set outside any stream
// capture; the launchers call them too.
cudaError_t prepare_decode_simt();
cudaError_t prepare_decode_tc();
cudaError_t launch_uv_proj(const float* out, const void* w_uv, void* y, int T, int h, long long wait_limit,
                           int stall, int* status, cudaStream_t stream);
// Indexer top-k: cluster size C (CTAs per query token), positions per CTA and threads
// per CTA for T tokens over S candidate positions on a GPU with n_sms SMs.
void topk_plan(int T, int S, int n_sms, int& C, int& chunk, int& threads);
cudaError_t launch_topk(const float* scores, long long row_stride, const int32_t* seq_lens, int B, int Q, int S,
                        int k, int32_t* out, cudaStream_t stream);
cudaError_t launch_kv_write(void* kv, long long num_slots, const int32_t* slot_mapping, const void* rows, int T,
                            int* status, cudaStream_t stream);
cudaError_t launch_lse_merge(const float* out_part, const float* lse_part, int n_splits, int rows,
                             int dv, float* out, float* lse, cudaStream_t stream);

// tcgen05 path: whether it handles this problem, its workspace, and its launch.  Three
// kernels: the CTA-pair kernel (any h <= 128), the small-head kernel (h <= 32) and the
// stacked-half kernel (33 <= h <= 64).
bool tc_supports(int h, int block_size);
// the tcgen05 path also needs 16-byte aligned q, kv and out (TMA tensor maps)
bool tc_supports_ptrs(const void* q, const void* kv, const void* out);
size_t tc_workspace_bytes(int T, int h, int top_k, int n_splits);
int tc_launches(int T, int h, int top_k, int n_splits);
// kernel: 1 = CTA pair, 2 = small head, 3 = stacked halves
cudaError_t launch_decode_tc(const DecodeParams& p, int kernel, cudaStream_t stream);
// the small-head kernel (sfa_narrow.cu): heads it serves, its one-time set-up, its
// cluster size for `units` (token, shard) units on n_sms SMs, and its launch with the
// cache-row map (64 columns x 1 row, 128-byte swizzle) and q's rope map (64 columns x h)
bool narrow_supports(int h);
cudaError_t prepare_decode_narrow();
int narrow_cluster_size(long long units, int n_sms);
cudaError_t launch_decode_narrow(const DecodeParams& p, const CUtensorMap& rows_map, const CUtensorMap& qrope_map,
                                 cudaStream_t stream);
// the stacked-half kernel (sfa_stack.cu, 33 <= h <= 64): the same maps (q's rope map with
// boxes of 16 heads) and the output map (32 columns x h heads), one CTA (or a cluster of
// 2 or 4 when units are few) per unit
bool stack_supports(int h);
// workspace that lets the stacked-half kernel balance `units` units over n_sms SMs (0 when
// it would not: other head counts, or no more units than SMs)
size_t stack_workspace_bytes(long long units, int h, int top_k, int n_sms);
cudaError_t prepare_decode_stack();
cudaError_t launch_decode_stack(const DecodeParams& p, const CUtensorMap& rows_map, const CUtensorMap& qrope_map,
                                const CUtensorMap& out_map, int n_sms, cudaStream_t stream);
// SM count of the current device (looked up once per device)
int device_sm_count();

}  // namespace sfa
