// sfa_api.cu -- the C ABI of libsfa.so (declared in include/sfa.h): argument
// checks, kernel selection, the per-device status word and the host-buffer
// entry point.  Every step of the computation runs in this library's kernels.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <climits>

#include "sfa.h"
#include "sfa_internal.h"

namespace {

// Per-device status word written by kernels (first error wins), read and
// cleared by sfa_last_device_status().
__device__ int g_sfa_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
std::atomic<long long> g_wait_limit{0};
std::atomic<int> g_kernel_path{0};  // 0 automatic, 1 CUDA-core only, 2 CTA-pair tcgen05 for every h
std::atomic<int> g_stall{0};        // test hook: kernels first wait on a barrier nothing completes

// 0: CUDA-core kernel, 1: CTA-pair tcgen05 kernel, 2: small-head tcgen05 kernel,
// 3: stacked-half tcgen05 kernel
int kernel_choice(int h, int block_size) {
  const int path = g_kernel_path.load();
  if (path == 1 || !sfa::tc_supports(h, block_size)) return 0;
  if (path == 2) return 1;
  if (sfa::narrow_supports(h)) return 2;
  return sfa::stack_supports(h) ? 3 : 1;
}
constexpr long long kDefaultWaitLimit = 1LL << 26;  // iterations of a bounded device wait

// helper streams of sfa_decode_host, created once per device on first use
constexpr int kHostGroups = 4;
constexpr double kHostPipeMinOutBytes = 4.0 * (1 << 20);   // smaller results: one group
struct HostPipe {
  std::mutex mu;   // one enqueue sequence at a time uses the shared events
  cudaStream_t s[kHostGroups] = {};
  cudaEvent_t start = nullptr, done[kHostGroups] = {};
};
std::mutex g_pipe_mu;
HostPipe* g_pipe[kMaxDevices] = {};
bool g_pipe_failed[kMaxDevices] = {};

HostPipe* host_pipe(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  if (g_pipe[dev] || g_pipe_failed[dev]) return g_pipe[dev];
  HostPipe* hp = new HostPipe;
  bool ok = cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) == cudaSuccess;
  for (int g = 0; ok && g < kHostGroups; ++g)
    ok = cudaStreamCreateWithFlags(&hp->s[g], cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp->done[g], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    g_pipe_failed[dev] = true;   // fall back to a single group on the caller's stream
    return nullptr;
  }
  g_pipe[dev] = hp;
  return hp;
}

int* status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sfa_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  return g_status_ptr[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

sfa_status check_decode_args(const void* q, const void* kv, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* topk_idx, int B, int Q, int h,
                             int top_k, int num_blocks, int block_size, int max_blocks_per_seq,
                             float scale, int n_splits) {
  if (B < 0 || Q < 1 || top_k < 0 || num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1 ||
      n_splits < 1 || h < 1 || !isfinite(scale))
    return SFA_ERR_INVALID_ARG;
  if (h > SFA_MAX_HEADS || n_splits > SFA_MAX_SPLITS) return SFA_ERR_UNSUPPORTED;
  if ((long long)B * Q > 0x7fffffffLL) return SFA_ERR_UNSUPPORTED;
  if ((long long)B * Q == 0) return SFA_OK;
  if (!q || !kv || !block_table || !seq_lens || (!topk_idx && top_k > 0)) return SFA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(topk_idx, 4))
    return SFA_ERR_INVALID_ARG;
  return SFA_OK;
}

}  // namespace

// A captured sfa_decode_host step (see include/sfa.h).
struct sfa_host_plan_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

extern "C" {

const char* sfa_status_string(sfa_status s) {
  switch (s) {
    case SFA_OK: return "SFA_OK";
    case SFA_ERR_INVALID_ARG: return "SFA_ERR_INVALID_ARG";
    case SFA_ERR_UNSUPPORTED: return "SFA_ERR_UNSUPPORTED";
    case SFA_ERR_WORKSPACE: return "SFA_ERR_WORKSPACE";
    case SFA_ERR_CUDA: return "SFA_ERR_CUDA";
    case SFA_ERR_DEVICE_TIMEOUT: return "SFA_ERR_DEVICE_TIMEOUT";
    case SFA_ERR_DEVICE_BAD_BLOCK: return "SFA_ERR_DEVICE_BAD_BLOCK";
  }
  return "SFA_UNKNOWN_STATUS";
}

int sfa_set_kernel_path(int path) {
  if (path < 0 || path > 2) return -1;
  return g_kernel_path.exchange(path);
}

long long sfa_set_wait_limit(long long iterations) {
  return g_wait_limit.exchange(iterations < 0 ? 0 : iterations);
}

int sfa_set_stall_injection(int on) { return g_stall.exchange(on ? 1 : 0); }

size_t sfa_decode_workspace_bytes(int B, int Q, int h, int top_k, int n_splits) {
  if (B <= 0 || Q <= 0 || h <= 0 || top_k < 0 || n_splits < 1) return 0;
  if (g_kernel_path.load() != 0) return 0;
  return sfa::tc_workspace_bytes(B * Q, h, top_k, n_splits);
}

int sfa_decode_launches(int B, int Q, int h, int top_k, int block_size, int n_splits, int merge,
                        int* tensor_core_path) {
  if (B < 0 || Q < 1 || h < 1 || h > SFA_MAX_HEADS || top_k < 0 || block_size < 1 ||
      n_splits < 1 || n_splits > SFA_MAX_SPLITS)
    return -1;
  const int choice = kernel_choice(h, block_size);
  const bool tc = choice != 0;
  if (tensor_core_path) *tensor_core_path = choice;
  if ((long long)B * Q == 0) return 0;
  int n = tc ? sfa::tc_launches(B * Q, h, top_k, n_splits) : 1;
  if (n_splits > 1 && merge) n += 1;
  return n;
}

sfa_status sfa_lse_merge(const float* out_part, const float* lse_part, int n_splits, int rows,
                         int dv, float* out, float* lse, sfa_stream stream) {
  if (n_splits < 1 || rows < 0 || dv < 1) return SFA_ERR_INVALID_ARG;
  if (n_splits > SFA_MAX_SPLITS) return SFA_ERR_UNSUPPORTED;
  if (rows == 0) return SFA_OK;
  if (!out_part || !lse_part || !out || !lse) return SFA_ERR_INVALID_ARG;
  if (!aligned(out_part, 16) || !aligned(out, 16) || !aligned(lse_part, 4) || !aligned(lse, 4))
    return SFA_ERR_INVALID_ARG;
  cudaError_t e = sfa::launch_lse_merge(out_part, lse_part, n_splits, rows, dv, out, lse,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

sfa_status sfa_decode(const void* q, const void* kv, const int32_t* block_table,
                      const int32_t* seq_lens, const int32_t* topk_idx, int B, int Q, int h,
                      int top_k, int num_blocks, int block_size, int max_blocks_per_seq,
                      float scale, int n_splits, float* out, float* lse, float* out_part,
                      float* lse_part, void* workspace, size_t workspace_bytes,
                      sfa_stream stream) {
  return sfa_decode_ex(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks, block_size,
                       max_blocks_per_seq, scale, n_splits, 0, 0, out, lse, out_part, lse_part, workspace,
                       workspace_bytes, stream);
}

sfa_status sfa_decode_ex(const void* q, const void* kv, const int32_t* block_table, const int32_t* seq_lens,
                         const int32_t* topk_idx, int B, int Q, int h, int top_k, int num_blocks, int block_size,
                         int max_blocks_per_seq, float scale, int n_splits, int interleave_size, int flags,
                         float* out, float* lse, float* out_part, float* lse_part, void* workspace,
                         size_t workspace_bytes, sfa_stream stream) {
  sfa_status st = check_decode_args(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k,
                                    num_blocks, block_size, max_blocks_per_seq, scale, n_splits);
  if (st != SFA_OK) return st;
  if (interleave_size < 0 || (flags & ~SFA_BLOCK_TABLE_PER_TOKEN) != 0) return SFA_ERR_INVALID_ARG;
  const int T = B * Q;
  if (T == 0) return SFA_OK;
  const bool merge_after = n_splits > 1 && out && lse;
  if (n_splits == 1) {
    if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) return SFA_ERR_INVALID_ARG;
  } else {
    if (!out_part || !lse_part || !aligned(out_part, 16) || !aligned(lse_part, 4))
      return SFA_ERR_INVALID_ARG;
    if ((out && !lse) || (!out && lse)) return SFA_ERR_INVALID_ARG;
    if (merge_after && (!aligned(out, 16) || !aligned(lse, 4))) return SFA_ERR_INVALID_ARG;
  }
  // the workspace is optional: without enough of it the kernels use a schedule that needs none
  const size_t need = sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits);
  if (need == 0 || !workspace || workspace_bytes < need || !aligned(workspace, 256)) {
    workspace = nullptr;
    workspace_bytes = 0;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
  int* status = status_word(dev);
  if (!status) return SFA_ERR_CUDA;

  sfa::DecodeParams p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.topk_idx = topk_idx;
  p.B = B;
  p.Q = Q;
  p.h = h;
  p.top_k = top_k;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.scale = scale;
  p.n_splits = n_splits;
  p.out = n_splits == 1 ? out : out_part;
  p.lse = n_splits == 1 ? lse : lse_part;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  p.status = status;
  const long long wl = g_wait_limit.load();
  p.wait_limit = wl > 0 ? wl : kDefaultWaitLimit;
  p.interleave = interleave_size;
  p.bt_per_token = (flags & SFA_BLOCK_TABLE_PER_TOKEN) ? 1 : 0;
  p.stall = g_stall.load();

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int choice = kernel_choice(h, block_size);
  const bool tc = choice != 0 && sfa::tc_supports_ptrs(q, kv, p.out);
  cudaError_t e = tc ? sfa::launch_decode_tc(p, choice, s) : sfa::launch_decode_simt(p, s);
  if (e != cudaSuccess) return SFA_ERR_CUDA;
  if (merge_after) {
    e = sfa::launch_lse_merge(out_part, lse_part, n_splits, T * h, SFA_D_V, out, lse, s);
    if (e != cudaSuccess) return SFA_ERR_CUDA;
  }
  return SFA_OK;
}

size_t sfa_decode_host_staging_bytes(int B, int Q, int h, int top_k, int max_blocks_per_seq,
                                     int n_splits) {
  if (B < 0 || Q < 1 || h < 1 || top_k < 0 || max_blocks_per_seq < 1 || n_splits < 1) return 0;
  const size_t T = (size_t)B * Q, a = 256;
  size_t n = 0;
  n += round_up(T * h * SFA_D_QK * 2, a);                 // q
  n += round_up((size_t)B * max_blocks_per_seq * 4, a);   // block_table
  n += round_up((size_t)B * 4, a);                        // seq_lens
  n += round_up(T * top_k * 4, a);                        // topk_idx
  n += round_up(T * h * SFA_D_V * 4, a);                  // out
  n += round_up(T * h * 4, a);                            // lse
  if (n_splits > 1) {
    n += round_up((size_t)n_splits * T * h * SFA_D_V * 4, a);  // out_part
    n += round_up((size_t)n_splits * T * h * 4, a);            // lse_part
  }
  n += round_up(sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits), a);
  return n;
}

// The argument checks of sfa_decode_host (SFA_OK also for an empty batch).
static sfa_status check_host_args(const void* q_host, const void* kv, const int32_t* block_table_host,
                                  const int32_t* seq_lens_host, const int32_t* topk_idx_host, int B, int Q, int h,
                                  int top_k, int num_blocks, int block_size, int max_blocks_per_seq, float scale,
                                  int n_splits, const float* out_host, const float* lse_host, const void* staging,
                                  size_t staging_bytes) {
  const sfa_status st = check_decode_args(q_host, kv, block_table_host, seq_lens_host, topk_idx_host, B, Q, h,
                                          top_k, num_blocks, block_size, max_blocks_per_seq, scale, n_splits);
  if (st != SFA_OK || (long long)B * Q == 0) return st;
  if (!out_host || !lse_host) return SFA_ERR_INVALID_ARG;
  const size_t need = sfa_decode_host_staging_bytes(B, Q, h, top_k, max_blocks_per_seq, n_splits);
  if (!staging || staging_bytes < need || !aligned(staging, 256)) return SFA_ERR_WORKSPACE;
  return SFA_OK;
}

sfa_status sfa_decode_host(const void* q_host, const void* kv, const int32_t* block_table_host,
                           const int32_t* seq_lens_host, const int32_t* topk_idx_host, int B,
                           int Q, int h, int top_k, int num_blocks, int block_size,
                           int max_blocks_per_seq, float scale, int n_splits, float* out_host,
                           float* lse_host, void* staging, size_t staging_bytes,
                           sfa_stream stream) {
  sfa_status st = check_host_args(q_host, kv, block_table_host, seq_lens_host, topk_idx_host, B, Q, h, top_k,
                                  num_blocks, block_size, max_blocks_per_seq, scale, n_splits, out_host, lse_host,
                                  staging, staging_bytes);
  if (st != SFA_OK) return st;
  const size_t T = (size_t)B * Q;
  if (T == 0) return SFA_OK;

  char* base = static_cast<char*>(staging);
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    char* p = base + off;
    off += round_up(bytes, 256);
    return p;
  };
  const size_t q_bytes = T * h * SFA_D_QK * 2, bt_bytes = (size_t)B * max_blocks_per_seq * 4,
               sl_bytes = (size_t)B * 4, idx_bytes = T * top_k * 4,
               out_bytes = T * h * SFA_D_V * 4, lse_bytes = T * h * 4;
  void* q_d = carve(q_bytes);
  int32_t* bt_d = reinterpret_cast<int32_t*>(carve(bt_bytes));
  int32_t* sl_d = reinterpret_cast<int32_t*>(carve(sl_bytes));
  int32_t* idx_d = reinterpret_cast<int32_t*>(carve(idx_bytes));
  float* out_d = reinterpret_cast<float*>(carve(out_bytes));
  float* lse_d = reinterpret_cast<float*>(carve(lse_bytes));
  float* op_d = nullptr;
  float* lp_d = nullptr;
  if (n_splits > 1) {
    op_d = reinterpret_cast<float*>(carve((size_t)n_splits * out_bytes));
    lp_d = reinterpret_cast<float*>(carve((size_t)n_splits * lse_bytes));
  }
  const size_t ws_bytes = sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits);
  void* ws_d = ws_bytes ? carve(ws_bytes) : nullptr;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // A batch large enough to be copy-bound is split into groups of whole sequences, each
  // on its own helper stream forked from `s`: group g's results travel back while later
  // groups are still being copied in or computed, and copies in both directions use
  // separate copy engines.  Each group uses its own slices of the staging buffers.
  int groups = 1;
  HostPipe* hp = nullptr;
  if ((double)out_bytes >= kHostPipeMinOutBytes && B >= 2) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) hp = host_pipe(dev);
    if (hp) groups = B < kHostGroups ? B : kHostGroups;
  }
  // the block table, sequence lengths and index lists go first, whole, on `s`; each
  // group then copies only its q in and its out back, and lse returns in one copy at the end
  if (cudaMemcpyAsync(bt_d, block_table_host, bt_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(sl_d, seq_lens_host, sl_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      (idx_bytes && cudaMemcpyAsync(idx_d, topk_idx_host, idx_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess))
    return SFA_ERR_CUDA;
  std::unique_lock<std::mutex> lk;
  if (groups > 1) {
    lk = std::unique_lock<std::mutex>(hp->mu);
    if (cudaEventRecord(hp->start, s) != cudaSuccess) return SFA_ERR_CUDA;
  }
  for (int g = 0; g < groups; ++g) {
    const int b0 = (int)((long long)B * g / groups), b1 = (int)((long long)B * (g + 1) / groups);
    const int Bg = b1 - b0;
    if (Bg == 0) continue;
    cudaStream_t gs = groups > 1 ? hp->s[g] : s;
    if (groups > 1 && cudaStreamWaitEvent(gs, hp->start, 0) != cudaSuccess) return SFA_ERR_CUDA;
    const size_t t0 = (size_t)b0 * Q, Tg = (size_t)Bg * Q;
    const size_t qo = t0 * h * SFA_D_QK * 2, io = t0 * top_k, oo = t0 * h * SFA_D_V, lo = t0 * h;
    const size_t bo = (size_t)b0 * max_blocks_per_seq;
    char* qg = static_cast<char*>(q_d) + qo;
    if (cudaMemcpyAsync(qg, static_cast<const char*>(q_host) + qo, Tg * h * SFA_D_QK * 2,
                        cudaMemcpyHostToDevice, gs) != cudaSuccess)
      return SFA_ERR_CUDA;
    // a group's shard partials are its own [n_splits, Tg, h, ...] block
    float* opg = op_d ? op_d + (size_t)n_splits * oo : nullptr;
    float* lpg = lp_d ? lp_d + (size_t)n_splits * lo : nullptr;
    st = sfa_decode(qg, kv, bt_d + bo, sl_d + b0, idx_d + io, Bg, Q, h, top_k, num_blocks, block_size,
                    max_blocks_per_seq, scale, n_splits, out_d + oo, lse_d + lo, opg, lpg, ws_d, ws_bytes, gs);
    if (st != SFA_OK) return st;
    if (cudaMemcpyAsync(out_host + oo, out_d + oo, Tg * h * SFA_D_V * 4, cudaMemcpyDeviceToHost, gs) !=
        cudaSuccess)
      return SFA_ERR_CUDA;
    if (groups > 1 && (cudaEventRecord(hp->done[g], gs) != cudaSuccess ||
                       cudaStreamWaitEvent(s, hp->done[g], 0) != cudaSuccess))
      return SFA_ERR_CUDA;
  }
  if (cudaMemcpyAsync(lse_host, lse_d, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SFA_ERR_CUDA;
  return SFA_OK;
}

sfa_status sfa_host_plan_create(const void* q_host, const void* kv, const int32_t* block_table_host,
                                const int32_t* seq_lens_host, const int32_t* topk_idx_host, int B, int Q, int h,
                                int top_k, int num_blocks, int block_size, int max_blocks_per_seq, float scale,
                                int n_splits, float* out_host, float* lse_host, void* staging,
                                size_t staging_bytes, sfa_host_plan* plan) {
  if (!plan) return SFA_ERR_INVALID_ARG;
  *plan = nullptr;
  const sfa_status chk = check_host_args(q_host, kv, block_table_host, seq_lens_host, topk_idx_host, B, Q, h,
                                         top_k, num_blocks, block_size, max_blocks_per_seq, scale, n_splits,
                                         out_host, lse_host, staging, staging_bytes);
  if (chk != SFA_OK) return chk;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
  // everything that is set up once per device happens here, outside the capture
  if (!status_word(dev)) return SFA_ERR_CUDA;
  host_pipe(dev);
  if (sfa::prepare_decode_tc() != cudaSuccess || sfa::prepare_decode_narrow() != cudaSuccess ||
      sfa::prepare_decode_stack() != cudaSuccess ||
      sfa::prepare_decode_simt() != cudaSuccess)
    return SFA_ERR_CUDA;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return SFA_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return SFA_ERR_CUDA;
  }
  const sfa_status st = sfa_decode_host(q_host, kv, block_table_host, seq_lens_host, topk_idx_host, B, Q, h, top_k,
                                        num_blocks, block_size, max_blocks_per_seq, scale, n_splits, out_host,
                                        lse_host, staging, staging_bytes, cs);
  cudaGraph_t graph = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (st != SFA_OK || ce != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    return st != SFA_OK ? st : SFA_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return SFA_ERR_CUDA;
  }
  *plan = new sfa_host_plan_s{graph, exec};
  return SFA_OK;
}

sfa_status sfa_host_plan_launch(sfa_host_plan plan, sfa_stream stream) {
  if (!plan) return SFA_ERR_INVALID_ARG;
  return cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

void sfa_host_plan_destroy(sfa_host_plan plan) {
  if (!plan) return;
  cudaGraphExecDestroy(plan->exec);
  cudaGraphDestroy(plan->graph);
  delete plan;
}

sfa_status sfa_uv_proj(const float* out, const void* w_uv, void* y, int T, int h, sfa_stream stream) {
  if (T < 0 || h < 1 || h > 65535) return SFA_ERR_INVALID_ARG;
  if (T == 0) return SFA_OK;
  if (!out || !w_uv || !y || !aligned(out, 16) || !aligned(w_uv, 16) || !aligned(y, 2)) return SFA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
  int* status = status_word(dev);
  if (!status) return SFA_ERR_CUDA;
  const long long wl = g_wait_limit.load();
  return sfa::launch_uv_proj(out, w_uv, y, T, h, wl > 0 ? wl : kDefaultWaitLimit, g_stall.load(), status,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

sfa_status sfa_kv_write(void* kv, long long num_slots, const int32_t* slot_mapping, const void* rows, int T,
                        sfa_stream stream) {
  if (T < 0 || num_slots < 0) return SFA_ERR_INVALID_ARG;
  if (T == 0) return SFA_OK;
  if (!kv || !slot_mapping || !rows || !aligned(kv, 16) || !aligned(rows, 16) || !aligned(slot_mapping, 4))
    return SFA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
  int* status = status_word(dev);
  if (!status) return SFA_ERR_CUDA;
  return sfa::launch_kv_write(kv, num_slots, slot_mapping, rows, T, status, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

static_assert(SFA_TOPK_MAX_S == sfa::kTopkMaxS, "top-k limit of the header and the kernel");

sfa_status sfa_topk(const float* scores, long long row_stride, const int32_t* seq_lens, int B, int Q, int S, int k,
                    int32_t* topk_idx, sfa_stream stream) {
  if (B < 0 || Q < 1 || S < 0 || k < 1 || row_stride < S || row_stride % 4 != 0) return SFA_ERR_INVALID_ARG;
  if ((long long)B * Q > INT_MAX / 8) return SFA_ERR_UNSUPPORTED;
  if (S > sfa::kTopkMaxS) return SFA_ERR_UNSUPPORTED;
  if (B == 0) return SFA_OK;
  if (!topk_idx || !aligned(topk_idx, 4) || (S > 0 && (!scores || !aligned(scores, 16))) ||
      (seq_lens && !aligned(seq_lens, 4)))
    return SFA_ERR_INVALID_ARG;
  return sfa::launch_topk(scores, row_stride, seq_lens, B, Q, S, k, topk_idx, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

sfa_status sfa_last_device_status(sfa_stream stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
  int* status = status_word(dev);
  if (!status) return SFA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SFA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SFA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return SFA_ERR_CUDA;
  return static_cast<sfa_status>(v);
}

}  // extern "C"
