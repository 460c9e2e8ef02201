// sfa_noalloc.cu -- sfa_decode_noalloc: the decode + merge step for callers
// that cannot allocate device memory themselves.
//
// Some callers have no allocator to hand: a serving engine that gives all free
// HBM to its KV-cache pool at start-up and refuses later cudaMalloc calls, a
// plugin host that hands a kernel library only its input and output tensors, or
// a decode loop that must not pay cudaMalloc's implicit device-wide
// synchronisation.  For them the shard partials that sfa_decode normally writes
// into caller-provided buffers live in a fixed, file-scope device array instead.
//
// The array is one per device, sized SFA_NOALLOC_SCRATCH_BYTES, and every GPU
// that loads this library keeps it until the process exits.  Host code cannot
// use the array's name as a device address, so its address is looked up once
// per device (on the first call that needs scratch, with that device current) and
// cached for the life of the process: a device reset invalidates it.
// Every call overwrites all of the scratch it uses before reading it, so nothing
// needs clearing between calls; calls that overlap on the GPU (two streams, or
// two threads) share the one array and race.
#include <mutex>

#include "sfa.h"
#include "sfa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SFA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device).
void* scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" sfa_status sfa_decode_noalloc(const void* q, const void* kv, const int32_t* block_table,
                                         const int32_t* seq_lens, const int32_t* topk_idx, int B,
                                         int Q, int h, int top_k, int num_blocks, int block_size,
                                         int max_blocks_per_seq, float scale, int n_splits,
                                         float* out, float* lse, sfa_stream stream) {
  if (!out || !lse) return SFA_ERR_INVALID_ARG;   // no result buffer: nothing a caller could read
  if (B < 0 || Q < 1 || h < 1 || n_splits < 1 || top_k < 0) return SFA_ERR_INVALID_ARG;
  if (h > SFA_MAX_HEADS || n_splits > SFA_MAX_SPLITS) return SFA_ERR_UNSUPPORTED;
  const size_t T = (size_t)B * Q;
  // scratch this call needs: the shard partials (n_splits > 1) and the decode workspace
  const size_t part_out = n_splits > 1 ? align256((size_t)n_splits * T * h * SFA_D_V * 4) : 0;
  const size_t part_lse = n_splits > 1 ? align256((size_t)n_splits * T * h * 4) : 0;
  const size_t ws = align256(sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits));
  const size_t need = part_out + part_lse + ws;
  if (need > (size_t)SFA_NOALLOC_SCRATCH_BYTES) return SFA_ERR_WORKSPACE;
  if (T == 0) return SFA_OK;

  // a call that needs no scratch does not touch the array (nor load or look it up)
  unsigned char* base = nullptr;
  if (need > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SFA_ERR_CUDA;
    base = static_cast<unsigned char*>(scratch_address(dev));
    if (!base) return SFA_ERR_CUDA;
  }
  float* out_part = n_splits > 1 ? reinterpret_cast<float*>(base) : nullptr;
  float* lse_part = n_splits > 1 ? reinterpret_cast<float*>(base + part_out) : nullptr;
  void* workspace = ws ? static_cast<void*>(base + part_out + part_lse) : nullptr;
  return sfa_decode(q, kv, block_table, seq_lens, topk_idx, B, Q, h, top_k, num_blocks,
                    block_size, max_blocks_per_seq, scale, n_splits, out, lse, out_part, lse_part,
                    workspace, ws, stream);
}
