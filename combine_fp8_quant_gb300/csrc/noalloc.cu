// noalloc.cu -- moe_dispatch_compact_noalloc: the compact dispatch for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any other allocating routine: a
// plugin inside a host engine that owns every device allocation and hands the
// plugin only its inputs and outputs, a serving loop that forbids allocation
// after start-up so that its memory footprint stays fixed, or a runtime with
// a fixed device-memory budget. moe_dispatch_compact needs a small scratch
// workspace (a token counter, and the per-chunk expert table on the
// two-launch path), which such a caller would otherwise have to allocate.
// This variant keeps that scratch in one file-scope device array of fixed
// size instead. Every GPU that loads the library holds the array until the
// process exits.
//
// In host code the array's name is only a host-side stand-in, not a device
// address: handing it to a kernel would fault or silently use the wrong
// memory. The device address is therefore looked up with
// cudaGetSymbolAddress, with the device current, on the first call in each
// CUDA context (normally once per device: the primary context), and cached
// under the context's unique id. A context created again after
// cudaDeviceReset has a new id, so the address is looked up again there
// rather than reused.
//
// Nothing in the array has to start at zero: the route plan writes every
// chunk-table word before the scatter reads it and resets the token counter
// itself, so a call neither clears the array nor depends on what the previous
// call left in it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moeperm.h"
#include "common.cuh"

namespace {

// The largest workspace moe_workspace_bytes reports: a 64 KiB chunk table
// plus the 256-byte reserved header.
constexpr size_t kNoAllocScratchBytes = 64 * 1024 + 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxEntries = 64;
std::mutex g_setup_mutex;
ScratchEntry g_entries[kMaxEntries];
int g_nentries = 0;
int g_next = 0;  // entry replaced when the table is full

// Device address of the scratch array in the current context; the first call
// in a context looks it up (which also initialises the device's primary
// context if no context is current yet).
cudaError_t scratch_address(void** out) {
  using moeperm::current_context_id;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  unsigned long long id = 0;
  cudaError_t err = current_context_id(&id);
  if (err != cudaSuccess) return err;
  if (id != 0)
    for (int i = 0; i < g_nentries; ++i)
      if (g_entries[i].ctx_id == id) {
        *out = g_entries[i].addr;
        return cudaSuccess;
      }
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (err != cudaSuccess) return err;
  err = current_context_id(&id);
  if (err != cudaSuccess) return err;
  if (id != 0) {
    int slot = g_nentries < kMaxEntries ? g_nentries++ : (g_next++ % kMaxEntries);
    g_entries[slot] = ScratchEntry{id, p};
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_dispatch_compact_noalloc(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t block_e, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* m_indices, int64_t bound,
    int32_t* src2dst, int32_t* counts, int32_t* starts, int32_t* psum, int32_t* total,
    float* row_weights, int32_t* d_status, moe_stream_t stream) {
  const size_t need = moe_workspace_bytes(T, K, L);
  if (need == 0 || need > kNoAllocScratchBytes) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // moe_dispatch_compact validates every argument before it enqueues anything.
  return moe_dispatch_compact(x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L,
                              block_e, g, fmt, xq, scales, ld_s, m_indices, bound, src2dst,
                              counts, starts, psum, total, row_weights, scratch,
                              kNoAllocScratchBytes, d_status, stream);
}
