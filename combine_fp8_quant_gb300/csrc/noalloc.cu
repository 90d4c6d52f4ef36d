// noalloc.cu -- moe_dispatch_compact_noalloc: the compact dispatch for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine. Examples:
//   - code that runs while a CUDA graph is being captured, where allocation is
//     not allowed;
//   - plugins hosted by an engine that owns every device allocation and hands
//     out only inputs and outputs;
//   - latency-critical serving loops that forbid allocation after start-up.
// moe_dispatch_compact needs a small scratch workspace (the per-chunk expert
// table), which such a caller would otherwise have to allocate. This variant keeps that scratch in one file-scope device array of
// fixed size instead. Every GPU that loads the library holds the array until
// the process exits.
//
// The host cannot use the array's name as a device address: in host code the
// name is only a host-side stand-in. The address is therefore looked up once
// per device with cudaGetSymbolAddress, on the first call made with that
// device current, and cached. Calls after that only enqueue a memset of the
// used part of the array (so no call can see a previous call's table) and the
// two dispatch kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moeperm.h"

namespace {

// 64 KiB chunk table plus the 256-byte reserved header of the workspace layout.
constexpr size_t kNoAllocScratchBytes = 64 * 1024 + 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: clear the part this call uses.
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_dispatch_compact(x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L,
                              block_e, g, fmt, xq, scales, ld_s, m_indices, bound, src2dst,
                              counts, starts, psum, total, row_weights, scratch,
                              kNoAllocScratchBytes, d_status, stream);
}
