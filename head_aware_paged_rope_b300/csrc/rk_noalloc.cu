// rk_segpaged_decode_noalloc: the decode entry point for callers that cannot allocate
// device memory.  Its scratch (work list and split-KV partials) lives in a fixed
// file-scope device array instead of a caller workspace; everything else is the regular
// decode path, called unchanged.
#include "rk_internal.cuh"

#include <mutex>

namespace {

// Shared by every call on a device; loaded with the library and held until process exit.
static __device__ __align__(256) uint8_t g_decode_scratch[RK_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" rk_status rk_segpaged_decode_noalloc(const rk_attn_args* args, rk_stream_t stream) {
  const size_t need = rk_segpaged_decode_workspace_size(args);
  if (need == 0)   // invalid arguments or nothing to do: the regular path returns the status
    return rk_segpaged_decode(args, nullptr, 0, stream);
  if (need > RK_DECODE_NOALLOC_SCRATCH_BYTES) return RK_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RK_ERR_CUDA;
  void* scratch = nullptr;
  {
    // one-time set-up per device, with that device current: the device address of the
    // array (its host-side name is only a stand-in for it)
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return RK_ERR_CUDA;
      // the decode workspace's split counters start at zero (each call leaves them so); the
      // zeroing is ordered before this call's decode on the caller's stream
      if (cudaMemsetAsync(p, 0, rk::kDecCounterBytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RK_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return rk_segpaged_decode(args, scratch, RK_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
