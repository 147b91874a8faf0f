// kda_chunk_fwd_noalloc: the chunk prefill for callers that cannot allocate
// device memory.
//
// kda_chunk_fwd needs a caller-provided workspace (the device status block and
// any kernel scratch).  Some callers own nothing but their input and output
// buffers and cannot obtain more device memory: a host framework whose device
// memory is entirely reserved by its own allocator, a plug-in that is handed
// tensors but no allocator, or a latency-critical path where cudaMalloc (which
// can synchronise the whole device) is not acceptable.  This entry point gives
// them the same computation with the workspace taken from a buffer compiled
// into the library instead.
//
// The buffer is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads this library holds it until the process exits.  Its device
// address is looked up once per device, on the first call made while that
// device is current, so that first call should come before any stream
// capture.  All calls on a device share the one buffer and it keeps the last
// call's contents; the status block in it is cleared by every call, as
// kda_chunk_fwd does with a caller workspace.  Calls whose kernels overlap on
// the GPU (different streams, or different host threads) race on the buffer:
// order them on one stream.
#include <cuda_runtime_api.h>

#include <atomic>

#include "kda.h"

namespace {

constexpr size_t kScratchBytes = 256 * 1024;
constexpr size_t kMinWorkspaceBytes = 256;  // the device status block
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char kda_noalloc_scratch[kScratchBytes];

std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of the built-in buffer on the current device, or nullptr.
void *scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, kda_noalloc_scratch) != cudaSuccess || addr == nullptr) {
    cudaGetLastError();  // do not leave the lookup failure as a sticky "last error"
    return nullptr;
  }
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const kda_shape *shape, const void *q, const void *k,
                                     const void *v, const void *g, const void *beta,
                                     const float *init_state, const int32_t *cu_seqlens,
                                     void *out, float *final_state, cudaStream_t stream) {
  if (kda_chunk_fwd_workspace_bytes(shape) == 0) return shape ? KDA_ERR_SHAPE : KDA_ERR_NULL;
  // every schedule needs the status block; kda_chunk_fwd runs the one that fits the rest
  if (kMinWorkspaceBytes > kScratchBytes) return KDA_ERR_NOALLOC_LIMIT;
  void *scratch = scratch_on_current_device();
  if (!scratch) return KDA_ERR_DEVICE;
  return kda_chunk_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state, scratch,
                       kScratchBytes, stream);
}
