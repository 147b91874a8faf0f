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
// address is looked up once per device and context, on the first call made
// while that device is current, so that first call should come before any
// stream capture.  kda_noalloc_status() reads the status block in it, as
// kda_workspace_status() does for a caller workspace.  All calls on a device share the one buffer and it keeps the last
// call's contents; the status block in it is cleared by every call, as
// kda_chunk_fwd does with a caller workspace.  Calls whose kernels overlap on
// the GPU (different streams, or different host threads) race on the buffer:
// order them on one stream.
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <mutex>

#include "kda.h"

namespace kda {
size_t chunk_fwd_required_workspace(const kda_shape *s);  // kda_abi.cu
}

namespace {

constexpr size_t kScratchBytes = 256 * 1024;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char kda_noalloc_scratch[kScratchBytes];

// The buffer's address per device, with the context it was looked up in: after a
// cudaDeviceReset (or in another context of the device) the address is looked up
// again instead of reusing one that no longer belongs to the current context.
struct Cached {
  CUcontext ctx;
  void *addr;
};
Cached g_cache[kMaxDevices];
std::mutex g_cache_lock;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CUcontext current_context() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

// Device address of the built-in buffer in the current context, or nullptr.
void *scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (cudaSetDevice(dev) != cudaSuccess) return nullptr;  // makes the device's context current
  const CUcontext ctx = current_context();
  if (!ctx) return nullptr;
  std::lock_guard<std::mutex> lock(g_cache_lock);
  if (g_cache[dev].addr && g_cache[dev].ctx == ctx) return g_cache[dev].addr;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, kda_noalloc_scratch) != cudaSuccess || addr == nullptr) {
    cudaGetLastError();  // do not leave the lookup failure as a sticky "last error"
    return nullptr;
  }
  g_cache[dev] = Cached{ctx, addr};
  return addr;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const kda_shape *shape, const void *q, const void *k,
                                     const void *v, const void *g, const void *beta,
                                     const float *init_state, const int32_t *cu_seqlens,
                                     void *out, float *final_state, cudaStream_t stream) {
  if (!shape) return KDA_ERR_NULL;
  const size_t need = kda::chunk_fwd_required_workspace(shape);
  if (need == 0) return KDA_ERR_SHAPE;
  // the status block and one recomputation flag per sequence-head must fit (the
  // schedule that fits the rest runs): beyond about 65,000 sequence-heads they do not
  if (need > kScratchBytes) return KDA_ERR_NOALLOC_LIMIT;
  void *scratch = scratch_on_current_device();
  if (!scratch) return KDA_ERR_DEVICE;
  return kda_chunk_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state, scratch,
                       kScratchBytes, stream);
}

extern "C" int kda_noalloc_status(uint32_t *words, cudaStream_t stream) {
  void *scratch = scratch_on_current_device();
  if (!scratch) return KDA_ERR_DEVICE;
  const int rc = kda_workspace_status(scratch, stream);  // synchronises the stream
  if (words && rc != KDA_ERR_LAUNCH &&
      cudaMemcpy(words, scratch, 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  return rc;
}
