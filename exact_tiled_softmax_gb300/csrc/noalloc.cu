// attn_bwd_noalloc: the reverse pass for callers that cannot allocate device
// memory.
//
// attn_bwd needs a caller-provided workspace (the status word, delta, L log2 e
// and the fp32 dQ accumulator).  Some callers have no way to provide one: a
// plugin whose host hands it only its input and output buffers, or code that
// must not let a device allocation (which can synchronise the device, or fail
// under a memory cap) happen on its path.  This entry point instead uses a
// scratch array that lives in this library's own device memory: a file-scope
// __device__ array of kScratchBytes (64 MiB), which every GPU that loads this
// part of the library keeps until the process exits.  It allocates nothing.
//
// The array's name in host code is only a host-side stand-in, not a device
// address, so the device address is looked up with cudaGetSymbolAddress once
// per device, with that device current, on the first call made on it; that
// first call should come before any stream capture.  Every call shares the
// array: attn_bwd clears the status word and the dQ accumulator itself on each
// call, and calls whose work overlaps on the GPU (for example on two streams)
// race on the array and must not be issued.  The kernels' status word (an
// empty allowed set, a bounded wait that gave up) is word 0 of the array;
// exattn_noalloc_device_status reads it back.
#include <atomic>

#include "../../include/exattn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of g_bwd_scratch on the current device, or nullptr.
void* scratch_on_current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    exattn::record_error("attn_bwd_noalloc: cudaGetDevice", static_cast<int>(e),
                         cudaGetErrorString(e));
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    exattn::record_error("attn_bwd_noalloc: device ordinal out of range", dev, "");
    return nullptr;
  }
  void* ptr = g_scratch_ptr[dev].load();
  if (ptr) return ptr;
  e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
  if (e != cudaSuccess || ptr == nullptr) {
    exattn::record_error("attn_bwd_noalloc: cudaGetSymbolAddress", static_cast<int>(e),
                         cudaGetErrorString(e));
    return nullptr;
  }
  g_scratch_ptr[dev].store(ptr);
  return ptr;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const exattn_shape* shape, const void* Q, const void* K,
                                const void* V, const void* Y, const void* dY, const float* L,
                                float scale, int mask_kind, int window,
                                const uint32_t* bitmask, void* dQ, void* dK, void* dV,
                                void* cuda_stream) {
  const size_t need = exattn_bwd_workspace_size(shape, mask_kind);
  if (need == 0) return EXATTN_INVALID_ARG;
  if (need > kScratchBytes) {
    exattn::record_error("attn_bwd_noalloc: scratch needed exceeds the 64 MiB static array",
                         EXATTN_WORKSPACE_TOO_SMALL, "");
    return EXATTN_WORKSPACE_TOO_SMALL;
  }
  void* scratch = scratch_on_current_device();
  if (!scratch) return EXATTN_CUDA_ERROR;
  return attn_bwd(shape, Q, K, V, Y, dY, L, scale, mask_kind, window, bitmask, dQ, dK, dV,
                  scratch, kScratchBytes, cuda_stream);
}

extern "C" int exattn_noalloc_device_status(void* cuda_stream) {
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    exattn::record_error("exattn_noalloc_device_status: cudaStreamSynchronize",
                         static_cast<int>(e), cudaGetErrorString(e));
    return EXATTN_CUDA_ERROR;
  }
  void* scratch = scratch_on_current_device();
  if (!scratch) return EXATTN_CUDA_ERROR;
  unsigned word = 0;
  e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    exattn::record_error("exattn_noalloc_device_status: cudaMemcpy", static_cast<int>(e),
                         cudaGetErrorString(e));
    return EXATTN_CUDA_ERROR;
  }
  if (word & 2u) return EXATTN_TIMEOUT;
  if (word & 1u) return EXATTN_EMPTY_ROW;
  return EXATTN_OK;
}
