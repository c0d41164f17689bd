// Fused sub-block forward that allocates nothing.
//
// Some callers cannot obtain a device workspace at call time: an inference
// engine that plans all device memory before it runs hands its plugins only
// their input and output buffers and does not allow cudaMalloc while it
// executes, and a process whose caching allocator has already reserved the
// GPU's memory may see a fresh cudaMalloc fail.  For them this entry point
// uses a workspace that the library itself holds: a fixed-size array in
// device global memory, reserved when the library's module is loaded on a GPU
// (with CUDA's lazy module loading, at the first lookup below) and kept until
// the process exits.
//
// Host code cannot use the array's name as a device address (in host code the
// symbol is only a host-side stand-in), so the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current, the
// first time this entry point is called on it; make that first call during
// set-up, before the caller's allocator takes the device's memory and before
// any stream capture begins.  The address is kept for the life of the
// process: a cudaDeviceReset() of the device is not supported.  All calls on a device share the one array and
// the last call's contents stay in it; nothing in it needs to start at zero
// (each stage writes its part before any stage reads it).  Calls whose work
// overlaps on the GPU (different streams without ordering between them) race
// on the array: order them.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

#include "../../include/h3attn.h"

namespace {

constexpr size_t kScratchBytes = H3_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_block_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_block_scratch on the current device (looked up once).
h3_status scratch_on_current_device(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return H3_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_block_scratch) != cudaSuccess || p == nullptr)
      return H3_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *addr = p;
  return H3_OK;
}

}  // namespace

extern "C" h3_status h3_attn_block_fwd_noalloc(const h3_block_desc* desc, const uint16_t* x,
                                               const uint8_t* mod, const int32_t* pos,
                                               const float* shift, const float* scale,
                                               const float* gate, const uint16_t* Wqkv,
                                               const uint16_t* Wo, uint16_t* out,
                                               h3_stream_t stream) {
  size_t need = 0;
  if (h3_status s = h3_workspace_size(desc, &need)) return s;
  if (need > kScratchBytes) return H3_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (h3_status s = scratch_on_current_device(&scratch)) return s;
  return h3_attn_block_fwd(desc, x, mod, pos, shift, scale, gate, Wqkv, Wo, scratch,
                           kScratchBytes, out, stream);
}
