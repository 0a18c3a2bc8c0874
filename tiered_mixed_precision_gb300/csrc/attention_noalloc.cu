// fade_decode_attention_noalloc: decode attention whose split-KV scratch lives in a fixed
// array inside the library, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run attention:
// code that runs inside an allocator-free region of a serving engine, a plugin that receives
// only its inputs and outputs from a host framework, or code that must not perturb a memory
// pool it does not own. They still pass q, the cache and the outputs; the split partials that
// fade_decode_attention normally keeps in a caller-provided workspace go to the array below.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds it
// (kNoAllocScratchBytes) until the process exits. In host code its name is only a host-side
// stand-in, not a device address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)FADE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attention_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
fade_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_decode_attention_noalloc: cudaGetDevice: %s",
                     cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(FADE_ERR_UNSUPPORTED, "fade_decode_attention_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attention_scratch);
    if (e != cudaSuccess || !p)
      return set_error(FADE_ERR_CUDA,
                       "fade_decode_attention_noalloc: cudaGetSymbolAddress failed: %s",
                       cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FADE_OK;
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_decode_attention_noalloc(const fade_config_t* cfg,
                                                       const fade_layer_t* layer,
                                                       const uint16_t* q_rot, uint16_t* out,
                                                       float* logits_ws, float* ml_ws,
                                                       void* stream) {
  clear_error();
  FADE_RANGE("fade_decode_attention_noalloc");
  void* scratch = nullptr;
  fade_status_t st = scratch_on_current_device(&scratch);
  if (st) return st;
  // The split partials are written in full by every call before they are read, so nothing in
  // the array has to start at zero.
  st = fade_decode_attention(cfg, layer, q_rot, out, logits_ws, ml_ws, scratch,
                             kNoAllocScratchBytes, stream);
  if (st == FADE_ERR_CAPACITY && strstr(fade_last_error(), "attention workspace")) {
    char why[400];
    snprintf(why, sizeof(why), "%s", fade_last_error());
    return set_error(FADE_ERR_CAPACITY,
                     "fade_decode_attention_noalloc: this shape needs more split scratch than "
                     "the library's fixed %zu bytes (%s); use fade_decode_attention with a "
                     "caller-allocated workspace",
                     kNoAllocScratchBytes, why);
  }
  return st;
}
