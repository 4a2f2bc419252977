// adp_decode_step_noalloc: one decode step whose scratch lives in a static device array of this
// file instead of in buffers that the model allocated, so that the call itself allocates no
// device memory (no cudaMalloc/cudaFree, no allocating library routine).
//
// The array's device address is looked up per device by adp_create_model (with the model's device
// current), because that lookup may load this file's module, and loading the module is what puts
// the array in device memory: creation allocates anyway, the no-alloc call must not.
//
// Every call, from every model, shares the one array.  Its contents must start at zero: they do
// when the module is loaded, every completed step leaves them in a state the next step accepts
// (attention and sampling counters back at zero, the epoch base advanced past every tag written),
// and this file clears the array again whenever a model with a different layout uses it, a step
// ends in a device-side error, or the 32-bit epoch tags would run past 2^32.  Calls that overlap in time (two host threads, or two streams)
// race on the array and give wrong results: serialise them.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/adp.h"
#include "scratch.h"

namespace {
constexpr size_t kStaticScratchBytes = (size_t)8 << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

struct DeviceSlot {
  unsigned char* addr = nullptr;  // device address of g_step_scratch on this device
  bool have_layout = false;
  adp::ScratchLayout layout{};    // layout of the last step taken in the array
  uint64_t epochs_used = 0;       // epochs handed out since the array was last zeroed
};

std::mutex g_mutex;
DeviceSlot g_slots[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

int adp::noalloc_prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) {
    adp::set_last_error("adp_create_model: CUDA device index beyond the no-alloc step's device table");
    return ADP_ERR_UNSUPPORTED_CONFIG;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSlot& s = g_slots[dev];
  if (s.addr) return ADP_OK;
  // set-up, once per device, with that device current (the caller's contract)
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_step_scratch);
  if (e != cudaSuccess || !ptr) {
    char msg[200];
    std::snprintf(msg, sizeof msg, "adp_create_model: cudaGetSymbolAddress of the no-alloc scratch: %s",
                  cudaGetErrorString(e));
    adp::set_last_error(msg);
    return ADP_ERR_CUDA;
  }
  s.addr = static_cast<unsigned char*>(ptr);
  return ADP_OK;
}

extern "C" int adp_decode_step_noalloc(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                                       int32_t* next_token, float* dev_logits) {
  adp::ScratchLayout lay;
  if (adp::scratch_layout(m, &lay) != ADP_OK || !kv || !next_token) return ADP_ERR_INVALID_ARG;
  if (lay.total > kStaticScratchBytes) {
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "adp_decode_step_noalloc: this model's step needs %zu bytes of scratch, more than the %zu bytes "
                  "of the static array",
                  lay.total, kStaticScratchBytes);
    adp::set_last_error(msg);
    return ADP_ERR_UNSUPPORTED_CONFIG;
  }
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    adp::set_last_error("adp_decode_step_noalloc: no usable current CUDA device");
    return ADP_ERR_CUDA;
  }
  if (dev != adp::model_device(m)) {
    // the array of one device and a stream of another would not meet: refuse before any work
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "adp_decode_step_noalloc: the current CUDA device (%d) is not the model's device (%d)", dev,
                  adp::model_device(m));
    adp::set_last_error(msg);
    return ADP_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSlot& s = g_slots[dev];
  if (!s.addr) {  // adp_create_model sets every model's device up; nothing is looked up (or loaded) here
    adp::set_last_error("adp_decode_step_noalloc: the device's static scratch was not set up");
    return ADP_ERR_CUDA;
  }
  // A model with another layout would read words that the last one left at other offsets.
  // ... and 32-bit epoch tags must not run past 2^32: start over before they would.
  const bool same = s.have_layout && std::memcmp(&s.layout, &lay, sizeof lay) == 0 &&
                    s.epochs_used + 2 * lay.n_phases < (1ull << 32);
  const size_t zero = same ? 0 : kStaticScratchBytes;
  if (!same) s.epochs_used = 0;
  s.layout = lay;
  s.have_layout = true;
  const int rc = adp::decode_step_in_scratch(m, kv, token, sampling, next_token, dev_logits, s.addr, lay, zero,
                                             kStaticScratchBytes);
  if (rc != ADP_OK) s.have_layout = false;  // the next call starts the array over from zero
  else s.epochs_used += lay.n_phases;
  return rc;
}
