// Decode step with its scratch in caller-given device memory (engine.cu <-> noalloc.cu).
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "../../include/adp.h"

namespace adp {

// Byte offsets, in one scratch area, of everything a decode step writes besides the KV cache:
// the epoch-tagged exchange vectors and attention partials, the epoch base, the
// sampling and argmax words, the grid-barrier counter, the error word, the router choices, the
// step state and the logits.  Each region starts at a multiple of 256 bytes.
struct ScratchLayout {
  size_t x, q, attn, h, rlog, knew, vnew, epoch, tok_word, part_m, part_l, part_o, sblock, sample_ctr, argkey,
      lm_ctr, bar_ctr, err, sel_out, state, logits;
  size_t total;
  size_t n_phases;  // epochs one step takes
};

// Layout for model m (host only, no CUDA call).  Returns ADP_ERR_INVALID_ARG for a null model.
int scratch_layout(const adp_model* m, ScratchLayout* out);

// adp_decode_step's work with the step's scratch at `base` (laid out as `lay`, all of it zero
// before the model's first step there): one persistent launch on the model's stream, then a wait
// for the result.  If zero_bytes > 0 the first `zero_bytes` bytes at base are cleared first.  On
// a device-side error the first `clear_bytes` bytes are cleared before the error is returned.
int decode_step_in_scratch(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                           int32_t* next_token, float* dev_logits, uint8_t* base, const ScratchLayout& lay,
                           size_t zero_bytes, size_t clear_bytes);

// Record a message for adp_last_error().
void set_last_error(const char* msg);

// The CUDA device a model was created on (-1 for a null model).
int model_device(const adp_model* m);

// Set-up of adp_decode_step_noalloc for the current device (noalloc.cu): looks up the device
// address of the static scratch array once per device.  Called by adp_create_model with the
// model's device current, where allocation is expected: loading the array's module is what places
// the array in device memory, so no later no-alloc call on that device can be the one that does.
int noalloc_prepare_device(int device);

}  // namespace adp
