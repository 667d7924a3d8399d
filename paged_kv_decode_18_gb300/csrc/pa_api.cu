// pa_api.cu -- the library-wide entry points of the C ABI that own no kernel:
// status strings, the device error word, the version.
#include "pa_host.h"

extern "C" const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_ARG: return "PA_ERR_ARG: invalid argument (null pointer, size or shape)";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: shape not built (head_dim, block_size, group)";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA runtime call failed";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE: a device-side check failed";
    default: return "unknown pa_status";
  }
}

extern "C" int pa_debug_read_error(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PA_OK;
  unsigned word = pa::take_error_word_cache(st, &rc);
  word |= pa::take_error_word_decode(st, &rc);
  word |= pa::take_error_word_varlen(st, &rc);
  word |= pa::take_error_word_prefill(st, &rc);
  word |= pa::take_error_word_cascade(st, &rc);
  if (rc != PA_OK) return rc;
  return static_cast<int>(word);
}

extern "C" const char* pa_version(void) { return "pagedattn 0.1 sm_103a"; }
