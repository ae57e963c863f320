// Library-wide entry points: status strings and the device error word.
#include "common.cuh"

extern "C" cudaError_t moe_detail_take_error_quantize(unsigned int* out);
extern "C" cudaError_t moe_detail_take_error_sort(unsigned int* out);
extern "C" cudaError_t moe_detail_take_error_combine(unsigned int* out);
extern "C" cudaError_t moe_detail_take_error_gmm(unsigned int* out);

extern "C" const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or mode)";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape, mode or device (needs sm_103)";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE: return "device error word set (see moe_get_device_error)";
  }
  return "unknown status";
}

extern "C" moe_status moe_get_device_error(moe_stream_t stream, int* code) {
  if (!code) return MOE_ERR_INVALID_ARG;
  *code = 0;
  if (cudaStreamSynchronize(moe::as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned int all = 0, v = 0;
  cudaError_t (*take[])(unsigned int*) = {moe_detail_take_error_quantize, moe_detail_take_error_sort,
                                          moe_detail_take_error_combine, moe_detail_take_error_gmm};
  for (auto fn : take) {
    if (fn(&v) != cudaSuccess) return MOE_ERR_CUDA;
    all |= v;
  }
  *code = static_cast<int>(all);
  return all ? MOE_ERR_DEVICE : MOE_OK;
}
