// Library-level entry points: status names and the device error-word check.
#include "common.cuh"
#include "linear_internal.h"

namespace qspec {
unsigned int* verify_error_word(void* ws);
qspec_status read_and_clear_decode_error(cudaStream_t s, unsigned int* bits);
}

extern "C" const char* qspec_status_string(qspec_status status) {
  switch (status) {
    case QSPEC_OK: return "QSPEC_OK";
    case QSPEC_ERR_INVALID_ARG: return "QSPEC_ERR_INVALID_ARG";
    case QSPEC_ERR_UNSUPPORTED_SHAPE: return "QSPEC_ERR_UNSUPPORTED_SHAPE";
    case QSPEC_ERR_MISALIGNED: return "QSPEC_ERR_MISALIGNED";
    case QSPEC_ERR_WORKSPACE: return "QSPEC_ERR_WORKSPACE";
    case QSPEC_ERR_CUDA: return "QSPEC_ERR_CUDA";
    case QSPEC_ERR_TIMEOUT: return "QSPEC_ERR_TIMEOUT";
  }
  return "QSPEC_ERR_UNKNOWN";
}

extern "C" qspec_status qspec_check_status(void* ws, qspec_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return QSPEC_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return QSPEC_ERR_CUDA;
  unsigned int lin = 0, ver = 0;
  unsigned int dec = 0;
  if (qspec::read_and_clear_linear_error(s, &lin) != QSPEC_OK) return QSPEC_ERR_CUDA;
  if (qspec::read_and_clear_decode_error(s, &dec) != QSPEC_OK) return QSPEC_ERR_CUDA;
  if (ws) {
    unsigned int* w = qspec::verify_error_word(ws);
    if (cudaMemcpyAsync(&ver, w, sizeof(ver), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return QSPEC_ERR_CUDA;
    if (ver && (cudaMemsetAsync(w, 0, sizeof(unsigned int), s) != cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess))
      return QSPEC_ERR_CUDA;
  }
  if (lin & qspec::kErrTimeout) return QSPEC_ERR_TIMEOUT;
  if (lin & qspec::kErrWorkspace) return QSPEC_ERR_WORKSPACE;
  if ((ver & 2u) || (dec & 4u)) return QSPEC_ERR_INVALID_ARG;
  return QSPEC_OK;
}
