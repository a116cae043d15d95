// Internal interface between the linear entry points and their kernel families.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qspec.h"

namespace qspec {

// abits: activation width of the mode -- 16 (W4A16), 4 (W4A4) or 8 (W4A8).

// CUDA-core kernels: every shape the entry points accept.
qspec_status linear_simt(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M,
                         int N, int K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                         cudaStream_t stream);

// Tensor-core (tcgen05) kernels: the shapes for which linear_tc_supported() is true.
bool linear_tc_supported(int abits, int M, int N, int K);
size_t linear_tc_workspace_size(int abits, int M, int N, int K);
qspec_status linear_tc(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M,
                       int N, int K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

// The per-token quantiser as its own kernel (one CTA per token): codes [M, K] and fp32 scales [M],
// plus the optional int8 codes and scales out.  The codes are bf16 for the tensor-core path; with
// gemv_layout they are the GEMV's staged fp16 chunks (elements 2, 3, 6, 7 of each 8 divided by 16).  ws_codes gives the workspace's code and scale
// buffers for a quantised mode (false for W4A16).
qspec_status quantise_tokens(int abits, const uint16_t* x, int M, int K, bool gemv_layout, uint16_t* codes,
                             float* s_a, int8_t* xq_out, float* xs_out, cudaStream_t stream);
bool ws_codes(int abits, int M, int N, int K, void* ws, uint16_t** codes, float** s_a);

// The largest tensor-core workspace over the three modes for one shape (the GEMV's own regions
// follow it).
size_t linear_tc_workspace_size_all(int M, int N, int K);

// Register-fragment MMA GEMV for every mode at decode sizes (M <= 16; K is split into chunks
// across CTAs when the staged activations of all K do not fit shared memory).
bool gemv_supported(int M, int N, int K);
size_t gemv_workspace_bytes(int M, int N, int K);  // beyond linear_tc_workspace_size_all
qspec_status gemv(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K,
                  uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws, cudaStream_t stream);

// Reads (synchronously) and clears the error bits the linear kernels set on the current device.
qspec_status read_and_clear_linear_error(cudaStream_t stream, unsigned int* bits);

}  // namespace qspec
