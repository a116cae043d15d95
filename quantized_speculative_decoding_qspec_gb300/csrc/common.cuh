// Shared helpers of the qspec CUDA library (sm_103a).  Nothing here is method arithmetic beyond
// bit-level bf16 handling.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "qspec.h"

namespace qspec {

constexpr int kGroup = QSPEC_GROUP;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Status of the launches just enqueued on this thread.
inline qspec_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// bf16 bit pattern (low 16 bits of b) -> fp32, exact.
__device__ __forceinline__ float bf16_lo(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t b) { return __uint_as_float(b & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (the hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// a / b rounded to nearest (IEEE), given rb = 1 / b rounded to nearest: Markstein's division
// refinement -- q0 = a * rb is within one ulp of a / b, the FMA gives the remainder a - b q0
// exactly, and one more FMA rounds q0 + remainder * rb correctly.  That needs the remainder to be
// representable: with b >= 2^-100 it is whenever |a / b| >= 1/4, the only quotients whose rounding
// can change a code (smaller ones give code 0 either way).  The quantisers keep the IEEE division
// for smaller b (and for the 8-bit divisor 127, which the check below does not cover).  Checked exhaustively against the IEEE division for every bf16 amax (b = amax / 7)
// and every bf16 |a| <= amax: identical codes, identical quotients wherever |a / b| >= 1/4.
__device__ __forceinline__ float div_rn_markstein(float a, float b, float rb) {
  const float q0 = a * rb;
  const float r = fmaf(-b, q0, a);
  return fmaf(r, rb, q0);
}

// 16-byte streaming load that does not allocate in L1 (data read exactly once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Launch with programmatic dependent launch allowed: the kernel may start while the previous
// kernel in the stream drains; it must execute griddepcontrol.wait before touching global memory
// that the previous kernel writes or reads.
template <typename... KArgs, typename... Args>
inline qspec_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

}  // namespace qspec
