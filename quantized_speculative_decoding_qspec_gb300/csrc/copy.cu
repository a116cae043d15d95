// qspec_copy: a step's small inputs and results moved by the SMs instead of a copy engine.
//
// A decode step's per-step host traffic is tiny (a few tokens' activations in, a few verify results
// out), so a copy-engine transfer is all fixed latency, and the kernel after it cannot start its
// prologue until the transfer has finished.  Here one kernel reads the source with 16-byte loads
// (pinned host memory through its device mapping, over the host link) and writes the destination;
// it launches with programmatic dependent launch, so the next kernel's first weight fetches overlap
// it.  It writes only after waiting for the previous kernel; a source in host memory (which no
// kernel writes) is read before that wait, a source in device memory after it.
#include "common.cuh"

namespace qspec {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                              size_t n16, int src_on_host) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads * kCopyUnroll;
  const size_t first = static_cast<size_t>(blockIdx.x) * kCopyThreads * kCopyUnroll + threadIdx.x;
  bool waited = false;
  if (!src_on_host) {  // the previous kernel may write src
    asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
  }
  for (size_t i0 = first; i0 < n16; i0 += stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const size_t i = i0 + static_cast<size_t>(u) * kCopyThreads;
      v[u] = i < n16 ? src[i] : make_uint4(0, 0, 0, 0);
    }
    if (!waited) {  // the previous kernel may still read dst
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const size_t i = i0 + static_cast<size_t>(u) * kCopyThreads;
      if (i < n16) dst[i] = v[u];
    }
  }
  if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The device address of p: itself for device or managed memory, the device mapping of pinned or
// registered host memory; null for memory the GPU cannot address (pageable host memory).
const void* device_view(const void* p, bool* on_host) {
  *on_host = false;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // (clear the error it recorded, so that later checks do not report it)
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      if (!a.devicePointer || !a.hostPointer) return nullptr;
      *on_host = true;
      // the device view of p: the same offset from the device pointer as p from the host pointer
      // (the two are equal under unified addressing)
      return static_cast<const char*>(a.devicePointer) +
             (static_cast<const char*>(p) - static_cast<const char*>(a.hostPointer));
    default:
      return nullptr;
  }
}

}  // namespace
}  // namespace qspec

extern "C" qspec_status qspec_copy(void* dst, const void* src, size_t bytes, qspec_stream_t stream) {
  using namespace qspec;
  if (!dst || !src || bytes == 0) return QSPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) & 15u) return QSPEC_ERR_MISALIGNED;
  bool dst_host = false, src_host = false;
  void* d = const_cast<void*>(device_view(dst, &dst_host));
  const void* s = device_view(src, &src_host);
  if (!d || !s) return QSPEC_ERR_INVALID_ARG;
  const size_t n16 = bytes / 16;
  const size_t per_cta = static_cast<size_t>(kCopyThreads) * kCopyUnroll;
  const size_t want = (n16 + per_cta - 1) / per_cta;
  const int grid = static_cast<int>(want < static_cast<size_t>(4 * num_sms()) ? want : static_cast<size_t>(4 * num_sms()));
  return launch_pdl(copy16_kernel, dim3(grid), dim3(kCopyThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                    static_cast<uint4*>(d), static_cast<const uint4*>(s), n16, src_host ? 1 : 0);
}
