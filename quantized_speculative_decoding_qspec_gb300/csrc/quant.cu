// Step a3 as its own kernel: the per-token activation quantiser (and its 8-bit variant for W4A8),
// run once for a batch of tokens whose codes the linear kernels then stage.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 : 重みと活性値の両方を 4-bit に量子化": the draft mode quantises the activations as well.
// Per token m over all K: s_a = amax / qmax in fp32 (qmax = 7, or 127 for W4A8), codes =
// clamp(rint(x / s_a), -qmax - 1, qmax); s_a == 0 gives zeros.
#include "common.cuh"
#include "linear_internal.h"

namespace qspec {
namespace {

constexpr int kQThreads = 1024;

// One CTA per token: 16-byte loads of the row for the amax (bf16 bit patterns of |x| order like the
// values), then a second pass (from L2) writing 8 codes per 16-byte store: bf16 codes for the
// tensor-core path, or (f16 set) the GEMV's staged fp16 chunk, whose elements 2, 3, 6, 7 hold the
// code / 16 (exact in fp16).
__global__ void __launch_bounds__(kQThreads) quantise_kernel(const uint16_t* __restrict__ x, int K, int qbits, bool f16,
                                                             uint16_t* __restrict__ codes, float* __restrict__ s_a,
                                                             int8_t* __restrict__ xq_out, float* __restrict__ xs_out,
                                                             const WsGuard guard) {
  __shared__ int s_ok;
  // the codes go to the linear workspace: it must hold this shape's layout (or none yet)
  if (threadIdx.x == 0) s_ok = ws_claim(guard) ? 1 : 0;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(m) * K);
  const int n8 = K / 8;
  uint32_t mx = 0;
  for (int v = threadIdx.x; v < n8; v += kQThreads) {
    const uint4 u = __ldg(xr + v);
    mx = max(mx, max(max(u.x & 0x7FFFu, (u.x >> 16) & 0x7FFFu), max(u.y & 0x7FFFu, (u.y >> 16) & 0x7FFFu)));
    mx = max(mx, max(max(u.z & 0x7FFFu, (u.z >> 16) & 0x7FFFu), max(u.w & 0x7FFFu, (u.w >> 16) & 0x7FFFu)));
  }
  __shared__ unsigned int s_w[kQThreads / 32];
  __shared__ float s_scale[2];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (!s_ok) return;  // (uniform over the CTA: written before the barrier above)
  if (threadIdx.x < 32) {
    unsigned int v = s_w[threadIdx.x];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    if (threadIdx.x == 0) {
      const float sa = __fdiv_rn(__uint_as_float(v << 16), qbits == 8 ? 127.0f : 7.0f);
      s_scale[0] = sa;
      s_scale[1] = __frcp_rn(sa);
      s_a[m] = sa;
      if (xs_out) xs_out[m] = sa;
    }
  }
  __syncthreads();
  const float sa = s_scale[0], rsa = s_scale[1];
  const float qmax = qbits == 8 ? 127.0f : 7.0f;
  const bool fast = qbits == 4 && sa >= 0x1p-100f;  // see div_rn_markstein
  uint4* cr = reinterpret_cast<uint4*>(codes + static_cast<long long>(m) * K);
  uint2* qr = xq_out ? reinterpret_cast<uint2*>(xq_out + static_cast<long long>(m) * K) : nullptr;
  for (int v = threadIdx.x; v < n8; v += kQThreads) {
    const uint4 u = __ldg(xr + v);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t c[4];
    uint32_t q8[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float c0 = 0.0f, c1 = 0.0f;
      if (sa != 0.0f) {
        const float x0 = bf16_lo(w[i]), x1 = bf16_hi(w[i]);
        const float d0 = fast ? div_rn_markstein(x0, sa, rsa) : __fdiv_rn(x0, sa);
        const float d1 = fast ? div_rn_markstein(x1, sa, rsa) : __fdiv_rn(x1, sa);
        c0 = fminf(fmaxf(rintf(d0), -qmax - 1.0f), qmax);
        c1 = fminf(fmaxf(rintf(d1), -qmax - 1.0f), qmax);
      }
      if (f16) {
        const float f = (i & 1) ? 0.0625f : 1.0f;
        const __half2 h = __floats2half2_rn(c0 * f, c1 * f);
        c[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        c[i] = static_cast<uint32_t>(f32_to_bf16_bits(c0)) | (static_cast<uint32_t>(f32_to_bf16_bits(c1)) << 16);
      }
      q8[i >> 1] |= ((static_cast<uint32_t>(static_cast<int>(c0)) & 0xFFu) |
                     ((static_cast<uint32_t>(static_cast<int>(c1)) & 0xFFu) << 8))
                    << (16 * (i & 1));
    }
    cr[v] = make_uint4(c[0], c[1], c[2], c[3]);
    if (qr) qr[v] = make_uint2(q8[0], q8[1]);
  }
}

}  // namespace

qspec_status quantise_tokens(int abits, const uint16_t* x, int M, int K, bool gemv_layout, uint16_t* codes,
                             float* s_a, int8_t* xq_out, float* xs_out, const WsGuard& guard, cudaStream_t stream) {
  return launch_pdl(quantise_kernel, dim3(M), dim3(kQThreads), 0, stream, x, K, abits, gemv_layout, codes, s_a,
                    xq_out, xs_out, guard);
}

}  // namespace qspec
