// Steps a2 (W4A16 linear), a3 (per-token activation quantiser) and a4 (W4A4 linear) over the one
// shared packed INT4 weight tensor.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": W4A16 converts 4-bit weights while multiplying 16-bit activations; W4A4
// quantises the activations to 4 bits as well.  Section "QSpec の W4A4 モードと W4A16 モード":
// both modes read the same 4-bit weights.
//
// This file holds the argument checks, the entry points and the CUDA-core (SIMT) kernels, which
// serve when the tensor-core path of linear_tc.cu cannot (no TMA descriptor encoder in the driver).
#include "common.cuh"
#include "linear_internal.h"

namespace qspec {

namespace {

constexpr int kMT = 8;          // tokens per block
constexpr int kWarps = 8;       // output rows per block (one per warp)

// 32 packed nibbles (16 bytes) -> 32 signed codes as floats.
__device__ __forceinline__ void unpack32(const uint4 w, float (&c)[32]) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      // nibble t holds channel 8i + 2t (t < 4) or 8i + 2(t - 4) + 1 (t >= 4)
      const int nib = static_cast<int>((words[i] >> (4 * t)) & 0xFu);
      c[8 * i + (t < 4 ? 2 * t : 2 * (t - 4) + 1)] = static_cast<float>(nib >= 8 ? nib - 16 : nib);
    }
  }
}

// 32 consecutive bf16 activations -> fp32.
__device__ __forceinline__ void load_x32(const uint16_t* p, float (&x)[32]) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(v + i);
    const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      x[8 * i + 2 * t] = bf16_lo(words[t]);
      x[8 * i + 2 * t + 1] = bf16_hi(words[t]);
    }
  }
}

// Per-token activation quantiser of step a3: s_a = amax / qmax (fp32), code = clamp(rint(x / s_a),
// -qmax - 1, qmax); qmax = 7 (W4A4) or 127 (W4A8).
__device__ __forceinline__ float quant_act(float x, float s_a, float qmax) {
  if (s_a == 0.0f) return 0.0f;
  return fminf(fmaxf(rintf(__fdiv_rn(x, s_a)), -qmax - 1.0f), qmax);
}

// grid: (N / 8, ceil(M / 8)); block: 8 warps; warp w computes row n = 8 * blockIdx.x + w for the
// block's 8 tokens.  Lane l walks K in 32-weight chunks c = l, l + 32, ...; the 4 lanes sharing a
// 128-channel group in one pass are 4j..4j+3 (K % 128 == 0 keeps a group inside one pass).
template <int QB>
__global__ void __launch_bounds__(256) linear_simt_kernel(const uint16_t* __restrict__ x,
                                                          const uint8_t* __restrict__ Wp,
                                                          const __half* __restrict__ S, int M,
                                                          int N, int K, uint16_t* __restrict__ y,
                                                          int8_t* __restrict__ xq_out,
                                                          float* __restrict__ xs_out,
                                                          int32_t* __restrict__ acc_out) {
  __shared__ float s_amax[kMT];
  __shared__ float s_red[kWarps][kMT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + warp;
  const int m0 = blockIdx.y * kMT;
  const int mt = min(kMT, M - m0);
  const int G = K / kGroup;

  constexpr bool kA4 = QB != 0;  // activations quantised (W4A4 or W4A8)
  constexpr float kQmax = QB == 8 ? 127.0f : 7.0f;
  float s_a[kMT];
  if constexpr (kA4) {
    // Per-token amax over all of K (step a3), block-wide.
    for (int m = 0; m < kMT; ++m) {
      uint32_t mx = 0;
      if (m < mt) {
        const uint16_t* xr = x + static_cast<int64_t>(m0 + m) * K;
        for (int k = threadIdx.x; k < K; k += blockDim.x) mx = max(mx, static_cast<uint32_t>(xr[k]) & 0x7FFFu);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      if (lane == 0) s_red[warp][m] = __uint_as_float(mx << 16);
    }
    __syncthreads();
    if (threadIdx.x < kMT) {
      float a = 0.0f;
      for (int w = 0; w < kWarps; ++w) a = fmaxf(a, s_red[w][threadIdx.x]);
      s_amax[threadIdx.x] = __fdiv_rn(a, kQmax);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMT; ++m) s_a[m] = s_amax[m];
    if (blockIdx.x == 0) {
      if (xs_out && threadIdx.x < mt) xs_out[m0 + threadIdx.x] = s_a[threadIdx.x];
      if (xq_out) {
        for (int m = 0; m < mt; ++m) {
          const uint16_t* xr = x + static_cast<int64_t>(m0 + m) * K;
          for (int k = threadIdx.x; k < K; k += blockDim.x)
            xq_out[static_cast<int64_t>(m0 + m) * K + k] =
                static_cast<int8_t>(quant_act(bf16_lo(xr[k]), s_a[m], kQmax));
        }
      }
    }
  }

  float acc[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) acc[m] = 0.0f;

  const uint8_t* wrow = Wp + static_cast<int64_t>(n) * (K / 2);
  const int chunks = K / 32;
  for (int base = 0; base < chunks; base += 32) {
    const int c = base + lane;
    const bool valid = c < chunks;  // uniform over each 4-lane group set
    const int g = c >> 2;
    float code[32];
    if (valid) {
      unpack32(__ldg(reinterpret_cast<const uint4*>(wrow) + c), code);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) code[i] = 0.0f;
    }
    const float s = valid ? __half2float(S[static_cast<int64_t>(n) * G + g]) : 0.0f;
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      if (m < mt) {  // uniform across the warp
        float xv[32];
        if (valid) {
          load_x32(x + static_cast<int64_t>(m0 + m) * K + 32 * c, xv);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) xv[i] = 0.0f;
        }
        if constexpr (kA4) {
          int part = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) part += static_cast<int>(quant_act(xv[i], s_a[m], kQmax)) * static_cast<int>(code[i]);
          // exact group sum over the 4 lanes sharing group g
          part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
          part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
          if (valid && (lane & 3) == 0) {
            acc[m] += s * static_cast<float>(part);
            if (acc_out) acc_out[(static_cast<int64_t>(m0 + m) * N + n) * G + g] = part;
          }
        } else {
          float part = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) part = fmaf(xv[i], code[i], part);
          acc[m] = fmaf(s, part, acc[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kMT; ++m) {
    float v = acc[m];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0 && m < mt) {
      if constexpr (kA4) v *= s_a[m];
      y[static_cast<int64_t>(m0 + m) * N + n] = f32_to_bf16_bits(v);
    }
  }
}

}  // namespace

qspec_status linear_simt(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M,
                         int N, int K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                         cudaStream_t stream) {
  dim3 grid(N / kWarps, (M + kMT - 1) / kMT);
  const __half* Sh = reinterpret_cast<const __half*>(S);
  if (abits == 4)
    linear_simt_kernel<4><<<grid, 256, 0, stream>>>(x, Wp, Sh, M, N, K, y, xq_out, xs_out, acc_out);
  else if (abits == 8)
    linear_simt_kernel<8><<<grid, 256, 0, stream>>>(x, Wp, Sh, M, N, K, y, xq_out, xs_out, acc_out);
  else
    linear_simt_kernel<0><<<grid, 256, 0, stream>>>(x, Wp, Sh, M, N, K, y, nullptr, nullptr, nullptr);
  return launch_status();
}

}  // namespace qspec

namespace {
qspec_status check_linear_args(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                               int64_t N, int64_t K, const uint16_t* y) {
  using namespace qspec;
  if (!x || !Wp || !S || !y) return QSPEC_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return QSPEC_ERR_INVALID_ARG;
  if (M > QSPEC_MAX_M || N % 8 != 0 || K % kGroup != 0 || N > (int64_t(1) << 30) ||
      K > (int64_t(1) << 30) || N * K >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(Wp) || !aligned16(S) || !aligned16(y)) return QSPEC_ERR_MISALIGNED;
  return QSPEC_OK;
}
}  // namespace

extern "C" size_t qspec_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > QSPEC_MAX_M || N % 8 != 0 || K % qspec::kGroup != 0 ||
      N > (int64_t(1) << 30) || K > (int64_t(1) << 30))
    return 0;
  const size_t tc = qspec::linear_tc_workspace_size_all(int(M), int(N), int(K));
  return ((tc + 255) & ~size_t(255)) + qspec::gemv_workspace_bytes(int(M), int(N), int(K));
}

extern "C" qspec_status qspec_linear_w4a16(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                           int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                           size_t ws_bytes, qspec_stream_t stream) {
  const qspec_status st = check_linear_args(x, Wp, S, M, N, K, y);
  if (st != QSPEC_OK) return st;
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!qspec::aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_workspace_size(M, N, K)) return QSPEC_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (qspec::gemv_supported(int(M), int(N), int(K)))
    return qspec::gemv(16, x, Wp, S, int(M), int(N), int(K), y, nullptr, nullptr, nullptr, ws, s);
  if (qspec::linear_tc_supported(16, int(M), int(N), int(K)))
    return qspec::linear_tc(16, x, Wp, S, int(M), int(N), int(K), y, nullptr, nullptr, nullptr, ws, ws_bytes, s);
  return qspec::linear_simt(16, x, Wp, S, int(M), int(N), int(K), y, nullptr, nullptr, nullptr, s);
}

namespace {
// The quantised-activation linears (steps a3 + a4, and the W4A8 variant): abits = 4 or 8.
qspec_status linear_quantised(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                              int64_t N, int64_t K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                              void* ws, size_t ws_bytes, qspec_stream_t stream) {
  const qspec_status st = check_linear_args(x, Wp, S, M, N, K, y);
  if (st != QSPEC_OK) return st;
  if ((xq_out && !qspec::aligned16(xq_out)) || (xs_out && !qspec::aligned16(xs_out)) ||
      (acc_out && !qspec::aligned16(acc_out)))
    return QSPEC_ERR_MISALIGNED;
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!qspec::aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_workspace_size(M, N, K)) return QSPEC_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (qspec::gemv_supported(int(M), int(N), int(K)))
    return qspec::gemv(abits, x, Wp, S, int(M), int(N), int(K), y, xq_out, xs_out, acc_out, ws, s);
  if (qspec::linear_tc_supported(abits, int(M), int(N), int(K)))
    return qspec::linear_tc(abits, x, Wp, S, int(M), int(N), int(K), y, xq_out, xs_out, acc_out, ws, ws_bytes, s);
  return qspec::linear_simt(abits, x, Wp, S, int(M), int(N), int(K), y, xq_out, xs_out, acc_out, s);
}
}  // namespace

extern "C" qspec_status qspec_linear_w4a4(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                          int64_t M, int64_t N, int64_t K, uint16_t* y,
                                          int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws,
                                          size_t ws_bytes, qspec_stream_t stream) {
  return linear_quantised(4, x, Wp, S, M, N, K, y, xq_out, xs_out, acc_out, ws, ws_bytes, stream);
}

extern "C" qspec_status qspec_linear_w4a8(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                          int64_t M, int64_t N, int64_t K, uint16_t* y,
                                          int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws,
                                          size_t ws_bytes, qspec_stream_t stream) {
  return linear_quantised(8, x, Wp, S, M, N, K, y, xq_out, xs_out, acc_out, ws, ws_bytes, stream);
}
