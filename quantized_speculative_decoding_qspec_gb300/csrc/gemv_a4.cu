// Draft-mode (W4A4) linear for decode-sized M (1..4 tokens) on the CUDA cores.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 : 重みと活性値の両方を 4-bit に量子化": weights and activations are both 4-bit, so the
// product is an integer dot product.  Here it runs on the SM's integer dot-product unit (dp4a):
//
//  * activations are quantised per token once per CTA (amax over all K, s_a = amax / 7 in fp32,
//    codes = clamp(rint(x / s_a), -8, 7)) and kept in shared memory, pre-arranged so that one
//    32-bit word of packed weight nibbles meets two 32-bit words of activation codes;
//  * a weight word w (channels k0..k7 as two's complement nibbles in the packed order k0, k2, k4,
//    k6, k1, k3, k5, k7) becomes two vectors of signed bytes by moving each nibble into the high
//    half of its byte: (w << 4) & 0xF0F0F0F0 holds k0, k4, k1, k5 and w & 0xF0F0F0F0 holds k2, k6,
//    k3, k7, each byte equal to 16 * code; dp4a against activation words laid out in the same
//    channel order gives 16 * sum(code * a) exactly, and the 1/16 is folded into the fp32 group
//    scale, so every 128-channel group sum is the exact integer sum of code * a;
//  * y[m, n] = s_a[m] * sum_g s[n, g] * acc[m, n, g] in fp32, rounded to bf16 once.
//
// Work split: a warp covers RPW weight rows x (32 / RPW) lanes along K (RPW = 1 for one token, 4
// for three or four), so each load instruction reads RPW contiguous row segments and each
// activation word is broadcast to RPW lanes.  KS warps of
// a CTA share one group of rows and split K (KS = 1 for wide layers, up to 8 for narrow ones); CTAs
// loop over row groups.  Memory-bound on the packed weights: 0.5 B + 1/64 B per weight.
#include <algorithm>

#include "common.cuh"
#include "linear_internal.h"

namespace qspec {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kBatch = 4;      // chunks loaded per lane before they are consumed
// Rows per warp: fewer rows give longer contiguous segments per load instruction; more rows share
// each activation word between more lanes (shared-memory traffic per weight is M / RPW bytes).
constexpr int kRowsPerWarpM1 = 1;

__device__ __forceinline__ int dp4a_s32(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Per-token quantiser (step a3) into shared memory: codes per 32-channel chunk as 8 words
// (word 2t holds k = 8t+0,4,1,5 and word 2t+1 holds k = 8t+2,6,3,7 as signed bytes, matching the
// two byte vectors of a packed weight word) and the chunk sum of the codes.
template <int M>
__device__ void quantise_tokens(const uint16_t* __restrict__ x, int K, uint32_t* codes, int* csum, float* s_a,
                                unsigned int* amax_bits, int8_t* __restrict__ xq_out, float* __restrict__ xs_out) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int C = K / 32;
  if (tid < M) amax_bits[tid] = 0;
  __syncthreads();
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(m) * K);
    uint32_t mx = 0;
    for (int i = tid; i < K / 8; i += kThreads) {
      const uint4 v = __ldg(xr + i);
      mx = max(mx, max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu)));
      mx = max(mx, max(max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu)));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) atomicMax(&amax_bits[m], mx);
  }
  __syncthreads();
  if (tid < M) {
    s_a[tid] = __fdiv_rn(__uint_as_float(amax_bits[tid] << 16), 7.0f);
    if (xs_out && blockIdx.x == 0) xs_out[tid] = s_a[tid];
  }
  __syncthreads();
  for (int i = tid; i < M * C; i += kThreads) {
    const int m = i / C, c = i - m * C;
    const float sa = s_a[m];
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(m) * K + 32 * c);
    int q[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 u = __ldg(xr + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {
          const float xv = hl ? bf16_hi(w[e]) : bf16_lo(w[e]);
          q[8 * v + 2 * e + hl] =
              sa == 0.0f ? 0 : static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(xv, sa)), -8.0f), 7.0f));
        }
      }
    }
    int sum = 0;
    uint32_t out[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t ev = 0, od = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // byte j of the even-nibble vector is channel 4(j & 1) + (j >> 1); of the odd one, that + 2
        const int k = 8 * t + 4 * (j & 1) + (j >> 1);
        ev |= (static_cast<uint32_t>(q[k]) & 0xFFu) << (8 * j);
        od |= (static_cast<uint32_t>(q[k + 2]) & 0xFFu) << (8 * j);
        sum += q[k] + q[k + 2];
      }
      out[2 * t] = ev;
      out[2 * t + 1] = od;
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + (static_cast<long long>(m) * C + c) * 8);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    csum[m * C + c] = sum;
    if (xq_out && blockIdx.x == 0) {
      int8_t* xo = xq_out + static_cast<long long>(m) * K + 32 * c;
#pragma unroll
      for (int k = 0; k < 32; ++k) xo[k] = static_cast<int8_t>(q[k]);
    }
  }
  __syncthreads();
}

template <int M, int RPW>
__global__ void __launch_bounds__(kThreads, 3) gemv_a4_kernel(const uint16_t* __restrict__ x,
                                                             const uint8_t* __restrict__ Wp,
                                                             const __half* __restrict__ S, int N, int K, int KS,
                                                             uint16_t* __restrict__ y, int8_t* __restrict__ xq_out,
                                                             float* __restrict__ xs_out,
                                                             int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int C = K / 32;  // 32-channel chunks per row
  const int G = K / kGroup;
  uint32_t* codes = reinterpret_cast<uint32_t*>(sm);                          // [M][C][8]
  int* csum = reinterpret_cast<int*>(codes + static_cast<size_t>(M) * C * 8);  // [M][C] (quantiser scratch)
  float* red = reinterpret_cast<float*>(csum + M * C);                         // [8 warps][RPW rows][M]
  __shared__ unsigned int amax_bits[M];
  __shared__ float s_a[M];

  constexpr int LPR = 32 / RPW;  // lanes per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane / LPR, kl = lane % LPR;
  const int wg = warp / KS, ks = warp - wg * KS;  // row group within the CTA, K slice
  const int groups_per_cta = 8 / KS;
  const int cs = C / KS;  // chunks per K slice (a multiple of 4: slices hold whole groups)
  const int c_beg = ks * cs, c_end = c_beg + cs;
  const int row_step = gridDim.x * groups_per_cta * RPW;
  const int cta_first = blockIdx.x * groups_per_cta * RPW;
  // Every warp of the CTA walks the same (row-group iteration, batch) items, so the CTA-level
  // reductions and every full-warp shuffle are reached by all lanes.
  const int nb = (cs + LPR * kBatch - 1) / (LPR * kBatch);  // batches per row group
  const int iters = cta_first < N ? (N - cta_first + row_step - 1) / row_step : 0;
  const size_t row_bytes = static_cast<size_t>(K) / 2;

  // item cursor (iteration, batch) advanced without divisions
  auto load_item = [&](int it, int bi, uint4 (&wv)[kBatch], float (&sg)[kBatch]) {
    const int n = cta_first + it * row_step + wg * RPW + r;
    const bool valid = it < iters && n < N;
    const uint8_t* wrow = Wp + (valid ? static_cast<size_t>(n) : 0) * row_bytes;
    const __half* srow = S + (valid ? static_cast<size_t>(n) : 0) * G;
    const int cb = c_beg + bi * LPR * kBatch + kl;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int c = cb + LPR * b;
      const bool ok = valid && c < c_end;
      wv[b] = ok ? ld_stream_v4(wrow + 16 * c) : make_uint4(0, 0, 0, 0);
      // the nibble sits in the high half of each byte below, so every product is 16x too large
      sg[b] = ok ? __half2float(srow[c >> 2]) * 0.0625f : 0.0f;
    }
  };

  uint4 wa[kBatch], wb[kBatch];
  float sa_[kBatch], sb_[kBatch];
  // The first weights are requested before waiting for the predecessor kernel (no library kernel
  // that may run ahead of this one writes packed weights or scales), so their latency overlaps its
  // tail and the activation quantiser below.
  load_item(0, 0, wa, sa_);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  quantise_tokens<M>(x, K, codes, csum, s_a, amax_bits, xq_out, xs_out);

  float yacc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) yacc[m] = 0.0f;

  auto consume = [&](int it, int bi, const uint4 (&wv)[kBatch], const float (&sg)[kBatch]) {
    const int n = cta_first + it * row_step + wg * RPW + r;
    const bool valid = n < N;
    const int cb = c_beg + bi * LPR * kBatch + kl;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int c = cb + LPR * b;
      const bool in = c < c_end;  // uniform across each 4-lane set that shares a 128-channel group
      const uint32_t w[4] = {wv[b].x, wv[b].y, wv[b].z, wv[b].w};
      // signed bytes 16 * code: nibbles 0, 2, 4, 6 shifted into the high half of their byte,
      // nibbles 1, 3, 5, 7 masked there
      uint32_t ev[4], od[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        ev[t] = (w[t] << 4) & 0xF0F0F0F0u;
        od[t] = w[t] & 0xF0F0F0F0u;
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        int acc = 0;
        if (in) {
          const uint4* ap = reinterpret_cast<const uint4*>(codes + (m * C + c) * 8);
          const uint4 a0 = ap[0], a1 = ap[1];
          acc = dp4a_s32(ev[0], a0.x, acc);
          acc = dp4a_s32(od[0], a0.y, acc);
          acc = dp4a_s32(ev[1], a0.z, acc);
          acc = dp4a_s32(od[1], a0.w, acc);
          acc = dp4a_s32(ev[2], a1.x, acc);
          acc = dp4a_s32(od[2], a1.y, acc);
          acc = dp4a_s32(ev[3], a1.z, acc);
          acc = dp4a_s32(od[3], a1.w, acc);
        }
        if (acc_out) {  // exact 128-channel group sum over the 4 lanes of the group (all lanes shuffle)
          int gsum = acc + __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
          gsum += __shfl_xor_sync(0xFFFFFFFFu, gsum, 2);
          if (in && valid && (kl & 3) == 0)
            acc_out[(static_cast<size_t>(m) * N + n) * G + (c >> 2)] = gsum >> 4;  // exact: a multiple of 16
        }
        yacc[m] = fmaf(sg[b], static_cast<float>(acc), yacc[m]);
      }
    }
    if (bi != nb - 1) return;
    // end of the row group: reduce over the lanes of each row, then over the KS warps
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = yacc[m];
#pragma unroll
      for (int off = 1; off < LPR; off <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      yacc[m] = v;
    }
    if (KS == 1) {
      if (kl == 0 && valid) {
#pragma unroll
        for (int m = 0; m < M; ++m) y[static_cast<size_t>(m) * N + n] = f32_to_bf16_bits(yacc[m] * s_a[m]);
      }
    } else {
      if (kl == 0) {
#pragma unroll
        for (int m = 0; m < M; ++m) red[(warp * RPW + r) * M + m] = yacc[m];
      }
      __syncthreads();
      if (ks == 0 && kl == 0 && valid) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = 0.0f;
          for (int j = 0; j < KS; ++j) v += red[((wg * KS + j) * RPW + r) * M + m];
          y[static_cast<size_t>(m) * N + n] = f32_to_bf16_bits(v * s_a[m]);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < M; ++m) yacc[m] = 0.0f;
  };

  // two register batches: the next item's loads are issued before the current one is consumed
  int it = 0, bi = 0;
  auto advance = [&](int& i_, int& b_) {
    if (++b_ == nb) {
      b_ = 0;
      ++i_;
    }
  };
  while (it < iters) {
    int it1 = it, bi1 = bi;
    advance(it1, bi1);
    load_item(it1, bi1, wb, sb_);
    consume(it, bi, wa, sa_);
    if (it1 >= iters) break;
    int it2 = it1, bi2 = bi1;
    advance(it2, bi2);
    load_item(it2, bi2, wa, sa_);
    consume(it1, bi1, wb, sb_);
    it = it2;
    bi = bi2;
  }
}

template <int M, int RPW>
qspec_status launch_gemv_a4(const uint16_t* x, const uint8_t* Wp, const __half* S, int N, int K, uint16_t* y,
                            int8_t* xq_out, float* xs_out, int32_t* acc_out, cudaStream_t stream) {
  const int C = K / 32, G = K / kGroup;
  // Split K over KS warps of a CTA only when whole rows per warp would leave the persistent grid
  // (3 resident CTAs per SM) less than half filled: thinner K slices cost a CTA-wide reduction
  // per row group, which measured slower than an uneven last iteration.
  const long long row_groups = (static_cast<long long>(N) + RPW - 1) / RPW;
  const long long resident = 3LL * num_sms();
  int KS = 1;
  while (KS < 8 && (row_groups + (8 / KS) - 1) / (8 / KS) < resident / 2 && G % (KS * 2) == 0) KS *= 2;
  const long long ctas_needed = (row_groups + (8 / KS) - 1) / (8 / KS);
  const int grid = static_cast<int>(std::min<long long>(ctas_needed, resident));
  const size_t smem = static_cast<size_t>(M) * C * 32 + static_cast<size_t>(M) * C * 4 + 8 * RPW * M * sizeof(float);
  auto kern = gemv_a4_kernel<M, RPW>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return QSPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, x, Wp, S, N, K, KS, y, xq_out, xs_out, acc_out) == cudaSuccess
             ? QSPEC_OK
             : QSPEC_ERR_CUDA;
}

}  // namespace

bool gemv_a4_supported(int M, int N, int K) {
  // activation codes for all of K stay in shared memory
  return M >= 1 && M <= 4 && N >= 1 && static_cast<size_t>(M) * K * 9 / 8 + 512 <= 200 * 1024;
}

qspec_status gemv_a4(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K, uint16_t* y,
                     int8_t* xq_out, float* xs_out, int32_t* acc_out, cudaStream_t stream) {
  const __half* Sh = reinterpret_cast<const __half*>(S);
  switch (M) {
    case 1: return launch_gemv_a4<1, kRowsPerWarpM1>(x, Wp, Sh, N, K, y, xq_out, xs_out, acc_out, stream);
    case 2: return launch_gemv_a4<2, 2>(x, Wp, Sh, N, K, y, xq_out, xs_out, acc_out, stream);
    case 3: return launch_gemv_a4<3, 4>(x, Wp, Sh, N, K, y, xq_out, xs_out, acc_out, stream);
    default: return launch_gemv_a4<4, 4>(x, Wp, Sh, N, K, y, xq_out, xs_out, acc_out, stream);
  }
}

}  // namespace qspec
