// Building blocks of the speculative decode loop around the hot path: a row gather (embedding
// lookup, reordering logits rows) and per-row next-token selection.
//
// Tutorial "Speculative Decodingとは？LLM生成を速くする方法" (kasblo.com), section "draft modelと
// target modelの処理フロー": the draft model extends the prefix one token at a time, gamma times,
// each token chosen from its own distribution q (the most likely token when decoding greedily,
// a draw from q when sampling); the target then scores the prefix plus the gamma candidates at once.
#include <float.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace qspec {

__device__ unsigned int g_decode_error = 0;  // bit 2: a gather index was out of range

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelVec = 8;                       // elements per thread and tile in the scan pass
constexpr int kSelTile = kSelThreads * kSelVec;

// ------------------------------------------------------------------ row gather

// dst[m, :] = src[idx[m], :] for rows of row_bytes; U is the copy unit (uint4 when row_bytes is a
// multiple of 16, else uint32).  Out-of-range ids give a zero row and set the decode error bit.
template <typename U>
__global__ void __launch_bounds__(256) gather_rows_kernel(const U* __restrict__ src, int64_t n_src,
                                                          int64_t row_units, const int32_t* __restrict__ idx,
                                                          U* __restrict__ dst) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t m = blockIdx.x;
  const int32_t r = idx[m];
  const bool ok = r >= 0 && r < n_src;
  if (!ok && threadIdx.x == 0) atomicOr(&g_decode_error, 4u);
  const U* s = src + int64_t(ok ? r : 0) * row_units;
  U* d = dst + m * row_units;
  for (int64_t v = threadIdx.x; v < row_units; v += blockDim.x) d[v] = ok ? s[v] : U{};
}

// Gathers of rows of a few bytes (token ids): one thread per row.
__global__ void __launch_bounds__(256) gather_words_kernel(const uint32_t* __restrict__ src, int64_t n_src,
                                                           int64_t row_units, const int32_t* __restrict__ idx,
                                                           int64_t n, uint32_t* __restrict__ dst) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t m = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (m >= n) return;
  const int32_t r = idx[m];
  const bool ok = r >= 0 && r < n_src;
  if (!ok) atomicOr(&g_decode_error, 4u);
  for (int64_t v = 0; v < row_units; ++v) dst[m * row_units + v] = ok ? src[int64_t(r) * row_units + v] : 0u;
}

// ------------------------------------------------------------------ token selection

__device__ __forceinline__ void take_max(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
}

struct MS {
  float m, s;
};

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.0f};
  return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

__device__ __forceinline__ void ms_add(MS& a, float v) {
  if (v > a.m) {
    a.s = a.m == -INFINITY ? 0.0f : a.s * expf(a.m - v);
    a.m = v;
  }
  if (a.m != -INFINITY) a.s += expf(v - a.m);
}

template <typename T, typename F>
__device__ __forceinline__ T block_reduce(T v, F op, T* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = op(v, T::shfl(v, off));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  v = sh[lane < kSelThreads / 32 ? lane : 0];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = op(v, T::shfl(v, off));
  __syncthreads();
  return v;
}

struct ArgMax {
  float v;
  int i;
  __device__ static ArgMax shfl(ArgMax a, int off) {
    return {__shfl_xor_sync(0xFFFFFFFFu, a.v, off), __shfl_xor_sync(0xFFFFFFFFu, a.i, off)};
  }
};
struct MSv {
  MS a;
  __device__ static MSv shfl(MSv x, int off) {
    return {{__shfl_xor_sync(0xFFFFFFFFu, x.a.m, off), __shfl_xor_sync(0xFFFFFFFFu, x.a.s, off)}};
  }
};

// Loads element j of a bf16 row as fp32 (j < V); out-of-row slots read as -inf.
__device__ __forceinline__ float load_logit(const uint16_t* __restrict__ rp, int j, int V) {
  return j < V ? bf16_lo(rp[j]) : -INFINITY;
}

// One CTA per row.  u == NULL: the most likely token (lowest index among equal maxima).  Otherwise
// the smallest j with sum_{i<=j} exp(l_i - m) > u[row] * sum_i exp(l_i - m) (inverse CDF in index
// order, strict '>'); if rounding leaves no such j, the last j with a nonzero term.
template <bool kVec>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const uint16_t* __restrict__ L, int V,
                                                             const float* __restrict__ u,
                                                             int32_t* __restrict__ tok) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t row = blockIdx.x;
  const uint16_t* rp = L + row * V;
  __shared__ ArgMax sh_am[kSelThreads / 32];
  __shared__ MSv sh_ms[kSelThreads / 32];

  if (u == nullptr) {
    ArgMax a{-INFINITY, INT_MAX};
    if (kVec) {
      const uint4* vp = reinterpret_cast<const uint4*>(rp);
      for (int v = threadIdx.x; v < V / 8; v += kSelThreads) {
        const uint4 w = __ldg(vp + v);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          take_max(a.v, a.i, bf16_lo(ww[e]), 8 * v + 2 * e);
          take_max(a.v, a.i, bf16_hi(ww[e]), 8 * v + 2 * e + 1);
        }
      }
    } else {
      for (int j = threadIdx.x; j < V; j += kSelThreads) take_max(a.v, a.i, bf16_lo(rp[j]), j);
    }
    a = block_reduce(a, [](ArgMax x, ArgMax y) { take_max(x.v, x.i, y.v, y.i); return x; }, sh_am);
    if (threadIdx.x == 0) tok[row] = a.i == INT_MAX ? 0 : a.i;
    return;
  }

  // pass 1: max and sum of exp(l - max)
  MSv st{{-INFINITY, 0.0f}};
  if (kVec) {
    const uint4* vp = reinterpret_cast<const uint4*>(rp);
    for (int v = threadIdx.x; v < V / 8; v += kSelThreads) {
      const uint4 w = __ldg(vp + v);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ms_add(st.a, bf16_lo(ww[e]));
        ms_add(st.a, bf16_hi(ww[e]));
      }
    }
  } else {
    for (int j = threadIdx.x; j < V; j += kSelThreads) ms_add(st.a, bf16_lo(rp[j]));
  }
  st = block_reduce(st, [](MSv x, MSv y) { return MSv{ms_merge(x.a, y.a)}; }, sh_ms);
  const float m = st.a.m, S = st.a.s;
  if (m == -INFINITY || !(S > 0.0f)) {
    if (threadIdx.x == 0) tok[row] = 0;
    return;
  }
  const float T = u[row] * S;

  // pass 2: tiles of kSelThreads x kSelVec consecutive elements.  P_t = running sum up to the end of
  // thread t's elements (block scan); the first thread with P_t > T holds the crossing, which it finds
  // by adding its own terms to P_{t-1}.  Every decision compares the same computed P values, so
  // exactly one thread answers even where fp32 rounding makes the scan and the walk disagree.
  __shared__ float sh_sum[kSelThreads / 32];
  __shared__ float sh_last[kSelThreads / 32];
  __shared__ int s_thr;
  __shared__ int s_last_nz;
  if (threadIdx.x == 0) { s_thr = INT_MAX; s_last_nz = -1; }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float base = 0.0f;
  bool found = false;
  for (int t0 = 0; t0 < V; t0 += kSelTile) {
    const int j0 = t0 + threadIdx.x * kSelVec;
    float r[kSelVec];
    float mine = 0.0f;
    int last_nz = -1;
#pragma unroll
    for (int e = 0; e < kSelVec; ++e) {
      r[e] = expf(load_logit(rp, j0 + e, V) - m);
      mine += r[e];
      if (r[e] > 0.0f) last_nz = j0 + e;
    }
    float incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) sh_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      float w = sh_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xFFFFFFFFu, w, off);
        if (lane >= off) w += o;
      }
      sh_sum[lane] = w;
    }
    __syncthreads();
    const float P = base + (warp > 0 ? sh_sum[warp - 1] : 0.0f) + incl;
    if (lane == 31) sh_last[warp] = P;
    __syncthreads();
    float Pprev = __shfl_up_sync(0xFFFFFFFFu, P, 1);
    if (lane == 0) Pprev = warp > 0 ? sh_last[warp - 1] : base;
    if (P > T) atomicMin(&s_thr, static_cast<int>(threadIdx.x));
    if (last_nz >= 0) atomicMax(&s_last_nz, last_nz);
    __syncthreads();
    if (s_thr != INT_MAX) {
      if (threadIdx.x == static_cast<unsigned int>(s_thr)) {
        float c = Pprev;
        int hit = -1;
#pragma unroll
        for (int e = 0; e < kSelVec; ++e) {
          c += r[e];
          if (hit < 0 && c > T) hit = j0 + e;
        }
        tok[row] = hit >= 0 ? hit : (last_nz >= 0 ? last_nz : j0);
      }
      found = true;
      break;
    }
    base = sh_last[kSelThreads / 32 - 1];
  }
  if (!found && threadIdx.x == 0) tok[row] = s_last_nz >= 0 ? s_last_nz : 0;
}

}  // namespace

qspec_status read_and_clear_decode_error(cudaStream_t s, unsigned int* bits) {
  *bits = 0;
  if (cudaMemcpyFromSymbolAsync(bits, g_decode_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QSPEC_ERR_CUDA;
  if (*bits) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return QSPEC_ERR_CUDA;
  }
  return QSPEC_OK;
}

}  // namespace qspec

using namespace qspec;

extern "C" qspec_status qspec_gather_rows(const void* src, int64_t n_src, int64_t row_bytes, const int32_t* idx,
                                          int64_t n, void* dst, qspec_stream_t stream) {
  if (!src || !idx || !dst || n_src <= 0 || row_bytes <= 0 || n <= 0) return QSPEC_ERR_INVALID_ARG;
  if (row_bytes % 4 != 0 || n > INT_MAX || n_src > (int64_t(1) << 40) / row_bytes)
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if ((reinterpret_cast<uintptr_t>(idx) & 3u) != 0) return QSPEC_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (row_bytes % 16 == 0 && row_bytes >= 1024) {
    if (!aligned16(src) || !aligned16(dst)) return QSPEC_ERR_MISALIGNED;
    return launch_pdl(gather_rows_kernel<uint4>, dim3(unsigned(n)), dim3(256), 0, s, static_cast<const uint4*>(src),
                      n_src, row_bytes / 16, idx, static_cast<uint4*>(dst));
  }
  if ((reinterpret_cast<uintptr_t>(src) & 3u) != 0 || (reinterpret_cast<uintptr_t>(dst) & 3u) != 0)
    return QSPEC_ERR_MISALIGNED;
  return launch_pdl(gather_words_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, s,
                    static_cast<const uint32_t*>(src), n_src, row_bytes / 4, idx, n, static_cast<uint32_t*>(dst));
}

extern "C" qspec_status qspec_select_tokens(const uint16_t* logits, int32_t R, int32_t V, const float* u,
                                            int32_t* tok, qspec_stream_t stream) {
  if (!logits || !tok || R <= 0 || V <= 0) return QSPEC_ERR_INVALID_ARG;
  if (V < 2 || V > QSPEC_MAX_V || int64_t(R) * V >= (int64_t(1) << 40)) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(logits) || (reinterpret_cast<uintptr_t>(tok) & 3u) || (reinterpret_cast<uintptr_t>(u) & 3u))
    return QSPEC_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (V % 8 == 0) return launch_pdl(select_kernel<true>, dim3(unsigned(R)), dim3(kSelThreads), 0, s, logits, int(V), u, tok);
  return launch_pdl(select_kernel<false>, dim3(unsigned(R)), dim3(kSelThreads), 0, s, logits, int(V), u, tok);
}
