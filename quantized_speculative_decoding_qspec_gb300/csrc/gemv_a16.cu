// Verify-mode (W4A16) linear for decode-sized M (1..8 tokens): register-resident dequantised
// weight fragments fed straight into warp-level tensor-core MMAs.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": W4A16 keeps the 16-bit activations and converts the 4-bit weights while
// multiplying.  At decode sizes the product is a GEMV bound by the weight stream (0.5 B per weight);
// the tcgen05 path would have to expand every weight to bf16 in TMEM (4x the streamed bytes, written
// and read back on chip), which measured slower than the HBM stream itself, so here the expanded
// weights never leave registers:
//
//  * a warp owns 16 weight rows x a K slice.  Lane (g, t) = (lane / 4, lane % 4) loads 16 bytes of
//    each of its two rows g and g + 8 per 128-channel group: packed words 4t..4t+3, i.e. channels
//    32t..32t+31 of the group;
//  * one shift + LOP3 + bf16 subtract turns a nibble pair of a word into an exact bf16x2 code pair
//    (the packed word keeps channels 2i and 2i+1 in nibbles i and i + 4), which is directly an A
//    fragment register of mma.m16n8k16: the MMA's 16 k-slots of lane t are mapped onto the
//    channels lane t holds (a fixed permutation of K inside the group), and the activations are
//    staged in shared memory in exactly that order, so one 16-byte shared load gives the B
//    fragments of two MMAs;
//  * per group the fp32 MMA result is scaled by s[n, g] and accumulated in fp32; K slices of a
//    tile are summed through shared memory in a fixed order; y is rounded to bf16 once.
//
// Tokens are the MMA's N = 8 side (rows >= M are zero), weight rows its M = 16 side.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "linear_internal.h"

namespace qspec {
namespace {

constexpr int kThreads = 512;  // 16 warps, one CTA per SM
constexpr int kWarps = kThreads / 32;

// 16 bytes of packed weights, read once: not kept in L1
__device__ __forceinline__ uint4 ld_weights(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// pair i of a packed word (channels 2i, 2i + 1 of its 8) -> exact bf16x2 codes
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int i) {
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43084308u));
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                   __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// d += A (16 x 16, row fragments a0..a3) * B (16 x 8, column fragments b0, b1), fp32 accumulate
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MT = token slots staged in shared memory (4 or 8); tokens >= M contribute zeros.  D = weight
// groups in flight per warp (a divisor of the groups per K slice, so that register slots line up
// with tile boundaries).
//
// A warp's work is one stream of (row tile, group) items: the tiles r * stride + blockIdx.x * per_cta
// + wtile for r = 0, 1, ..., and within each its K slice of groups.  Weights are fetched D items
// ahead across tile boundaries, so the stream never drains; the first fetches are issued before
// the kernel waits for its predecessor (no library kernel that may run ahead of this one writes
// packed weights or scales).
template <int MT, int D>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_a16_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ Wp, const __half* __restrict__ S,
                    int M, int N, int K, int KS, uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int G = K / kGroup;
  // activations: chunk ((gi * 4 + j) * MT + m) * 4 + t holds x[m, 128 gi + 32 t + 8 j .. + 7]
  uint4* xs = reinterpret_cast<uint4*>(sm);
  float4* red = reinterpret_cast<float4*>(xs + static_cast<size_t>(G) * 16 * MT);  // [2][kWarps][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  const int tiles = (N + 15) / 16;
  const int per_cta = kWarps / KS;  // row tiles a CTA works on at once
  const int wtile = warp / KS, ks = warp - wtile * KS;
  const int gs = G / KS, g_beg = ks * gs;
  const int stride = gridDim.x * per_cta;
  const int tile0 = blockIdx.x * per_cta + wtile;
  const int rounds = (tiles + stride - 1) / stride;  // the same for the KS warps of a tile slot
  const size_t row_bytes = static_cast<size_t>(K) / 2;

  // fetch cursor: the tile, its row pointers (at the slice's first group) and the group index
  const uint8_t* f_wlo = Wp;
  const uint8_t* f_whi = Wp;
  const __half* f_slo = S;
  const __half* f_shi = S;
  bool f_vlo = false, f_vhi = false;
  int f_tile = tile0, f_i = 0;
  auto point = [&]() {
    const int n_lo = f_tile * 16 + g, n_hi = n_lo + 8;
    f_vlo = f_tile < tiles && n_lo < N;
    f_vhi = f_tile < tiles && n_hi < N;
    f_wlo = Wp + static_cast<size_t>(f_vlo ? n_lo : 0) * row_bytes + g_beg * 64 + t * 16;
    f_whi = Wp + static_cast<size_t>(f_vhi ? n_hi : 0) * row_bytes + g_beg * 64 + t * 16;
    f_slo = S + static_cast<size_t>(f_vlo ? n_lo : 0) * G + g_beg;
    f_shi = S + static_cast<size_t>(f_vhi ? n_hi : 0) * G + g_beg;
  };
  uint4 wl[D], wh[D];
  float sl[D], sh[D];
  auto fetch = [&](int k) {  // next item of the stream into register slot k
    wl[k] = f_vlo ? ld_weights(f_wlo + f_i * 64) : make_uint4(0, 0, 0, 0);
    wh[k] = f_vhi ? ld_weights(f_whi + f_i * 64) : make_uint4(0, 0, 0, 0);
    sl[k] = f_vlo ? __half2float(f_slo[f_i]) : 0.0f;
    sh[k] = f_vhi ? __half2float(f_shi[f_i]) : 0.0f;
    if (++f_i == gs) {
      f_i = 0;
      f_tile += stride;
      point();
    }
  };
  point();
#pragma unroll
  for (int k = 0; k < D; ++k) fetch(k);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int c = threadIdx.x; c < G * 16 * MT; c += kThreads) {
    const int ct = c & 3, cm = (c >> 2) % MT, rest = c / (4 * MT);
    const int cj = rest & 3, gi = rest >> 2;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (cm < M)
      v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(cm) * K + gi * 128 + ct * 32 + cj * 8));
    xs[c] = v;
  }
  __syncthreads();

  for (int r = 0; r < rounds; ++r) {
    const int tile = r * stride + tile0;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // rows (tile * 16 + g, + 8) x tokens (2t, 2t + 1)
    for (int i0 = 0; i0 < gs; i0 += D) {
#pragma unroll
      for (int k = 0; k < D; ++k) {
        const uint4* xg = xs + static_cast<size_t>(g_beg + i0 + k) * 16 * MT;
        const uint32_t lo[4] = {wl[k].x, wl[k].y, wl[k].z, wl[k].w};
        const uint32_t hi[4] = {wh[k].x, wh[k].y, wh[k].z, wh[k].w};
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 xb = make_uint4(0, 0, 0, 0);
          if (MT == 8 || g < MT) xb = xg[(j * MT + g) * 4 + t];
          mma_16816(d, code_pair(lo[j], 0), code_pair(hi[j], 0), code_pair(lo[j], 1), code_pair(hi[j], 1), xb.x,
                    xb.y);
          mma_16816(d, code_pair(lo[j], 2), code_pair(hi[j], 2), code_pair(lo[j], 3), code_pair(hi[j], 3), xb.z,
                    xb.w);
        }
        acc[0] = fmaf(sl[k], d[0], acc[0]);
        acc[1] = fmaf(sl[k], d[1], acc[1]);
        acc[2] = fmaf(sh[k], d[2], acc[2]);
        acc[3] = fmaf(sh[k], d[3], acc[3]);
        fetch(k);
      }
    }
    if (KS > 1) {  // K slices summed in slice order by the slice-0 warp of the tile slot
      float4* rb = red + (r & 1) * kWarps * 32;
      rb[warp * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + wtile), "r"(KS * 32) : "memory");
      if (ks == 0) {
        float4 s4 = rb[warp * 32 + lane];
        for (int j = 1; j < KS; ++j) {
          const float4 o = rb[(warp + j) * 32 + lane];
          s4.x += o.x;
          s4.y += o.y;
          s4.z += o.z;
          s4.w += o.w;
        }
        acc[0] = s4.x;
        acc[1] = s4.y;
        acc[2] = s4.z;
        acc[3] = s4.w;
      }
    }
    if (ks == 0 && tile < tiles) {
      const int n_lo = tile * 16 + g, n_hi = n_lo + 8;
      const int m0 = 2 * t, m1 = 2 * t + 1;
      if (n_lo < N && m0 < M) y[static_cast<size_t>(m0) * N + n_lo] = f32_to_bf16_bits(acc[0]);
      if (n_lo < N && m1 < M) y[static_cast<size_t>(m1) * N + n_lo] = f32_to_bf16_bits(acc[1]);
      if (n_hi < N && m0 < M) y[static_cast<size_t>(m0) * N + n_hi] = f32_to_bf16_bits(acc[2]);
      if (n_hi < N && m1 < M) y[static_cast<size_t>(m1) * N + n_hi] = f32_to_bf16_bits(acc[3]);
    }
  }
}

size_t smem_bytes(int MT, int K) {
  return static_cast<size_t>(K / kGroup) * 16 * MT * 16 + 2 * static_cast<size_t>(kWarps) * 32 * 16;
}

template <int MT, int D>
qspec_status launch_d(const uint16_t* x, const uint8_t* Wp, const __half* S, int M, int N, int K, uint16_t* y,
                      int best_ks, int best_grid, cudaStream_t stream) {
  const size_t smem = smem_bytes(MT, K);
  auto kern = gemv_a16_kernel<MT, D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return QSPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(best_grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, x, Wp, S, M, N, K, best_ks, y) == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

template <int MT>
qspec_status launch(const uint16_t* x, const uint8_t* Wp, const __half* S, int M, int N, int K, uint16_t* y,
                    cudaStream_t stream) {
  const int G = K / kGroup;
  const long long tiles = (static_cast<long long>(N) + 15) / 16;
  const int sms = num_sms();
  // K split: the fewest rounds of (groups per slice + fixed cost), ties to the wider grid
  int best_ks = 1, best_grid = 1;
  long long best_cost = -1;
  for (int ks = 1; ks <= 16; ks *= 2) {
    if (G % ks != 0) continue;
    const long long slots = kWarps / ks;
    const int grid = static_cast<int>(std::min<long long>(sms, (tiles + slots - 1) / slots));
    const long long rounds = (tiles + grid * slots - 1) / (grid * slots);
    const long long cost = rounds * (G / ks + 2);
    if (best_cost < 0 || cost < best_cost || (cost == best_cost && grid > best_grid)) {
      best_cost = cost;
      best_ks = ks;
      best_grid = grid;
    }
  }
  const int gs = G / best_ks;
  if (gs % 4 == 0) return launch_d<MT, 4>(x, Wp, S, M, N, K, y, best_ks, best_grid, stream);
  if (gs % 2 == 0) return launch_d<MT, 2>(x, Wp, S, M, N, K, y, best_ks, best_grid, stream);
  return launch_d<MT, 1>(x, Wp, S, M, N, K, y, best_ks, best_grid, stream);
}

}  // namespace

bool gemv_a16_supported(int M, int N, int K) {
  if (M < 1 || M > 8 || N < 1 || K % kGroup != 0) return false;
  return smem_bytes(M <= 4 ? 4 : 8, K) <= 200 * 1024;
}

qspec_status gemv_a16(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K, uint16_t* y,
                      cudaStream_t stream) {
  const __half* Sh = reinterpret_cast<const __half*>(S);
  return M <= 4 ? launch<4>(x, Wp, Sh, M, N, K, y, stream) : launch<8>(x, Wp, Sh, M, N, K, y, stream);
}

}  // namespace qspec
