// One launch for a whole pass of decode-size linears (W4A16, W4A4 or W4A8 over a list of layers):
// the register-fragment GEMV of gemv_impl.cuh made persistent across layers.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "QSpec の W4A4 モードと W4A16 モード": a draft pass runs every linear of the model in W4A4 mode, a
// verify pass runs them in W4A16 mode, both over the same packed weights.  At decode sizes each
// linear is a stream of its 4-bit weights; a layer of a few megabytes lasts only a few microseconds,
// about what a launch costs in latency (CTA start, first DRAM round trip, activation staging, tail).
// Here one CTA per SM stays resident for the whole pass:
//
//  * every warp's weight stream (D groups in flight, as in the GEMV) runs on across layer
//    boundaries, so the next layer's first weights are in flight while the current one finishes;
//  * the next layer's activations are copied into shared memory with cp.async while the current
//    layer streams (each layer has its own place in a ring of staged activations);
//  * a layer marked as reading what earlier layers of the pass wrote (q, k, v -> o -> gate, up ->
//    down -> lm_head in a decoder) is preceded by a grid-wide barrier: every CTA arrives after its
//    outputs are visible and waits, with an iteration limit, for the others (on expiry the CTA sets
//    the timeout bit and leaves);
//  * consecutive layers with the same K and no barrier between them form a segment whose tiles are
//    dealt to the grid as one list (so the grid stays balanced up to each barrier); a segment with
//    fewer tiles than tile slots starts where the previous one left off, keeping other SMs busy.
//
// Measured on one GB300 (CUDA graphs of back-to-back passes): the eight Llama-3-8B-shaped decode
// linears in W4A4 at one token take 93 us as one pass without barriers against 102 us as eight
// GEMV launches; each grid barrier costs about 4 us (the tail of the earlier layers, the arrival and
// release, and restaging the activations), more than a kernel boundary under programmatic
// dependent launch, so dependent layers are better served by separate launches and the barrier is
// for callers without that choice.
//
// Arithmetic per layer is exactly the GEMV's (same conversion, MMA, group scaling, K-slice order).
#pragma once

#include "gemv_impl.cuh"

namespace qspec {
namespace pass_impl {

using namespace gemv_impl;

constexpr int kMaxLayers = 16;
constexpr int kArenaBytes = 200 * 1024;  // most shared memory the staged activations may take
constexpr long long kBarrierWaitLimit = 4000000000LL;  // clock cycles (about 2 s)

enum : int { kFlagBarrier = 1 };

struct Layer {
  const uint16_t* x;
  const uint8_t* Wp;
  const __half* S;
  uint16_t* y;
  int N, K;
  int vt0;       // first tile of the layer in its segment's tile list
  int act_off;   // 16-byte offset of the layer's staged activations in the arena
  int act_len;   // 16-byte chunks of the staged activations (token slots x K / 8)
};

struct Segment {
  int l0, nl;    // its layers
  int K;         // common to its layers
  int KS;        // warps per tile (K split among them)
  int gs;        // groups per warp slice (K / 128 / KS)
  int tiles;     // 16-row tiles of all its layers
  int rounds;    // ceil(tiles / (CTAs x tile slots per CTA))
  int rot;       // rotation of the CTA order
  int flags;     // kFlagBarrier: every CTA finishes the earlier segments first
};

struct Params {
  Layer L[kMaxLayers];
  Segment Sg[kMaxLayers];
  int n_seg;
  int M;
  int arena_chunks;   // 16-byte chunks of staged activations this pass uses (the rest of the SM's
                      // unified L1 / shared memory stays L1, which holds the loads in flight)
  int corr_floats;    // offsets of the largest segment: layers x groups x token slots
  unsigned int* bar;  // grid barrier: [0] arrivals, [1] generation (zero-filled once)
  unsigned int* err;  // linear error word
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <int QB, int MT, int D>
__global__ void __launch_bounds__(kThreads, 1) pass_kernel(const __grid_constant__ Params p) {
  constexpr bool QUANT = QB == 4 || QB == 8;
  constexpr bool A4 = QUANT;
  constexpr float kQmax = QB == 8 ? 127.0f : 7.0f;
  constexpr int NB = (MT + 7) / 8;
  extern __shared__ __align__(16) uint8_t sm[];
  uint4* arena = reinterpret_cast<uint4*>(sm);
  float4* red = reinterpret_cast<float4*>(sm + static_cast<size_t>(p.arena_chunks) * 16);  // [2][kWarps][NB][32]
  float* corr = reinterpret_cast<float*>(red + 2 * kWarps * NB * 32);  // [layer of the segment][G][MT]
  __shared__ unsigned int red_max[QUANT ? kMaxLayers * kWarps * MT : 1];
  __shared__ float s_a[QUANT ? kMaxLayers : 1][MT];
  __shared__ int quit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int P = gridDim.x;
  const int ns = p.n_seg, M = p.M;
  if (threadIdx.x == 0) quit = 0;

  // ------------------------------------------------------------ this CTA's / warp's place in a segment
  auto per_cta = [](const Segment& S) { return kWarps / S.KS; };
  auto slot_of = [&](const Segment& S) { return ((blockIdx.x + S.rot) % P) * per_cta(S) + warp / S.KS; };
  auto idle = [&](const Segment& S) { return ((blockIdx.x + S.rot) % P) * per_cta(S) >= S.tiles; };
  // segment tile v -> its layer (index into p.L) and the layer's own tile
  auto locate = [&](const Segment& S, int v, int& l, int& tile) {
    l = S.l0;
    while (l + 1 < S.l0 + S.nl && v >= p.L[l + 1].vt0) ++l;
    tile = v - p.L[l].vt0;
  };

  // ------------------------------------------------------------ weight stream (fetch cursor)
  // The cursor's segment constants live in registers; the layer is looked up once per tile.
  int f_s = 0, f_r = 0, f_i = 0, f_gs = 0x7FFFFFFF, f_rounds = 0, f_stride = 0, f_slot = 0;
  const uint8_t* f_wlo = nullptr;
  const uint8_t* f_whi = nullptr;
  const __half* f_slo = nullptr;
  const __half* f_shi = nullptr;
  bool f_vlo = false, f_vhi = false;
  auto point = [&]() {
    const Segment& S = p.Sg[f_s];
    const int v = f_r * f_stride + f_slot;
    int l = S.l0, tile = 1 << 30;
    if (v < S.tiles) locate(S, v, l, tile);
    const Layer& L = p.L[l];
    const int n_lo = tile * 16 + g, n_hi = n_lo + 8;
    const int G = S.K / kGroup, g_beg = (warp % S.KS) * S.gs;
    f_vlo = v < S.tiles && n_lo < L.N;
    f_vhi = v < S.tiles && n_hi < L.N;
    const size_t rb = static_cast<size_t>(S.K) / 2;
    f_wlo = L.Wp + static_cast<size_t>(f_vlo ? n_lo : 0) * rb + g_beg * 64 + t * 16;
    f_whi = L.Wp + static_cast<size_t>(f_vhi ? n_hi : 0) * rb + g_beg * 64 + t * 16;
    f_slo = L.S + static_cast<size_t>(f_vlo ? n_lo : 0) * G + g_beg;
    f_shi = L.S + static_cast<size_t>(f_vhi ? n_hi : 0) * G + g_beg;
  };
  auto enter = [&](int s) {  // the cursor moves to the first item of segment s or a later busy one
    while (s < ns && idle(p.Sg[s])) ++s;
    f_s = s;
    f_r = 0;
    f_i = 0;
    if (s < ns) {
      const Segment& S = p.Sg[s];
      f_gs = S.gs;
      f_rounds = S.rounds;
      f_stride = P * per_cta(S);
      f_slot = slot_of(S);
      point();
    } else {  // past the end: no more loads, and the cursor never advances again
      f_vlo = f_vhi = false;
      f_gs = 0x7FFFFFFF;
    }
  };
  uint4 wl[D], wh[D];
  float sl[D], sh[D];
  // next item into register slot k; slices hold a multiple of D groups, so the cursor can only
  // leave its tile after slot D - 1
  auto fetch = [&](int k) {
    wl[k] = f_vlo ? ld_weights(f_wlo + (f_i + k) * 64) : make_uint4(0, 0, 0, 0);
    wh[k] = f_vhi ? ld_weights(f_whi + (f_i + k) * 64) : make_uint4(0, 0, 0, 0);
    sl[k] = f_vlo ? __half2float(f_slo[f_i + k]) : 0.0f;
    sh[k] = f_vhi ? __half2float(f_shi[f_i + k]) : 0.0f;
    if (k == D - 1) {
      f_i += D;
      if (f_i == f_gs) {
        f_i = 0;
        if (++f_r == f_rounds) enter(f_s + 1);
        else point();
      }
    }
  };
  enter(0);
#pragma unroll
  for (int k = 0; k < D; ++k) fetch(k);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ------------------------------------------------------------ activation staging
  // chunk ((gi * 4 + j) * MT + m) * 4 + t of a layer holds x[m, 128 gi + 32 t + 8 j .. + 7]
  auto stage_async = [&](const Segment& S) {
    const int per_token = (S.K / kGroup) * 16, total = M * per_token;
    for (int l = S.l0; l < S.l0 + S.nl; ++l) {
      const Layer& L = p.L[l];
      const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(arena + L.act_off));
      for (int c = threadIdx.x; c < total; c += kThreads) {
        const int m = c / per_token, v = c - m * per_token;
        const int t_ = v & 3, j_ = (v >> 2) & 3, gi = v >> 4;
        const uint16_t* src = L.x + static_cast<size_t>(m) * S.K + gi * 128 + t_ * 32 + j_ * 8;
        cp_async16(base + static_cast<uint32_t>((((v >> 2) * MT + m) * 4 + (v & 3)) * 16), src);
      }
    }
    cp_async_commit();
  };
  auto seg_span = [&](const Segment& S, int& lo, int& hi) {  // arena chunks of a segment's layers
    lo = p.L[S.l0].act_off;
    hi = p.L[S.l0 + S.nl - 1].act_off + p.L[S.l0 + S.nl - 1].act_len;
  };

  // After the copies landed: W4A4 / W4A8 quantise every layer of the segment in place (per-token amax
  // with one reduction for all of them) and record the offsets the integer codes will carry (see
  // off_pair_f16_*) per (layer, group, token).  The 16 chunks of a token's group sit on 16
  // consecutive lanes, so a warp sums them with four shuffles; the loops are uniform over the CTA.
  auto finish_staging = [&](const Segment& S) {
    const int G = S.K / kGroup, per_token = G * 16, total = M * per_token;
    auto put_corr = [&](int li, int c, const uint4& st) {
      float o = 0.0f;
      if (c < total) o = chunk_offset_f16(st);
      o = sum16(o);
      if (c < total && (lane & 15) == 0) {
        const int m = c / per_token, v = c - m * per_token;
        corr[(li * G + (v >> 4)) * MT + m] = o;
      }
    };
    if constexpr (!QUANT) return;  // W4A16 converts its codes exactly: no offsets
    for (int li = 0; li < S.nl; ++li) {
      const uint4* xs = arena + p.L[S.l0 + li].act_off;
      unsigned int mx[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) mx[m] = 0;
      for (int c = threadIdx.x; c < total; c += kThreads) {
        const int m = c / per_token, v = c - m * per_token;
        const uint4 val = xs[((v >> 2) * MT + m) * 4 + (v & 3)];
        const unsigned int am =
            max(max(max(val.x & 0x7FFFu, (val.x >> 16) & 0x7FFFu), max(val.y & 0x7FFFu, (val.y >> 16) & 0x7FFFu)),
                max(max(val.z & 0x7FFFu, (val.z >> 16) & 0x7FFFu), max(val.w & 0x7FFFu, (val.w >> 16) & 0x7FFFu)));
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
          if (mm == m) mx[mm] = max(mx[mm], am);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx[m] = max(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], off));
        if (lane == 0) red_max[(li * kWarps + warp) * MT + m] = mx[m];
      }
    }
    __syncthreads();
    for (int li = 0; li < S.nl; ++li) {
      uint4* xs = arena + p.L[S.l0 + li].act_off;
      float sa_r[MT], rs_r[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        unsigned int m_all = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m_all = max(m_all, red_max[(li * kWarps + w) * MT + m]);
        sa_r[m] = __fdiv_rn(__uint_as_float(m_all << 16), kQmax);
        rs_r[m] = __frcp_rn(sa_r[m]);
        if (threadIdx.x == m && m < M) s_a[li][m] = sa_r[m];
      }
      for (int c0 = 0; c0 < total; c0 += kThreads) {
        const int c = c0 + threadIdx.x;
        uint4 st = make_uint4(0, 0, 0, 0);
        if (c < total) {
          const int m = c / per_token, v = c - m * per_token;
          const int sl_ = ((v >> 2) * MT + m) * 4 + (v & 3);
          float sa = sa_r[0], rsa = rs_r[0];
#pragma unroll
          for (int mm = 1; mm < MT; ++mm)
            if (m == mm) {
              sa = sa_r[mm];
              rsa = rs_r[mm];
            }
          const bool fast = QB == 4 && sa >= 0x1p-100f;  // see div_rn_markstein
          const uint4 val = xs[sl_];
          const uint32_t w[4] = {val.x, val.y, val.z, val.w};
          float c8[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float c0f = 0.0f, c1f = 0.0f;
            if (sa != 0.0f) {
              const float x0 = bf16_lo(w[i]), x1 = bf16_hi(w[i]);
              const float q0 = fast ? div_rn_markstein(x0, sa, rsa) : __fdiv_rn(x0, sa);
              const float q1 = fast ? div_rn_markstein(x1, sa, rsa) : __fdiv_rn(x1, sa);
              c0f = fminf(fmaxf(rintf(q0), -kQmax - 1.0f), kQmax);
              c1f = fminf(fmaxf(rintf(q1), -kQmax - 1.0f), kQmax);
            }
            c8[2 * i] = c0f;
            c8[2 * i + 1] = c1f;
          }
          st = codes_to_f16_chunk(c8);  // exact: small integers and their sixteenths
          xs[sl_] = st;
        }
        put_corr(li, c, st);
      }
    }
  };

  // grid-wide barrier before a segment that reads what earlier ones wrote; false if this CTA gave up
  auto grid_barrier = [&]() -> bool {
    __syncthreads();  // every warp of this CTA is done with the earlier segments
    if (threadIdx.x == 0) {
      const unsigned int gen = ld_acquire(p.bar + 1);
      __threadfence();  // this CTA's outputs before its arrival
      const unsigned int prev = atomicAdd(p.bar, 1u);
      if (prev == static_cast<unsigned int>(P - 1)) {
        atomicExch(p.bar, 0u);
        __threadfence();
        atomicAdd(p.bar + 1, 1u);  // release the others
      } else {
        const long long t0 = clock64();
        while (ld_acquire(p.bar + 1) == gen) {
          if (clock64() - t0 > kBarrierWaitLimit) {
            atomicOr(p.err, kErrTimeout);
            quit = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      __threadfence();
    }
    __syncthreads();
    return !quit;
  };

  // ------------------------------------------------------------ the segments
  unsigned int staged = 0;  // segments whose activations are already on their way (bit s)
  int rr = 0;               // reduction rounds so far (red buffer parity)
  for (int s = 0; s < ns; ++s) {
    const Segment& S = p.Sg[s];
    if ((S.flags & kFlagBarrier) && !grid_barrier()) return;
    if (idle(S)) continue;
    if (!(staged & (1u << s))) {
      __syncthreads();  // the arena may still be read for this CTA's previous segment
      stage_async(S);
    }
    cp_async_wait_all();
    __syncthreads();
    finish_staging(S);
    __syncthreads();
    // the next busy segment's activations travel while this one streams, if nothing stands between
    for (int s2 = s + 1; s2 < ns; ++s2) {
      const Segment& S2 = p.Sg[s2];
      if (S2.flags & kFlagBarrier) break;
      if (idle(S2)) continue;
      int a0, a1, b0, b1;
      seg_span(S, a0, a1);
      seg_span(S2, b0, b1);
      if (a1 <= b0 || b1 <= a0) {
        stage_async(S2);
        staged |= 1u << s2;
      }
      break;
    }

    const int KS = S.KS, gs = S.gs;
    const int wtile = warp / KS, ks = warp - wtile * KS, g_beg = ks * gs;
    const int stride = P * per_cta(S), slot = slot_of(S);
    for (int r = 0; r < S.rounds; ++r, ++rr) {
      const int v = r * stride + slot;
      int l = S.l0, tile = 1 << 30;
      if (v < S.tiles) locate(S, v, l, tile);
      const uint4* xs = arena + p.L[l].act_off;
      const float* cl = corr + (l - S.l0) * (S.K / kGroup) * MT;
      float acc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
      for (int i0 = 0; i0 < gs; i0 += D) {
#pragma unroll
        for (int k = 0; k < D; ++k) {
          const uint4* xg = xs + static_cast<size_t>(g_beg + i0 + k) * 16 * MT;
          float d[NB][4];
          item_mma<A4, NB, MT>(d, wl[k], wh[k], xg, cl + (g_beg + i0 + k) * MT, g, t);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] = fmaf(sl[k], d[nb][0], acc[nb][0]);
            acc[nb][1] = fmaf(sl[k], d[nb][1], acc[nb][1]);
            acc[nb][2] = fmaf(sh[k], d[nb][2], acc[nb][2]);
            acc[nb][3] = fmaf(sh[k], d[nb][3], acc[nb][3]);
          }
          fetch(k);
        }
      }
      if (KS > 1) {  // K slices summed in slice order by the slice-0 warp of the tile slot
        float4* rb = red + (rr & 1) * kWarps * NB * 32;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          rb[(warp * NB + nb) * 32 + lane] = make_float4(acc[nb][0], acc[nb][1], acc[nb][2], acc[nb][3]);
        asm volatile("bar.sync %0, %1;" ::"r"(1 + wtile), "r"(KS * 32) : "memory");
        if (ks == 0) {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            float4 s4 = rb[(warp * NB + nb) * 32 + lane];
            for (int j = 1; j < KS; ++j) {
              const float4 o = rb[((warp + j) * NB + nb) * 32 + lane];
              s4.x += o.x;
              s4.y += o.y;
              s4.z += o.z;
              s4.w += o.w;
            }
            acc[nb][0] = s4.x;
            acc[nb][1] = s4.y;
            acc[nb][2] = s4.z;
            acc[nb][3] = s4.w;
          }
        }
      }
      if (ks == 0 && v < S.tiles) {
        const Layer& L = p.L[l];
        const int n_lo = tile * 16 + g, n_hi = n_lo + 8;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int m0 = nb * 8 + 2 * t, m1 = m0 + 1;
          if constexpr (A4) {
            const float sa0 = m0 < M ? s_a[l - S.l0][m0] : 0.0f, sa1 = m1 < M ? s_a[l - S.l0][m1] : 0.0f;
            acc[nb][0] *= sa0;
            acc[nb][1] *= sa1;
            acc[nb][2] *= sa0;
            acc[nb][3] *= sa1;
          }
          if (n_lo < L.N && m0 < M) L.y[static_cast<size_t>(m0) * L.N + n_lo] = f32_to_bf16_bits(acc[nb][0]);
          if (n_lo < L.N && m1 < M) L.y[static_cast<size_t>(m1) * L.N + n_lo] = f32_to_bf16_bits(acc[nb][1]);
          if (n_hi < L.N && m0 < M) L.y[static_cast<size_t>(m0) * L.N + n_hi] = f32_to_bf16_bits(acc[nb][2]);
          if (n_hi < L.N && m1 < M) L.y[static_cast<size_t>(m1) * L.N + n_hi] = f32_to_bf16_bits(acc[nb][3]);
        }
      }
    }
  }
  cp_async_wait_all();  // nothing may still be copying into shared memory when the CTA exits
}

// dynamic shared memory: the staged activations, the K-slice reduction buffer (NB = 1), and the
// per-(layer, group, token) offsets of the largest segment (one float per 256 bytes of its staged
// activations, so at most kArenaBytes / 256 floats)
inline size_t pass_smem_bytes(int arena_chunks, int corr_floats) {
  return static_cast<size_t>(arena_chunks) * 16 + 2 * kWarps * 32 * 16 + static_cast<size_t>(corr_floats) * 4;
}

template <int QB, int MT, int D>
qspec_status launch_pass(const Params& prm, int grid, cudaStream_t stream) {
  auto kern = pass_kernel<QB, MT, D>;
  const size_t smem = pass_smem_bytes(prm.arena_chunks, prm.corr_floats);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(pass_smem_bytes(kArenaBytes / 16, kArenaBytes / 256))) != cudaSuccess)
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
  return cudaLaunchKernelEx(&cfg, kern, prm) == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

// The launcher of one activation mode (0: W4A16, 4: W4A4, 8: W4A8), one translation unit each.
template <int QB>
qspec_status launch_pass_mode(int MT, int D, const Params& prm, int grid, cudaStream_t stream);

#define QSPEC_PASS_MODE_UNIT(QB_)                                                                        \
  template <>                                                                                            \
  qspec_status launch_pass_mode<QB_>(int MT, int D, const Params& prm, int grid, cudaStream_t stream) {  \
    if (D == 4) {                                                                                        \
      switch (MT) {                                                                                      \
        case 1: return launch_pass<QB_, 1, 4>(prm, grid, stream);                                        \
        case 2: return launch_pass<QB_, 2, 4>(prm, grid, stream);                                        \
        default: return launch_pass<QB_, 4, 4>(prm, grid, stream);                                       \
      }                                                                                                  \
    }                                                                                                    \
    switch (MT) {                                                                                        \
      case 1: return launch_pass<QB_, 1, 1>(prm, grid, stream);                                          \
      case 2: return launch_pass<QB_, 2, 1>(prm, grid, stream);                                          \
      default: return launch_pass<QB_, 4, 1>(prm, grid, stream);                                         \
    }                                                                                                    \
  }

template <>
qspec_status launch_pass_mode<0>(int, int, const Params&, int, cudaStream_t);
template <>
qspec_status launch_pass_mode<4>(int, int, const Params&, int, cudaStream_t);
template <>
qspec_status launch_pass_mode<8>(int, int, const Params&, int, cudaStream_t);

}  // namespace pass_impl
}  // namespace qspec
