// Both linears at decode sizes (M = 1..16 tokens): register-resident weight fragments fed straight
// into warp-level tensor-core MMAs.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": W4A16 keeps the 16-bit activations and converts the 4-bit weights while
// multiplying; W4A4 also quantises the activations to 4 bits (per token here: s_a = amax / 7 in
// fp32, codes = clamp(rint(x / s_a), -8, 7)).  Section "QSpec の W4A4 モードと W4A16 モード": both
// modes read the same packed weights.  At decode sizes the product is a GEMV bound by the weight
// stream (0.5 B per weight); the tcgen05 path would have to expand every weight to bf16 in TMEM
// (4x the streamed bytes, written and read back on chip), which measured slower than the HBM stream
// itself, so here the expanded weights never leave registers:
//
//  * a warp owns 16 weight rows x a K slice (x up to 16 tokens in two MMA column blocks of 8).  Lane (g, t) = (lane / 4, lane % 4) loads 16 bytes of
//    each of its two rows g and g + 8 per 128-channel group: packed words 4t..4t+3, i.e. channels
//    32t..32t+31 of the group;
//  * one shift + LOP3 + bf16 subtract turns a nibble pair of a word into an exact bf16x2 code pair
//    (the packed word keeps channels 2i and 2i+1 in nibbles i and i + 4), which is directly an A
//    fragment register of mma.m16n8k16: the MMA's 16 k-slots of lane t are mapped onto the
//    channels lane t holds (a fixed permutation of K inside the group), and the activations are
//    staged in shared memory in exactly that order, so one 16-byte shared load gives the B
//    fragments of two MMAs.  W4A4 and W4A8 multiply in fp16 instead: the weight nibbles convert
//    without shifts to codes or 16 x codes (code_pair_f16_lo / _hi) and the activation codes are
//    staged in the same place with those meeting a 16 x weight code divided by 16 (all exact):
//    every product and every 128-channel sum is then a small integer, exact in the fp32 MMA
//    accumulator, so the group sums are the exact integer sums of code * code;
//  * per group the fp32 MMA result is scaled by s[n, g] and accumulated in fp32; K slices of a
//    tile are summed through shared memory in a fixed order; W4A4 multiplies by s_a at the end;
//    y is rounded to bf16 once.
//
// Tokens are the MMA's N = 8 side (rows >= M are zero), weight rows its M = 16 side.
#include <cuda_bf16.h>

#include <algorithm>

#pragma once

#include "common.cuh"
#include "linear_internal.h"

namespace qspec {
namespace gemv_impl {

constexpr int kThreads = 512;  // 16 warps, one CTA per SM
constexpr int kWarps = kThreads / 32;
constexpr int kStageU = 4;  // 16-byte activation chunks a thread loads per staging batch
constexpr int kMaxTokens = 32;  // token slots: 1, 2, 4, 8, 16 or 32 (two or four MMA column blocks above 8)

// 16 bytes of packed weights, read once: not kept in L1
__device__ __forceinline__ uint4 ld_weights(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// W4A16 (bf16): pair i of a packed word (channels 2i, 2i + 1 of its 8) shifted to bits 0..3 / 16..19
// with its top bit flipped into bf16 128.0 is 128 + (nibble ^ 8) = 136 + code; one bf16x2 subtract
// gives the exact code pair, which is directly an MMA operand register.  (Leaving the 136 in and
// removing 136 x the group's activation sum afterwards measured slower here: the saving is one
// subtract per pair, the price a sum per staged chunk on the critical path of every launch.)
__device__ __forceinline__ uint32_t code_pair_bf16(uint32_t w, int i) {
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43084308u));
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                   __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The integer-code modes (W4A4, W4A8, staged codes) multiply in fp16, whose 10-bit mantissa takes
// a nibble at bits 0..3 or 4..7 of each half without shifting it: XOR into 1032.0 (0x6408) gives
// 1024 + (nibble ^ 8) = 1032 + code, XOR into 1152.0 (0x6480) at bits 4..7 gives 1152 + 16 code.
// So pairs 0 and 2 of a word (the latter after one 8-bit shift) convert to 1032 + (code, code') and
// pairs 1 and 3 to 1152 + 16 (code, code'), all exact; the activation codes those pairs meet are
// staged divided by 16 (exact in fp16).  The offsets stay in ("offset form": no subtraction per
// pair): their contribution, 1032 x (activation codes of channels 0, 1, 4, 5 of every 8) + 72 x
// (channels 2, 3, 6, 7), is computed once per (token, group) while the codes are staged and removed
// from the MMA result.  Every product and partial sum is an integer below 2^24 (W4A8 included),
// exact in the fp32 accumulator, and so is the offset removed: the group sums stay exact.
__device__ __forceinline__ uint32_t off_pair_f16_lo(uint32_t w) {
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w), "r"(0x000F000Fu), "r"(0x64086408u));
  return v;
}
__device__ __forceinline__ uint32_t off_pair_f16_hi(uint32_t w) {
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w), "r"(0x00F000F0u), "r"(0x64806480u));
  return v;
}

// What the offsets add for one staged code chunk (8 channels of one token): 1032 x (elements 0, 1,
// 4, 5) + 1152 x (elements 2, 3, 6, 7, which hold code / 16); exact.
__device__ __forceinline__ float chunk_offset_f16(uint4 c) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&c.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&c.y));
  const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&c.z));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&c.w));
  return 1032.0f * ((a.x + a.y) + (e.x + e.y)) + 1152.0f * ((b.x + b.y) + (f.x + f.y));
}
// Sum over the 16 lanes of a half-warp (the 16 chunks of one token's 128-channel group).
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// Eight activation codes (as floats) -> the staged fp16 chunk: elements 2, 3, 6, 7 (the channels of
// pairs 1 and 3) divided by 16.
__device__ __forceinline__ uint4 codes_to_f16_chunk(const float (&c)[8]) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float f = (i & 1) ? 0.0625f : 1.0f;
    const __half2 h = __floats2half2_rn(c[2 * i] * f, c[2 * i + 1] * f);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// d += A (16 x 16, row fragments a0..a3) * B (16 x 8, column fragments b0, b1), fp32 accumulate;
// F16: fp16 operands (the integer-code modes), else bf16
template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// One item of a warp's stream: rows (g, g + 8) of a 16-row tile x one 128-channel group x the NB
// column blocks of 8 tokens, in 8 MMAs (the group's four 32-channel quarters j, two k16 steps each).
// Integer-code modes (F16) keep the weight codes offset and corr (the group's [MT] offsets) removes
// them; W4A16 converts exactly and has no offsets.
template <bool F16, int NB, int MT>
__device__ __forceinline__ void item_mma(float (&d)[NB][4], const uint4& wl, const uint4& wh, const uint4* xg,
                                         const float* corr, int g, int t) {
  const uint32_t lo[4] = {wl.x, wl.y, wl.z, wl.w};
  const uint32_t hi[4] = {wh.x, wh.y, wh.z, wh.w};
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) d[nb][0] = d[nb][1] = d[nb][2] = d[nb][3] = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 xb[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      xb[nb] = make_uint4(0, 0, 0, 0);
      if (MT % 8 == 0 || g < MT) xb[nb] = xg[(j * MT + nb * 8 + g) * 4 + t];
    }
    if constexpr (F16) {
      const uint32_t l8 = lo[j] >> 8, h8 = hi[j] >> 8;
      const uint32_t a0 = off_pair_f16_lo(lo[j]), a1 = off_pair_f16_lo(hi[j]), a2 = off_pair_f16_hi(lo[j]),
                     a3 = off_pair_f16_hi(hi[j]);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_16816<true>(d[nb], a0, a1, a2, a3, xb[nb].x, xb[nb].y);
      const uint32_t c0 = off_pair_f16_lo(l8), c1 = off_pair_f16_lo(h8), c2 = off_pair_f16_hi(l8),
                     c3 = off_pair_f16_hi(h8);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_16816<true>(d[nb], c0, c1, c2, c3, xb[nb].z, xb[nb].w);
    } else {
      const uint32_t a0 = code_pair_bf16(lo[j], 0), a1 = code_pair_bf16(hi[j], 0), a2 = code_pair_bf16(lo[j], 1),
                     a3 = code_pair_bf16(hi[j], 1);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_16816<false>(d[nb], a0, a1, a2, a3, xb[nb].x, xb[nb].y);
      const uint32_t c0 = code_pair_bf16(lo[j], 2), c1 = code_pair_bf16(hi[j], 2), c2 = code_pair_bf16(lo[j], 3),
                     c3 = code_pair_bf16(hi[j], 3);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_16816<false>(d[nb], c0, c1, c2, c3, xb[nb].z, xb[nb].w);
    }
  }
  if constexpr (!F16) return;
  // remove the offsets: tokens (8 nb + 2t, + 1), the same for both rows
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int m0 = nb * 8 + 2 * t;
    float c0 = 0.0f, c1 = 0.0f;
    if constexpr (MT % 2 == 0) {
      if (m0 < MT) {
        const float2 cc = *reinterpret_cast<const float2*>(corr + m0);
        c0 = cc.x;
        c1 = cc.y;
      }
    } else {
      if (m0 < MT) c0 = corr[m0];
    }
    d[nb][0] -= c0;
    d[nb][1] -= c1;
    d[nb][2] -= c0;
    d[nb][3] -= c1;
  }
}

// QB: activation bits of the quantised modes -- 4 (W4A4) or 8 (W4A8: the same per-token quantiser
// with divisor 127 and codes in [-128, 127], a configuration the speculative-decoding-with-
// quantisation summary on aibr.jp names in its section "中核となる技術的要素"), 0 for W4A16.  The
// quantised modes quantise the tokens (optional int8 codes / fp32 scales out); ACC: also the int32 group
// sums (a separate instantiation keeps their stores out of the hot loop when not asked for).
// MT = token slots staged in shared memory (1, 2, 4, 8 or 16; tokens >= M contribute zeros); the
// tokens form NB = ceil(MT / 8) MMA column blocks of 8 that share every weight fragment.  D = weight
// groups in flight per warp (a divisor of the groups per K slice, so that the slots line up with
// tile boundaries).
//
// A warp's work is one stream of (row tile, group) items: the tiles r * stride + blockIdx.x * per_cta
// + wtile for r = 0, 1, ..., and within each its K slice of groups.  Weights are fetched D items
// ahead across tile boundaries, so the stream never drains; the first fetches are issued before
// the kernel waits for its predecessor (no library kernel that may run ahead of this one writes
// packed weights or scales).
// Up to kMaxParts weight matrices that read the same activations (one linear, or e.g. the q, k and v
// projections of a decoder layer), streamed as one run of 16-row tiles: part i owns the tiles
// [tile_end[i - 1], tile_end[i]) and its rows, scales and outputs are its own.
constexpr int kMaxParts = 4;
struct Parts {
  int n;
  int tile_end[kMaxParts];
  int N[kMaxParts];
  const uint8_t* Wp[kMaxParts];
  const __half* S[kMaxParts];
  uint16_t* y[kMaxParts];
};

// Token slots for which the kernel serves several parts (above, one part: the lookup's registers
// would push the 16- and 32-slot kernels past their 128).
constexpr int kPartsMaxMT = 4;

// The part that tile belongs to (the last part for tiles past the end).  MP: the launch may have
// several parts (single-part launches skip the lookup: measured, the W4A16 kernels of up to 4 token
// slots run 5-9% faster without it; the quantised modes keep it, which measured no slower).
template <int MT, bool MP>
__device__ __forceinline__ int part_of(const Parts& p, int tile) {
  if constexpr (MT > kPartsMaxMT || !MP) {
    return 0;
  } else {
    int s = 0;
#pragma unroll
    for (int i = 0; i < kMaxParts - 1; ++i) s += (i + 1 < p.n && tile >= p.tile_end[i]) ? 1 : 0;
    return s;
  }
}

template <int QB, bool ACC, int MT, int D, bool CHUNK, bool MP>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const __grid_constant__ Parts parts, int M, int K, int KS,
                int KC_arg, int8_t* __restrict__ xq_out,
                float* __restrict__ xs_out, int32_t* __restrict__ acc_out, const float* __restrict__ s_a_in,
                float* __restrict__ part, unsigned int* __restrict__ tick, const WsGuard guard) {
  constexpr bool A4 = QB != 0;                       // activations quantised (W4A4 or W4A8)
  constexpr bool QUANT = QB == 4 || QB == 8;         // ... here (QB == 1: x holds the staged fp16
                                                     // code chunks, s_a_in the scales)
  constexpr float kQmax = QB == 8 ? 127.0f : 7.0f;   // codes in [-kQmax - 1, kQmax]
  extern __shared__ __align__(16) uint8_t sm[];
  const int G = K / kGroup;
  // K chunks: CTA c works on groups [gb, gb + Gc) of chunk kc = c % KC (KC = 1 unless the staged
  // activations of all K would not fit shared memory); the KC partial tiles are summed by the
  // chunk that finishes last
  const int KC = CHUNK ? KC_arg : 1;  // (CHUNK: a separate instantiation, so KC == 1 costs nothing)
  const int kc = blockIdx.x % KC, cb = blockIdx.x / KC;
  const int Gc = G / KC, gb = kc * Gc;
  // activations: chunk ((gi * 4 + j) * MT + m) * 4 + t holds x[m, 128 (gb + gi) + 32 t + 8 j .. + 7]
  uint4* xs = reinterpret_cast<uint4*>(sm);
  constexpr int NB = (MT + 7) / 8;
  float4* red = reinterpret_cast<float4*>(xs + static_cast<size_t>(Gc) * 16 * MT);  // [2][kWarps][NB][32]
  __shared__ unsigned int red_max[QUANT ? kWarps * MT : 1];
  __shared__ float s_a[MT];  // per-token scale, for the epilogue
  __shared__ int ws_ok;      // K chunks: the workspace holds this shape's layout (or none yet)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  const int tiles = parts.tile_end[parts.n - 1];
  const int per_cta = kWarps / KS;  // row tiles a CTA works on at once
  const int wtile = warp / KS, ks = warp - wtile * KS;
  const int gs = Gc / KS, g_beg = ks * gs;  // this warp's groups within the chunk
  const int stride = (gridDim.x / KC) * per_cta;
  const int tile0 = cb * per_cta + wtile;
  const int rounds = (tiles + stride - 1) / stride;  // the same for the KS warps of a tile slot
  const size_t row_bytes = static_cast<size_t>(K) / 2;

  // fetch cursor: the tile, its row pointers (at the slice's first group) and the group index
  const uint8_t* f_wlo = parts.Wp[0];
  const uint8_t* f_whi = parts.Wp[0];
  const __half* f_slo = parts.S[0];
  const __half* f_shi = parts.S[0];
  bool f_vlo = false, f_vhi = false;
  int f_tile = tile0, f_i = 0;
  auto point = [&]() {
    const int ps = part_of<MT, MP>(parts, f_tile);
    const int n_lo = (f_tile - (ps ? parts.tile_end[ps - 1] : 0)) * 16 + g, n_hi = n_lo + 8;
    const int Np = parts.N[ps];
    const uint8_t* Wp = parts.Wp[ps];
    const __half* S = parts.S[ps];
    f_vlo = f_tile < tiles && n_lo < Np;
    f_vhi = f_tile < tiles && n_hi < Np;
    f_wlo = Wp + static_cast<size_t>(f_vlo ? n_lo : 0) * row_bytes + (gb + g_beg) * 64 + t * 16;
    f_whi = Wp + static_cast<size_t>(f_vhi ? n_hi : 0) * row_bytes + (gb + g_beg) * 64 + t * 16;
    f_slo = S + static_cast<size_t>(f_vlo ? n_lo : 0) * G + gb + g_beg;
    f_shi = S + static_cast<size_t>(f_vhi ? n_hi : 0) * G + gb + g_beg;
  };
  uint4 wl[D], wh[D];
  float sl[D], sh[D];
  // next item of the stream into register slot k; the D slots are refilled in order and the slice
  // length is a multiple of D, so the cursor can only leave its tile after slot D - 1
  auto fetch = [&](int k) {
    wl[k] = f_vlo ? ld_weights(f_wlo + (f_i + k) * 64) : make_uint4(0, 0, 0, 0);
    wh[k] = f_vhi ? ld_weights(f_whi + (f_i + k) * 64) : make_uint4(0, 0, 0, 0);
    sl[k] = f_vlo ? __half2float(f_slo[f_i + k]) : 0.0f;
    sh[k] = f_vhi ? __half2float(f_shi[f_i + k]) : 0.0f;
    if (k == D - 1) {
      f_i += D;
      if (f_i == gs) {
        f_i = 0;
        f_tile += stride;
        point();
      }
    }
  };
  point();
#pragma unroll
  for (int k = 0; k < D; ++k) fetch(k);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the chunk partials and tickets live in the linear workspace; its claim is read after staging
  if (CHUNK && threadIdx.x == 0) ws_ok = ws_claim(guard) ? 1 : 0;

  // Staging: chunk (gi, j, t) of token m <- x[m, 128 gi + 32 t + 8 j .. + 7].  Slots of tokens
  // M..MT-1 are never written: they only feed MMA columns that are not stored.  A thread loads its
  // kU chunks before using any, so one L2 round trip covers them (all of x, for the usual sizes,
  // which W4A4 then keeps in registers between its two passes).
  const int per_token = Gc * 16;
  const int total = M * per_token;
  constexpr int kU = kStageU;
  auto locate = [&](int c, int& m, int& v) {
    m = c / per_token;
    v = c - m * per_token;  // (gi * 4 + j) * 4 + t
  };
  auto src_of = [&](int m, int v) {
    const int t_ = v & 3, j_ = (v >> 2) & 3, gi = v >> 4;
    return static_cast<size_t>(m) * K + (gb + gi) * 128 + t_ * 32 + j_ * 8;
  };
  auto load_batch = [&](int c0, uint4 (&u)[kU]) {
#pragma unroll
    for (int e = 0; e < kU; ++e) {
      const int c = c0 + e * kThreads;
      int m = 0, v = 0;
      if (c < total) locate(c, m, v);
      u[e] = c < total ? __ldg(reinterpret_cast<const uint4*>(x + src_of(m, v))) : make_uint4(0, 0, 0, 0);
    }
  };
  auto slot_of = [&](int m, int v) { return ((v >> 2) * MT + m) * 4 + (v & 3); };
  // W4A4 / W4A8: codes = clamp(rint(x / s_a), -qmax - 1, qmax) of one chunk, as exact bf16 (and the
  // int8 codes out)
  // per-token scale and its reciprocal, held by every thread (finish_scales)
  float sa_r[QUANT ? MT : 1], rs_r[QUANT ? MT : 1];
  auto quantise = [&](int m, int v, uint4 val) {
    float sa = sa_r[0], rsa = rs_r[0];
#pragma unroll
    for (int mm = 1; mm < (QUANT ? MT : 1); ++mm)
      if (m == mm) {
        sa = sa_r[mm];
        rsa = rs_r[mm];
      }
    // see div_rn_markstein (checked for the 4-bit divisor; W4A8 keeps the IEEE division)
    const bool fast = QB == 4 && sa >= 0x1p-100f;
    const uint32_t w[4] = {val.x, val.y, val.z, val.w};
    float c[8];
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
      c[2 * i] = c0f;
      c[2 * i + 1] = c1f;
    }
    if (xq_out && cb == 0) {
      uint32_t q8[2] = {0, 0};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        q8[e >> 2] |= (static_cast<uint32_t>(static_cast<int>(c[e])) & 0xFFu) << (8 * (e & 3));
      *reinterpret_cast<uint2*>(xq_out + src_of(m, v)) = make_uint2(q8[0], q8[1]);
    }
    return codes_to_f16_chunk(c);  // exact: small integers and their sixteenths
  };

  auto chunk_amax = [](uint4 val) {
    return max(max(max(val.x & 0x7FFFu, (val.x >> 16) & 0x7FFFu), max(val.y & 0x7FFFu, (val.y >> 16) & 0x7FFFu)),
               max(max(val.z & 0x7FFFu, (val.z >> 16) & 0x7FFFu), max(val.w & 0x7FFFu, (val.w >> 16) & 0x7FFFu)));
  };
  // per-token amax (bf16 bit patterns of |x| order like the values) -> s_a = amax / 7, 1 / s_a
  unsigned int mx[QUANT ? MT : 1];
  auto amax_add = [&](int m, uint4 val) {
    const unsigned int am = chunk_amax(val);
#pragma unroll
    for (int mm = 0; mm < MT; ++mm)
      if (mm == m) mx[mm] = max(mx[mm], am);
  };
  // every thread reduces the warps' maxima itself, so one barrier suffices
  auto finish_scales = [&]() {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mx[m] = max(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], off));
      if (lane == 0) red_max[warp * MT + m] = mx[m];
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      unsigned int m_all = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) m_all = max(m_all, red_max[w * MT + m]);
      sa_r[m] = __fdiv_rn(__uint_as_float(m_all << 16), kQmax);
      rs_r[m] = __frcp_rn(sa_r[m]);
      if (threadIdx.x == m && m < M) {  // for the epilogue (read after the staging barrier)
        s_a[m] = sa_r[m];
        if (xs_out && blockIdx.x == 0) xs_out[m] = sa_r[m];
      }
    }
  };
  if constexpr (QUANT) {
#pragma unroll
    for (int m = 0; m < MT; ++m) mx[m] = 0;
  }
  // a chunked CTA stages part of K but needs the amax over all of it: one extra read of x
  auto amax_full = [&]() {
    const int n16 = K / 8;
    for (int c = threadIdx.x; c < M * n16; c += kThreads) {
      const int m = c / n16;
      amax_add(m, __ldg(reinterpret_cast<const uint4*>(x) + c));
    }
  };
  if constexpr (QB == 1) {
    if (threadIdx.x < M) s_a[threadIdx.x] = s_a_in[threadIdx.x];
  }
  // offsets the integer codes carry (see off_pair_f16_*), per (group of this chunk, token): the 16 chunks of a
  // token's group sit on 16 consecutive lanes (the chunk order below), so every warp reduces them with
  // four shuffles and the group's first lane writes the sum; all lanes take part (uniform loops)
  float* corr = reinterpret_cast<float*>(red + 2 * kWarps * NB * 32);  // [Gc][MT]
  auto put_corr = [&](int c, const uint4& staged) {
    if constexpr (!A4) return;  // W4A16 converts its codes exactly: no offsets
    float o = 0.0f;
    if (c < total) o = chunk_offset_f16(staged);
    o = sum16(o);
    if (c < total && (lane & 15) == 0) {
      int m, v;
      locate(c, m, v);
      corr[(v >> 4) * MT + m] = o;
    }
  };
  uint4 u[kU];
  if (total <= kU * kThreads) {
    // one batch: x stays in registers between the passes
    load_batch(threadIdx.x, u);
    if constexpr (QUANT) {
      if (KC == 1) {
#pragma unroll
        for (int e = 0; e < kU; ++e) {
          const int c = threadIdx.x + e * kThreads;
          if (c < total) amax_add(c / per_token, u[e]);
        }
      } else {
        amax_full();
      }
      finish_scales();
    }
#pragma unroll
    for (int e = 0; e < kU; ++e) {
      // a warp whose chunks of this batch all lie past the tokens is done (the same for all its
      // lanes, so the offset sums' shuffles stay warp-uniform): one token of 4096 channels fills
      // only the first of a thread's kU chunk slots
      if (static_cast<int>(threadIdx.x & ~31u) + e * kThreads >= total) break;
      const int c = threadIdx.x + e * kThreads;
      uint4 st = make_uint4(0, 0, 0, 0);
      if (c < total) {
        int m, v;
        locate(c, m, v);
        st = QUANT ? quantise(m, v, u[e]) : u[e];
        xs[slot_of(m, v)] = st;
      }
      put_corr(c, st);
    }
  } else {
    // several batches: x goes to shared memory as it is, W4A4 then works there (no second trip
    // to L2)
    for (int b0 = 0; b0 < total; b0 += kU * kThreads) {
      load_batch(b0 + threadIdx.x, u);
#pragma unroll
      for (int e = 0; e < kU; ++e) {
        const int c = b0 + threadIdx.x + e * kThreads;
        if (c < total) {
          int m, v;
          locate(c, m, v);
          xs[slot_of(m, v)] = u[e];
          if constexpr (QUANT) {
            if (KC == 1) amax_add(m, u[e]);
          }
        }
        if constexpr (!QUANT) put_corr(c, u[e]);
      }
    }
    if constexpr (QUANT) {
      if (KC > 1) amax_full();
      finish_scales();
      for (int c0 = 0; c0 < total; c0 += kThreads) {
        const int c = c0 + threadIdx.x;
        uint4 st = make_uint4(0, 0, 0, 0);
        if (c < total) {
          int m, v;
          locate(c, m, v);
          const int sl_ = slot_of(m, v);
          st = quantise(m, v, xs[sl_]);
          xs[sl_] = st;
        }
        put_corr(c, st);
      }
    }
  }
  __syncthreads();
  if (CHUNK && !ws_ok) return;  // (uniform over the CTA) another shape's layout: touch nothing

  for (int r = 0; r < rounds; ++r) {
    const int tile = r * stride + tile0;
    // rows (tile * 16 + g, + 8) x tokens (8 nb + 2t, 8 nb + 2t + 1) of column block nb
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
    for (int i0 = 0; i0 < gs; i0 += D) {
#pragma unroll
      for (int k = 0; k < D; ++k) {
        const uint4* xg = xs + static_cast<size_t>(g_beg + i0 + k) * 16 * MT;
        float d[NB][4];
        item_mma<A4, NB, MT>(d, wl[k], wh[k], xg, corr + (g_beg + i0 + k) * MT, g, t);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          acc[nb][0] = fmaf(sl[k], d[nb][0], acc[nb][0]);
          acc[nb][1] = fmaf(sl[k], d[nb][1], acc[nb][1]);
          acc[nb][2] = fmaf(sh[k], d[nb][2], acc[nb][2]);
          acc[nb][3] = fmaf(sh[k], d[nb][3], acc[nb][3]);
        }
        if constexpr (A4 && ACC) {
          if (tile < tiles) {  // exact integer group sums (one part only)
            const int N = parts.N[0];
            const int n_lo = tile * 16 + g, n_hi = n_lo + 8, gi = gb + g_beg + i0 + k;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const int m0 = nb * 8 + 2 * t, m1 = m0 + 1;
              if (n_lo < N && m0 < M) acc_out[(static_cast<size_t>(m0) * N + n_lo) * G + gi] = static_cast<int32_t>(d[nb][0]);
              if (n_lo < N && m1 < M) acc_out[(static_cast<size_t>(m1) * N + n_lo) * G + gi] = static_cast<int32_t>(d[nb][1]);
              if (n_hi < N && m0 < M) acc_out[(static_cast<size_t>(m0) * N + n_hi) * G + gi] = static_cast<int32_t>(d[nb][2]);
              if (n_hi < N && m1 < M) acc_out[(static_cast<size_t>(m1) * N + n_hi) * G + gi] = static_cast<int32_t>(d[nb][3]);
            }
          }
        }
        fetch(k);
      }
    }
    if (KS > 1) {  // K slices summed in slice order by the slice-0 warp of the tile slot
      float4* rb = red + (r & 1) * kWarps * NB * 32;
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
    bool store = ks == 0 && tile < tiles;
    if (store && KC > 1) {
      // publish this chunk's partial tile; the chunk that arrives last sums all KC in chunk order
      float4* pp = reinterpret_cast<float4*>(part);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        pp[((static_cast<size_t>(kc) * tiles + tile) * NB + nb) * 32 + lane] =
            make_float4(acc[nb][0], acc[nb][1], acc[nb][2], acc[nb][3]);
      __threadfence();
      unsigned int prev = 0;
      if (lane == 0) prev = atomicAdd(tick + tile, 1u);
      prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
      store = prev == static_cast<unsigned int>(KC - 1);
      if (store) {
        __threadfence();
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          for (int kk = 0; kk < KC; ++kk) {
            const float4 o = __ldcg(pp + ((static_cast<size_t>(kk) * tiles + tile) * NB + nb) * 32 + lane);
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
        if (lane == 0) tick[tile] = 0;
      }
    }
    if (store) {
      const int ps = part_of<MT, MP>(parts, tile);
      const int N = parts.N[ps];
      uint16_t* y = parts.y[ps];
      const int n_lo = (tile - (ps ? parts.tile_end[ps - 1] : 0)) * 16 + g, n_hi = n_lo + 8;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m0 = nb * 8 + 2 * t, m1 = m0 + 1;
        if constexpr (A4) {
          const float sa0 = m0 < M ? s_a[m0] : 0.0f, sa1 = m1 < M ? s_a[m1] : 0.0f;
          acc[nb][0] *= sa0;
          acc[nb][1] *= sa1;
          acc[nb][2] *= sa0;
          acc[nb][3] *= sa1;
        }
        if (n_lo < N && m0 < M) y[static_cast<size_t>(m0) * N + n_lo] = f32_to_bf16_bits(acc[nb][0]);
        if (n_lo < N && m1 < M) y[static_cast<size_t>(m1) * N + n_lo] = f32_to_bf16_bits(acc[nb][1]);
        if (n_hi < N && m0 < M) y[static_cast<size_t>(m0) * N + n_hi] = f32_to_bf16_bits(acc[nb][2]);
        if (n_hi < N && m1 < M) y[static_cast<size_t>(m1) * N + n_hi] = f32_to_bf16_bits(acc[nb][3]);
      }
    }
  }
}

// dynamic shared memory for MT token slots over Gc staged groups (activations, K-slice reduction
// buffer, offsets of the integer-code modes)
inline size_t smem_bytes(int MT, int Gc) {
  return static_cast<size_t>(Gc) * 16 * MT * 16 + 2 * static_cast<size_t>(kWarps) * ((MT + 7) / 8) * 32 * 16 +
         static_cast<size_t>(Gc) * MT * sizeof(float);
}
constexpr size_t kSmemCap = 200 * 1024;

// K chunks across CTAs: the fewest (a divisor of the group count) whose staged activations fit
// shared memory; 0 if none does.
inline int pick_kc(int MT, int G) {
  for (int kc = 1; kc <= G; ++kc)
    if (G % kc == 0 && smem_bytes(MT, G / kc) <= kSmemCap) return kc;
  return 0;
}

// K split among a CTA's warps: the fewest rounds of (groups per slice + fixed cost), ties to the
// wider grid, among the splits whose slices hold a multiple of D groups; false if there is none.
inline bool pick_ks(long long tiles, int Gc, int KC, int D, int* best_ks, int* best_grid, long long* cost_out = nullptr) {
  const int chunk_grids = std::max(1, num_sms() / KC);  // CTAs per K chunk
  long long best_cost = -1;
  for (int ks = 1; ks <= kWarps; ks *= 2) {
    if (Gc % ks != 0 || (Gc / ks) % D != 0) continue;
    const long long slots = kWarps / ks;
    const int grid = static_cast<int>(std::min<long long>(chunk_grids, (tiles + slots - 1) / slots));
    const long long rounds = (tiles + grid * slots - 1) / (grid * slots);
    const long long cost = rounds * (Gc / ks + 2);
    if (best_cost < 0 || cost < best_cost || (cost == best_cost && grid > *best_grid)) {
      best_cost = cost;
      *best_ks = ks;
      *best_grid = grid;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best_cost >= 0;
}

// Groups in flight per warp for MT token slots (the weights wait in 8 registers per group and lane).
constexpr int depth_of(int MT) { return MT <= 16 ? 4 : 1; }

// K chunks for up to sixteen token slots: besides making the staged activations fit, chunks let a
// layer with few row tiles but long K keep more warps streaming (each warp's serial share is what
// a latency-bound stream pays for), and they shrink what every CTA stages: all CTAs read the same
// x, so staging 16 tokens' 128 KB per CTA takes ~5 us.  Among the chunk counts that fit, the one
// with the fewest groups per warp plus the fixup of split tiles (about 4 groups' time + a quarter
// per chunk) plus the staging (0.005 per staged (group, token slot): fitted to Llama-2-70B layers
// at 4 to 16 tokens), ties to fewer chunks.  E.g. the Llama-3-8B down layer (256 row tiles, 112
// groups) at one token takes seven chunks of 16 groups instead of one chunk in which only 1024 of
// the 2432 warps stream (28 groups each); at 16 tokens Llama-2-70B gate_up takes four chunks
// instead of two (46.3 -> 43.2 us), q/o four (22.7 -> 20.3 us), down eight instead of seven (51.1
// -> 45.4 us), and down at 4 tokens four instead of two (39.6 -> 37.4 us).  32 slots keep the
// fewest chunks that fit.  Deterministic in (MT, N, G, SM count), so the workspace size and the
// launch agree.
inline int plan_kc(int MT, int N, int G) {
  const int kc_min = pick_kc(MT, G);
  if (kc_min == 0 || MT > 16) return kc_min;
  const long long tiles = (static_cast<long long>(N) + 15) / 16;
  const int D = depth_of(MT);
  int best_kc = kc_min;
  double best = -1.0;
  for (int kc = kc_min; kc <= G; ++kc) {
    if (G % kc != 0 || smem_bytes(MT, G / kc) > kSmemCap) continue;
    int ks = 1, grid = 1;
    long long c = 0;
    if (!pick_ks(tiles, G / kc, kc, D, &ks, &grid, &c)) continue;
    const double cost = static_cast<double>(c) + (kc > 1 ? 4.0 + 0.25 * kc : 0.0) + 0.005 * (G / kc) * MT;
    if (best < 0.0 || cost < best) {
      best = cost;
      best_kc = kc;
    }
  }
  return best_kc;
}

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace bytes of the chunk partials and tile tickets (0 when K is not chunked).
inline size_t chunk_ws_bytes(int MT, int N, int G, int KC) {
  if (KC <= 1) return 0;
  const size_t tiles = (static_cast<size_t>(N) + 15) / 16;
  return al256(static_cast<size_t>(KC) * tiles * ((MT + 7) / 8) * 32 * 16) + al256(tiles * sizeof(unsigned int));
}

struct Outs {
  int8_t* xq;
  float* xs;
  int32_t* acc;
  const float* s_in;     // codes mode: the per-token scales of the staged codes
  float* part;           // K chunks: [KC][tiles][NB][32] float4 partial tiles
  unsigned int* tick;    // K chunks: [tiles] arrival counters (zero between calls)
  WsGuard guard;         // the workspace's layout claim
};

template <int QB, bool ACC, int MT, int D>
qspec_status launch_d(const uint16_t* x, const Parts& P, int M, int N, int K,
                      Outs o, int best_ks, int KC, int best_grid, cudaStream_t stream) {
  const size_t smem = smem_bytes(MT, K / kGroup / KC);
  // the part lookup is compiled in where several parts can reach it (see part_of)
  constexpr bool kMP = MT <= kPartsMaxMT && QB != 0;
  auto kern = KC > 1 ? gemv_kernel<QB, ACC, MT, D, true, kMP> : gemv_kernel<QB, ACC, MT, D, false, kMP>;
  if constexpr (MT <= kPartsMaxMT && QB == 0) {
    if (P.n > 1) kern = KC > 1 ? gemv_kernel<QB, ACC, MT, D, true, true> : gemv_kernel<QB, ACC, MT, D, false, true>;
  }
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
  return cudaLaunchKernelEx(&cfg, kern, x, P, M, K, best_ks, KC, o.xq, o.xs, o.acc, o.s_in, o.part,
                            o.tick, o.guard) == cudaSuccess
             ? QSPEC_OK
             : QSPEC_ERR_CUDA;
}

// The cheapest warp split over the depths D, D / 2, .., 1 (cost as in pick_ks); -1 if none fits.
inline long long cost_upto(long long tiles, int Gc, int KC, int D) {
  long long best = -1;
  for (int d = D; d >= 1; d /= 2) {
    int ks = 1, grid = 1;
    long long c = -1;
    if (pick_ks(tiles, Gc, KC, d, &ks, &grid, &c) && (best < 0 || c < best)) best = c;
  }
  return best;
}

// Launches with D groups in flight unless a shallower pipeline fits no split at D or allows a split
// at least a quarter cheaper: a slice of Gc groups must hold a multiple of D, so e.g. the Llama-3-8B
// down layer at sixteen tokens (4 chunks of 28 groups) only runs unsplit at D = 4 -- 16 warps to a
// CTA, 64 CTAs -- but two ways split at D = 2, on twice the CTAs.
template <int QB, bool ACC, int MT, int D>
qspec_status launch_depth(const uint16_t* x, const Parts& P, int M, int N, int K,
                          Outs o, int KC, cudaStream_t stream) {
  int ks = 1, grid = 1;
  long long c = -1;
  const long long tiles = (static_cast<long long>(N) + 15) / 16;
  const int Gc = K / kGroup / KC;
  const bool fits = pick_ks(tiles, Gc, KC, D, &ks, &grid, &c);
  if constexpr (D > 1) {
    const long long below = cost_upto(tiles, Gc, KC, D / 2);
    if (!fits || (below >= 0 && 4 * below <= 3 * c))
      return launch_depth<QB, ACC, MT, D / 2>(x, P, M, N, K, o, KC, stream);
  }
  if (!fits) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  return launch_d<QB, ACC, MT, D>(x, P, M, N, K, o, ks, KC, grid * KC, stream);
}

// Groups in flight per warp (the weights wait in 8 registers per group and lane): 4 up to eight
// tokens, 2 for sixteen (two column blocks of accumulators), 1 for 32; the checking path (int32
// group sums out) at most 2.
template <int QB, int MT>
qspec_status launch(const uint16_t* x, const Parts& P, int M, int N, int K,
                    Outs o, int KC, cudaStream_t stream) {
  if constexpr (QB != 0) {
    if (o.acc) return launch_depth<QB, true, MT, (MT < 32 ? 2 : 1)>(x, P, M, N, K, o, KC, stream);
  }
  return launch_depth<QB, false, MT, depth_of(MT)>(x, P, M, N, K, o, KC, stream);
}

// The modes that quantise inside the kernel (QB = 4, 8) serve at most three tokens (from four on
// the separate quantiser runs and QB = 1 stages its codes), so they are instantiated for up to 4
// token slots only; 32 slots serve W4A16 and codes.
template <int QB, int MT>
qspec_status launch_slots(const uint16_t* x, const Parts& P, int M, int N, int K,
                          Outs o, int KC, cudaStream_t stream) {
  if constexpr ((QB == 4 || QB == 8) && MT > 4) {
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  } else {
    return launch<QB, MT>(x, P, M, N, K, o, KC, stream);
  }
}

// The launcher of one activation mode (0: W4A16, 4: W4A4, 8: W4A8, 1: staged codes) for MT token
// slots; each mode is instantiated in a translation unit of its own (they compile in parallel).
template <int QB>
qspec_status launch_mode(int MT, const uint16_t* x, const Parts& P, int M, int N, int K, Outs o, int KC,
                         cudaStream_t stream);

template <>
qspec_status launch_mode<0>(int, const uint16_t*, const Parts&, int, int, int, Outs, int, cudaStream_t);
template <>
qspec_status launch_mode<1>(int, const uint16_t*, const Parts&, int, int, int, Outs, int, cudaStream_t);
template <>
qspec_status launch_mode<4>(int, const uint16_t*, const Parts&, int, int, int, Outs, int, cudaStream_t);
template <>
qspec_status launch_mode<8>(int, const uint16_t*, const Parts&, int, int, int, Outs, int, cudaStream_t);

#define QSPEC_GEMV_MODE_UNIT(QB_)                                                                      \
  template <>                                                                                          \
  qspec_status launch_mode<QB_>(int MT, const uint16_t* x, const Parts& P, int M, int N, int K, Outs o, \
                                int KC, cudaStream_t stream) {                                         \
    switch (MT) {                                                                                      \
      case 1: return launch_slots<QB_, 1>(x, P, M, N, K, o, KC, stream);                        \
      case 2: return launch_slots<QB_, 2>(x, P, M, N, K, o, KC, stream);                        \
      case 4: return launch_slots<QB_, 4>(x, P, M, N, K, o, KC, stream);                        \
      case 8: return launch_slots<QB_, 8>(x, P, M, N, K, o, KC, stream);                        \
      case 16: return launch_slots<QB_, 16>(x, P, M, N, K, o, KC, stream);                      \
      default: return launch_slots<QB_, 32>(x, P, M, N, K, o, KC, stream);                      \
    }                                                                                                  \
  }

}  // namespace gemv_impl
}  // namespace qspec
