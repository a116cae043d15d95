// Steps a5-a8: the fused verify step over vocabulary logits.
//
// Tutorial "Speculative Decodingとは？LLM生成を速くする方法" (kasblo.com):
//  - section "greedy decodingでは一致するprefixを採用する": accept draft tokens while they equal the
//    target argmax; the first mismatch takes the target token; all-match adds the next target token;
//  - section "samplingでもtargetの確率分布を保つ": accept x with probability a(x) = min(1, p(x)/q(x))
//    (eq. a(x)); on rejection draw from the residual max(0, p - q) / sum (eq. p'(x)).
//
// All passes are HBM-bound streams over bf16 logits.  One CTA per (row, chunk of the vocabulary)
// keeps every SM streaming; the per-sequence combine runs in whichever CTA of the sequence finishes
// last (an atomic ticket per sequence, no spinning).  Counters are reset by that CTA, so the
// workspace is ready for the next call.
#include <cuda.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace qspec {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;        // 16-byte loads in flight per thread in the streaming passes
constexpr int kPlanCTAs = 1216;   // about 8 CTAs per SM on a 152-SM part (measured: greedy verify over
                                  // [512, 152064] 33.8 -> 31.7 us against 608 CTAs x 8 loads)
constexpr int kMinChunk = 2048;   // elements per CTA at least (4 KB of bf16)
constexpr int kSeg2 = 8;          // pass 2: contiguous elements per thread
constexpr int kChunk2 = kThreads * kSeg2;
constexpr int kPass2Chunks = 2;   // pass 2: chunks per CTA (their loads are in flight together)

enum : unsigned int { kErrBadToken = 2u };

struct Plan {
  int chunks;      // chunks per row
  int chunk_len;   // elements per chunk (multiple of 8)
};

// Chunks per row.  The argmax passes (greedy, top-1, tree) take about kPlanCTAs CTAs in all (more,
// smaller CTAs measured faster for them: greedy over [64 x 8, 152064] 31.7 us with 1536 CTAs, 37.7
// us with 1024).  Sampling pass 1 (one_wave) takes no more chunks than keep every CTA resident at
// once (about 8 per SM), so no partial second wave idles most of the GPU: its largest cell ([64 x 15,
// 152064], 960 rows) 76.2 -> 72.0 us for both passes with one chunk per row instead of two.
Plan plan_rows(int64_t rows, int V, bool one_wave = false) {
  int64_t c = one_wave ? kPlanCTAs / rows : (kPlanCTAs + rows - 1) / rows;
  const int64_t max_c = (V + kMinChunk - 1) / kMinChunk;
  if (c > max_c) c = max_c;
  if (c < 1) c = 1;
  int64_t len = ((V + c - 1) / c + 7) / 8 * 8;
  c = (V + len - 1) / len;
  return {static_cast<int>(c), static_cast<int>(len)};
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace layout (bytes).  Both verify calls use the same layout for a given (B, gamma, V).
struct Layout {
  Plan p1;            // pass-1 plan over B * (2 gamma + 1) rows (greedy uses B * (gamma + 1) rows)
  Plan pg;
  Plan pt;            // top-1 statistics: B * 2 gamma rows
  int chunks2;
  size_t err, cnt1, cnt2, seq_n, rowstat, part1, part2, part3, rec2, total;
};

// What sampling pass 1 hands to pass 2 for one sequence, in one 32-byte record: the first rejected
// position n (gamma: all accepted) and the softmax statistics of target row n and draft row n.
struct Rec2 {
  int n;
  float mt, inv_st;  // target row n: max and 1 / sum exp(l - max)
  float md, inv_sd;  // draft row n (0, 0 for the bonus row)
  float pad[3];
};

Layout layout(int B, int gamma, int V) {
  Layout L;
  L.pg = plan_rows(int64_t(B) * (gamma + 1), V);
  L.p1 = plan_rows(int64_t(B) * (2 * gamma + 1), V, true);
  L.pt = plan_rows(int64_t(B) * (2 * gamma), V);
  L.chunks2 = (V + kChunk2 - 1) / kChunk2;
  size_t off = 0;
  L.err = off;      off += 256;
  L.cnt1 = off;     off = align256(off + sizeof(unsigned int) * B);
  L.cnt2 = off;     off = align256(off + sizeof(unsigned int) * B);
  L.seq_n = off;    off = align256(off + sizeof(int) * B);
  L.rowstat = off;  off = align256(off + sizeof(float2) * size_t(B) * (2 * gamma + 1));
  const size_t part_g = sizeof(float2) * size_t(B) * (gamma + 1) * L.pg.chunks;
  const size_t part_s = sizeof(float2) * size_t(B) * (2 * gamma + 1) * L.p1.chunks;
  L.part1 = off;    off = align256(off + (part_g > part_s ? part_g : part_s));
  L.part2 = off;    off = align256(off + sizeof(float) * size_t(B) * L.chunks2 * (kThreads / 32));
  L.part3 = off;    off = align256(off + sizeof(float4) * size_t(B) * (2 * gamma) * L.pt.chunks);
  L.rec2 = off;     off = align256(off + sizeof(Rec2) * size_t(B));
  L.total = off;
  return L;
}

struct WS {
  unsigned int* err;
  unsigned int* cnt1;
  unsigned int* cnt2;
  int* seq_n;
  float2* rowstat;
  float2* part1;
  float* part2;
  float4* part3;
  Rec2* rec2;
};

WS bind(void* base, const Layout& L) {
  char* p = static_cast<char*>(base);
  return {reinterpret_cast<unsigned int*>(p + L.err), reinterpret_cast<unsigned int*>(p + L.cnt1),
          reinterpret_cast<unsigned int*>(p + L.cnt2), reinterpret_cast<int*>(p + L.seq_n),
          reinterpret_cast<float2*>(p + L.rowstat), reinterpret_cast<float2*>(p + L.part1),
          reinterpret_cast<float*>(p + L.part2), reinterpret_cast<float4*>(p + L.part3),
          reinterpret_cast<Rec2*>(p + L.rec2)};
}

// ------------------------------------------------------------------ argmax (greedy)

// (value, index) order for argmax: larger value wins, equal values go to the lower index.
__device__ __forceinline__ void argmax_take(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
}

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
    argmax_take(bv, bi, ov, oi);
  }
}

// Block-wide argmax; every thread gets the result.
__device__ __forceinline__ void block_argmax(float& bv, int& bi) {
  __shared__ float sv[kThreads / 32];
  __shared__ int si[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  warp_argmax(bv, bi);
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  bv = lane < kThreads / 32 ? sv[lane] : -INFINITY;
  bi = lane < kThreads / 32 ? si[lane] : INT_MAX;
  warp_argmax(bv, bi);
  __syncthreads();
}

// Scan logits [beg, end) of one row with each thread taking 16-byte vectors t, t+256, ...
template <bool kVec>
__device__ __forceinline__ void scan_argmax(const uint16_t* __restrict__ rp, int beg, int end, float& bv,
                                            int& bi) {
  if (kVec) {
    const int nv = (end - beg) >> 3;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + beg);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kUnroll * kThreads) {
      uint4 u[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int v = v0 + t * kThreads;
        u[t] = v < nv ? ld_stream_v4(vp + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int v = v0 + t * kThreads;
        if (v < nv) {
          const int i0 = beg + 8 * v;
          const uint32_t w[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            argmax_take(bv, bi, bf16_lo(w[e]), i0 + 2 * e);
            argmax_take(bv, bi, bf16_hi(w[e]), i0 + 2 * e + 1);
          }
        }
      }
    }
  } else {
    for (int i = beg + threadIdx.x; i < end; i += kThreads) argmax_take(bv, bi, bf16_lo(rp[i]), i);
  }
}

// One CTA per (row, chunk); the last CTA of a sequence applies the greedy rule.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) greedy_kernel(const uint16_t* __restrict__ L,
                                                          const int32_t* __restrict__ d, int gamma,
                                                          int V, Plan plan, WS ws,
                                                          int32_t* __restrict__ accept_len,
                                                          int32_t* __restrict__ out_tok,
                                                          int32_t* __restrict__ tgt_argmax) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x / plan.chunks;
  const int c = blockIdx.x % plan.chunks;
  const int beg = c * plan.chunk_len;
  const int end = min(V, beg + plan.chunk_len);
  float bv = -INFINITY;
  int bi = INT_MAX;
  scan_argmax<kVec>(L + row * V, beg, end, bv, bi);
  block_argmax(bv, bi);

  __shared__ bool s_last;
  const int G1 = gamma + 1;
  const int b = static_cast<int>(row / G1);
  if (threadIdx.x == 0) {
    ws.part1[row * plan.chunks + c] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    const unsigned int prev = atomicAdd(ws.cnt1 + b, 1u);
    s_last = prev == static_cast<unsigned int>(G1 * plan.chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int s_t[QSPEC_MAX_GAMMA + 1];
  __shared__ int s_x[QSPEC_MAX_GAMMA];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the draft tokens, read by gamma threads at once (not one dependent read after another)
  if (threadIdx.x < gamma) {
    const int x = d[int64_t(b) * gamma + threadIdx.x];
    s_x[threadIdx.x] = x;
    if (x < 0 || x >= V) atomicOr(ws.err, kErrBadToken);
  }
  for (int i = warp; i < G1; i += kThreads / 32) {
    const int64_t r = int64_t(b) * G1 + i;
    float v = -INFINITY;
    int k = INT_MAX;
    for (int cc = lane; cc < plan.chunks; cc += 32) {
      const float2 pp = __ldcg(ws.part1 + r * plan.chunks + cc);
      argmax_take(v, k, pp.x, __float_as_int(pp.y));
    }
    warp_argmax(v, k);
    if (lane == 0) s_t[i] = k;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < gamma && s_x[n] == s_t[n]) ++n;
    accept_len[b] = n;
    for (int i = 0; i < G1; ++i) {
      out_tok[int64_t(b) * G1 + i] = i < n ? s_x[i] : (i == n ? s_t[n] : -1);
      if (tgt_argmax) tgt_argmax[int64_t(b) * G1 + i] = s_t[i];
    }
    ws.cnt1[b] = 0;
  }
}

// ------------------------------------------------------------------ softmax statistics (sampling)

// Running (max, sum of exp(l - max)) of a set of logits; -inf logits contribute nothing.
struct MS {
  float m, s;
};

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.0f};
  return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

// 2^x from the SFU (ex2.approx: relative error below 2^-22).  Used for the streamed row sums and the
// residual terms of pass 2 (exp_diff): the terms that matter have x near 0, and the fp32 summation
// of ~10^5 terms already carries a larger relative error; the probabilities reported per token use
// the accurate expf.
__device__ __forceinline__ float exp2_sfu(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
constexpr float kLog2e = 1.4426950408889634f;

// The reference m of a running (m, s) need not be the maximum: s = sum exp(l - m) stays exact in
// meaning for any m, and terms up to 2^24 cannot overflow fp32 over any row.  So the eight terms of
// a vector are taken against the current m first, and m moves only when their sum reaches 2^24 (a
// value more than ~16.6 above m) or is not finite (m still -inf, or an infinite / NaN logit): then
// the vector is redone against max(m, its maximum).  The common path carries no max and no branch
// per value; consumers use exp(l - m) / s.
constexpr float kMoveSum = 16777216.0f;  // 2^24

__device__ __forceinline__ float exp_sum8(const float (&v)[8], float m) {
  const float c = m * kLog2e;  // exp(v - m) = 2^(v log2e - m log2e), one FFMA per term
  float t[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) t[e] = exp2_sfu(fmaf(v[e], kLog2e, -c));
  return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));  // pairwise: depth 3
}

__device__ __forceinline__ void ms_add8(MS& a, const float (&v)[8]) {
  float sb = exp_sum8(v, a.m);
  if (!(sb < kMoveSum)) {
    const float m8 = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
    if (m8 > a.m) {
      a.s = a.m == -INFINITY ? 0.0f : a.s * expf(a.m - m8);
      a.m = m8;
    }
    sb = a.m == -INFINITY ? 0.0f : exp_sum8(v, a.m);
  }
  a.s += sb;
}

__device__ __forceinline__ MS warp_ms(MS a) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    MS o{__shfl_xor_sync(0xFFFFFFFFu, a.m, off), __shfl_xor_sync(0xFFFFFFFFu, a.s, off)};
    a = ms_merge(a, o);
  }
  return a;
}

__device__ __forceinline__ MS block_ms(MS a) {
  __shared__ float sm[kThreads / 32], ss[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  a = warp_ms(a);
  if (lane == 0) { sm[warp] = a.m; ss[warp] = a.s; }
  __syncthreads();
  MS r{lane < kThreads / 32 ? sm[lane] : -INFINITY, lane < kThreads / 32 ? ss[lane] : 0.0f};
  r = warp_ms(r);
  __syncthreads();
  return r;
}

template <bool kVec>
__device__ __forceinline__ MS scan_ms(const uint16_t* __restrict__ rp, int beg, int end) {
  MS a{-INFINITY, 0.0f};
  if (kVec) {
    const int nv = (end - beg) >> 3;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + beg);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kUnroll * kThreads) {
      uint4 u[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int v = v0 + t * kThreads;
        u[t] = v < nv ? ld_stream_v4(vp + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        if (v0 + t * kThreads < nv) {
          const uint32_t w[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
          float f[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) { f[2 * e] = bf16_lo(w[e]); f[2 * e + 1] = bf16_hi(w[e]); }
          ms_add8(a, f);
        }
      }
    }
  } else {
    for (int i = beg + threadIdx.x; i < end; i += kThreads) {
      float f[8];
      f[0] = bf16_lo(rp[i]);
#pragma unroll
      for (int e = 1; e < 8; ++e) f[e] = -INFINITY;
      ms_add8(a, f);
    }
  }
  return a;
}

// Pass 1 of sampling verify: softmax statistics of every target and draft row; the last CTA of a
// sequence evaluates a_i = min(1, p_i(d_i) / q_i(d_i)) at every draft position and the first
// rejection n.  Rows [0, B(gamma+1)) are target rows, the next B*gamma rows draft rows.
template <bool kVec>
__global__ void __launch_bounds__(kThreads, 8) sample_pass1_kernel(
    const uint16_t* __restrict__ Lt, const uint16_t* __restrict__ Ld, const int32_t* __restrict__ d,
    const float* __restrict__ u_acc, int B, int gamma, int V, Plan plan, WS ws,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tok, float* __restrict__ accept_prob,
    float* __restrict__ p_tok, float* __restrict__ q_tok) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x / plan.chunks;
  const int c = blockIdx.x % plan.chunks;
  const int G1 = gamma + 1;
  const int64_t n_tgt = int64_t(B) * G1;
  const bool is_tgt = row < n_tgt;
  const uint16_t* rp = is_tgt ? Lt + row * V : Ld + (row - n_tgt) * V;
  const int b = static_cast<int>(is_tgt ? row / G1 : (row - n_tgt) / gamma);
  const int beg = c * plan.chunk_len;
  const int end = min(V, beg + plan.chunk_len);
  MS a = scan_ms<kVec>(rp, beg, end);
  a = block_ms(a);

  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    ws.part1[row * plan.chunks + c] = make_float2(a.m, a.s);
    __threadfence();
    const unsigned int prev = atomicAdd(ws.cnt1 + b, 1u);
    s_last = prev == static_cast<unsigned int>((2 * gamma + 1) * plan.chunks - 1);
  }
  __syncthreads();
  // Pass 2 may start launching now; it waits for this grid's completion before reading.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!s_last) return;
  __threadfence();

  __shared__ float2 s_stat[2 * QSPEC_MAX_GAMMA + 1];  // [0, G1): target rows; then draft rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < 2 * gamma + 1; i += kThreads / 32) {
    const int64_t r = i < G1 ? int64_t(b) * G1 + i : n_tgt + int64_t(b) * gamma + (i - G1);
    MS t{-INFINITY, 0.0f};
    for (int cc = lane; cc < plan.chunks; cc += 32) {
      const float2 pp = __ldcg(ws.part1 + r * plan.chunks + cc);
      t = ms_merge(t, MS{pp.x, pp.y});
    }
    t = warp_ms(t);
    if (lane == 0) {
      s_stat[i] = make_float2(t.m, t.s);
      ws.rowstat[r] = make_float2(t.m, t.s);
    }
  }
  __syncthreads();
  // every draft position's test in a thread of its own (their reads of p and q at the draft token
  // are independent); thread 0 then takes the first rejection
  __shared__ int s_x[QSPEC_MAX_GAMMA], s_rej[QSPEC_MAX_GAMMA];
  if (threadIdx.x < gamma) {
    const int i = threadIdx.x;
    const int x = d[int64_t(b) * gamma + i];
    float p = 0.0f, q = 0.0f, acc = 0.0f;
    if (x >= 0 && x < V) {
      const float lt = bf16_lo(Lt[(int64_t(b) * G1 + i) * V + x]);
      const float ld = bf16_lo(Ld[(int64_t(b) * gamma + i) * V + x]);
      p = __fdiv_rn(expf(lt - s_stat[i].x), s_stat[i].y);
      q = __fdiv_rn(expf(ld - s_stat[G1 + i].x), s_stat[G1 + i].y);
      acc = q == 0.0f ? 1.0f : fminf(1.0f, __fdiv_rn(p, q));
    } else {
      atomicOr(ws.err, kErrBadToken);  // an invalid draft token is rejected
    }
    if (accept_prob) accept_prob[int64_t(b) * gamma + i] = acc;
    if (p_tok) p_tok[int64_t(b) * gamma + i] = p;
    if (q_tok) q_tok[int64_t(b) * gamma + i] = q;
    s_x[i] = x;
    s_rej[i] = !(u_acc[int64_t(b) * gamma + i] < acc);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = gamma;
    for (int i = gamma - 1; i >= 0; --i)
      if (s_rej[i]) n = i;
    accept_len[b] = n;
    for (int i = 0; i < G1; ++i)
      if (i != n) out_tok[int64_t(b) * G1 + i] = i < n ? s_x[i] : -1;
    ws.seq_n[b] = n;
    // the record as two 16-byte stores: n, max and 1 / sum of target row n, max and 1 / sum of draft
    // row n (zeros for the bonus row)
    const float md = n < gamma ? s_stat[G1 + n].x : 0.0f;
    const float inv_sd = n < gamma ? 1.0f / s_stat[G1 + n].y : 0.0f;
    int4* rec = reinterpret_cast<int4*>(ws.rec2 + b);
    rec[0] = make_int4(n, __float_as_int(s_stat[n].x), __float_as_int(1.0f / s_stat[n].y), __float_as_int(md));
    rec[1] = make_int4(__float_as_int(inv_sd), 0, 0, 0);
    ws.cnt1[b] = 0;
  }
}

// ------------------------------------------------------------------ residual / bonus resampling

struct RowPair {
  const uint16_t* t;  // target row n
  const uint16_t* q;  // draft row n (unused for the bonus row)
  float mt, inv_st, md, inv_sd;
  bool bonus;         // r = p (bonus token, or the p fallback when the residual sums to 0)
};

// exp(d) for d = l - m of two bf16-valued floats (exact in fp32): 2^(d log2 e) from the SFU.  The
// error is relative 2^-22 from ex2.approx plus |d| log2(e) 2^-24 ln 2 from rounding the product --
// largest for the smallest terms and never shared by a whole row, so a residual max(0, p - q) keeps
// its relative accuracy where p and q nearly cancel.
__device__ __forceinline__ float exp_diff(float d) { return exp2_sfu(d * kLog2e); }

__device__ __forceinline__ float resid(const RowPair& rp, float lt, float ld) {
  const float p = exp_diff(lt - rp.mt) * rp.inv_st;
  if (rp.bonus) return p;
  return fmaxf(0.0f, p - exp_diff(ld - rp.md) * rp.inv_sd);
}

// r values of the kSeg2 contiguous elements from i0 (zeros beyond V).
template <bool kVec>
__device__ __forceinline__ void seg_values_at(const RowPair& rp, int V, int i0, float (&r)[kSeg2]) {
  if (kVec && i0 + kSeg2 <= V) {
    const uint4 ut = ld_stream_v4(rp.t + i0);
    const uint4 uq = rp.bonus ? make_uint4(0, 0, 0, 0) : ld_stream_v4(rp.q + i0);
    const uint32_t wt[4] = {ut.x, ut.y, ut.z, ut.w};
    const uint32_t wq[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      r[2 * e] = resid(rp, bf16_lo(wt[e]), bf16_lo(wq[e]));
      r[2 * e + 1] = resid(rp, bf16_hi(wt[e]), bf16_hi(wq[e]));
    }
  } else {
#pragma unroll
    for (int e = 0; e < kSeg2; ++e) {
      const int i = i0 + e;
      r[e] = i < V ? resid(rp, bf16_lo(rp.t[i]), rp.bonus ? 0.0f : bf16_lo(rp.q[i])) : 0.0f;
    }
  }
}

// Pass 2 keeps one residual sum per warp segment: the 32 x kSeg2 = 256 contiguous elements that the
// lanes of one warp cover in a chunk (element c kChunk2 + (32 w + lane) kSeg2 + e).
constexpr int kSegsPerChunk = kThreads / 32;

// The sum of one warp segment's r values (lane sums, then a fixed xor-shuffle tree).
__device__ __forceinline__ float warp_segment_sum(const float (&r)[kSeg2]) {
  float v = 0.0f;
#pragma unroll
  for (int e = 0; e < kSeg2; ++e) v += r[e];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// Inclusive prefix sums over the block of four consecutive values per thread (in thread order), in a
// fixed order; excl gets the sum before the thread's first value; returns the block's total, which
// equals the last thread's last prefix.
__device__ __forceinline__ float block_incl_scan4(float (&v)[4], float& excl_out) {
  __shared__ float s_w[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v[1] += v[0];
  v[2] += v[1];
  v[3] += v[2];
  const float t = v[3];
  float incl = t;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  float wbase = 0.0f, total = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const float x = s_w[w];
    if (w < warp) wbase += x;
    total += x;
  }
  const float excl = wbase + (incl - t);
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] += excl;
  excl_out = excl;
  __syncthreads();  // s_w is reused by the next call
  return total;
}

// Pass 2: per (sequence, group of kPass2Chunks chunks of 2048) residual mass of row n, one sum per
// warp segment of 256 elements; the last CTA of a sequence scans the segment sums in index order
// (a block scan), finds the segment where the running sum passes u R, and one warp rescans those 256
// elements for the token (the inverse CDF).
template <bool kVec>
__global__ void __launch_bounds__(kThreads, 8) sample_pass2_kernel(
    const uint16_t* __restrict__ Lt, const uint16_t* __restrict__ Ld,
    const float* __restrict__ u_res, int B, int gamma, int V, int chunks2, int ctas_per_seq, WS ws,
    int32_t* __restrict__ out_tok) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int groups = (chunks2 + kPass2Chunks - 1) / kPass2Chunks;
  const int b = blockIdx.x / ctas_per_seq;
  const int g0 = blockIdx.x % ctas_per_seq;  // this CTA takes chunk groups g0, g0 + ctas_per_seq, ..
  const int G1 = gamma + 1;
  // pass 1's record for this sequence (one 32-byte read)
  const int4 r0 = __ldcg(reinterpret_cast<const int4*>(ws.rec2 + b));
  const int4 r1 = __ldcg(reinterpret_cast<const int4*>(ws.rec2 + b) + 1);
  const int n = r0.x;
  RowPair rp;
  rp.bonus = n == gamma;
  rp.t = Lt + (int64_t(b) * G1 + n) * V;
  rp.mt = __int_as_float(r0.y);
  rp.inv_st = __int_as_float(r0.z);
  rp.q = rp.bonus ? nullptr : Ld + (int64_t(b) * gamma + n) * V;
  rp.md = __int_as_float(r0.w);
  rp.inv_sd = __int_as_float(r1.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = chunks2 * kSegsPerChunk;
  float* segs = ws.part2 + int64_t(b) * nseg;
  for (int g = g0; g < groups; g += ctas_per_seq) {
    const int c0 = g * kPass2Chunks;
    float r[kPass2Chunks][kSeg2];
#pragma unroll
    for (int k = 0; k < kPass2Chunks; ++k) {
      if (c0 + k < chunks2) {
        seg_values_at<kVec>(rp, V, (c0 + k) * kChunk2 + threadIdx.x * kSeg2, r[k]);
      } else {
#pragma unroll
        for (int e = 0; e < kSeg2; ++e) r[k][e] = 0.0f;
      }
    }
#pragma unroll
    for (int k = 0; k < kPass2Chunks; ++k) {
      const float v = warp_segment_sum(r[k]);
      if (lane == 0 && c0 + k < chunks2) segs[(c0 + k) * kSegsPerChunk + warp] = v;
    }
  }
  __threadfence();  // every segment sum is published before the ticket below

  __shared__ bool s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(ws.cnt2 + b, 1u);
    s_last = prev == static_cast<unsigned int>(ctas_per_seq - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ float s_R, s_before;
  __shared__ int s_found, s_last_pos;
  const float u = u_res[int64_t(b) * G1 + n];
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (attempt == 1) {
      // The residual has no mass (p == q in fp32): draw from p instead.
      rp.bonus = true;
      for (int cc = 0; cc < chunks2; ++cc) {
        float r[kSeg2];
        seg_values_at<kVec>(rp, V, cc * kChunk2 + threadIdx.x * kSeg2, r);
        const float v = warp_segment_sum(r);
        if (lane == 0) segs[cc * kSegsPerChunk + warp] = v;
      }
      __threadfence();
      __syncthreads();
    }
    // Segment sums in tiles of 4 per thread: R first (pass 0), then the first segment whose running
    // sum passes u R (pass 1), with the running sum before it; the last segment with mass as the
    // fallback when rounding leaves no crossing.
    if (threadIdx.x == 0) {
      s_found = INT_MAX;
      s_last_pos = -1;
    }
    float R = 0.0f;
    for (int pass = 0; pass < 2; ++pass) {
      const float target = u * R;
      float carry = 0.0f;
      for (int t0 = 0; t0 < nseg; t0 += 4 * kThreads) {
        float v[4], raw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = t0 + threadIdx.x * 4 + e;
          raw[e] = i < nseg ? __ldcg(segs + i) : 0.0f;
          v[e] = raw[e];
        }
        float excl = 0.0f;
        const float tot = block_incl_scan4(v, excl);
        if (pass == 1) {
          // the prefixes rise with i (r >= 0), so the crossing is a thread's first e past the target
          // whose previous prefix is not; one atomic per warp for the lowest such lane, and likewise
          // for the last segment with mass
          int first = -1, lastp = -1;
          float prev = carry + excl, before = 0.0f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = t0 + threadIdx.x * 4 + e;
            if (i < nseg && first < 0 && carry + v[e] > target) {
              first = i;
              before = prev;
            }
            if (i < nseg && raw[e] > 0.0f) lastp = i;
            prev = carry + v[e];
          }
          const unsigned int fm = __ballot_sync(0xFFFFFFFFu, first >= 0);
          if (fm != 0u && lane == __ffs(fm) - 1) atomicMin(&s_found, first);
          const unsigned int lm = __ballot_sync(0xFFFFFFFFu, lastp >= 0);
          if (lm != 0u && lane == 31 - __clz(lm)) atomicMax(&s_last_pos, lastp);
          __syncthreads();
          if (first >= 0 && first == s_found) s_before = before;
          __syncthreads();
          if (s_found != INT_MAX) break;  // (uniform: read after the barrier)
        }
        carry += tot;
      }
      if (pass == 0) R = carry;
    }
    if (threadIdx.x == 0) s_R = R;
    __syncthreads();
    if (R > 0.0f || attempt == 1) break;
    __syncthreads();
  }
  // one warp rescans the chosen segment: the first element whose running sum (from the segment's
  // start) passes u R - (mass before it); if rounding leaves none, the segment's last element with
  // r > 0 (the row's last such element when no segment crossed: target infinity)
  if (warp == 0) {
    const bool crossed = s_found != INT_MAX;
    const int seg = crossed ? s_found : s_last_pos;
    int j = -1;
    if (seg >= 0) {
      const float tgt = crossed ? u * s_R - s_before : INFINITY;
      const int c = seg / kSegsPerChunk, w = seg - c * kSegsPerChunk;
      const int i0 = c * kChunk2 + (w * 32 + lane) * kSeg2;
      float r[kSeg2];
      seg_values_at<kVec>(rp, V, i0, r);
      float sum = 0.0f;
      int last_e = -1;
#pragma unroll
      for (int e = 0; e < kSeg2; ++e) {
        sum += r[e];
        if (r[e] > 0.0f) last_e = e;
      }
      float incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
      }
      int hit = -1;
      if (incl > tgt) {
        float run = incl - sum;
#pragma unroll
        for (int e = 0; e < kSeg2; ++e) {
          run += r[e];
          if (hit < 0 && run > tgt) hit = e;
        }
        if (hit < 0) hit = last_e;  // rounding: the lane's sum crossed but no element did
      }
      const unsigned int hits = __ballot_sync(0xFFFFFFFFu, hit >= 0);
      if (hits != 0u) {
        const int src = __ffs(hits) - 1;
        j = __shfl_sync(0xFFFFFFFFu, i0 + hit, src);
      } else {
        const unsigned int pos = __ballot_sync(0xFFFFFFFFu, last_e >= 0);
        if (pos != 0u) {
          const int src = 31 - __clz(pos);
          j = __shfl_sync(0xFFFFFFFFu, i0 + last_e, src);
        }
      }
    }
    if (lane == 0) {
      out_tok[int64_t(b) * G1 + n] = j;
      ws.cnt2[b] = 0;
    }
  }
}

// ------------------------------------------------------------------ top-1 statistics

// Per draft position i < gamma of each sequence: the most likely token of the target (W4A16) row i
// and of the draft (W4A4) row i, and the probability each row gives its own most likely token,
// softmax max = 1 / sum_j exp(l_j - max).  One pass per (row, chunk): argmax and online (max, sum);
// the last CTA of a sequence merges the chunks.  Rows [0, B gamma) are target rows, then draft rows.
// One read of logits [beg, end): argmax (lowest index on ties) and the running (max, sum exp).
template <bool kVec>
__device__ __forceinline__ void scan_top1(const uint16_t* __restrict__ rp, int beg, int end, float& bv, int& bi,
                                          MS& a) {
  if (kVec) {
    const int nv = (end - beg) >> 3;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + beg);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kUnroll * kThreads) {
      uint4 u[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int v = v0 + t * kThreads;
        u[t] = v < nv ? ld_stream_v4(vp + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int v = v0 + t * kThreads;
        if (v < nv) {
          const int i0 = beg + 8 * v;
          const uint32_t w[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
          float f[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) { f[2 * e] = bf16_lo(w[e]); f[2 * e + 1] = bf16_hi(w[e]); }
#pragma unroll
          for (int e = 0; e < 8; ++e) argmax_take(bv, bi, f[e], i0 + e);
          ms_add8(a, f);
        }
      }
    }
  } else {
    for (int i = beg + threadIdx.x; i < end; i += kThreads) {
      float f[8];
      f[0] = bf16_lo(rp[i]);
#pragma unroll
      for (int e = 1; e < 8; ++e) f[e] = -INFINITY;
      argmax_take(bv, bi, f[0], i);
      ms_add8(a, f);
    }
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) top1_kernel(const uint16_t* __restrict__ Lt,
                                                        const uint16_t* __restrict__ Ld, int B, int gamma,
                                                        int V, Plan plan, WS ws, int32_t* __restrict__ tgt_top1,
                                                        int32_t* __restrict__ draft_top1,
                                                        float* __restrict__ tgt_p1, float* __restrict__ draft_p1,
                                                        float high, double* __restrict__ tally) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x / plan.chunks;
  const int c = blockIdx.x % plan.chunks;
  const int64_t n_tgt = int64_t(B) * gamma;
  const bool is_tgt = row < n_tgt;
  const int64_t rr = is_tgt ? row : row - n_tgt;  // (b, i) = (rr / gamma, rr % gamma)
  const int b = static_cast<int>(rr / gamma), i = static_cast<int>(rr % gamma);
  const uint16_t* rp = is_tgt ? Lt + (int64_t(b) * (gamma + 1) + i) * V : Ld + rr * V;
  const int beg = c * plan.chunk_len;
  const int end = min(V, beg + plan.chunk_len);
  float bv = -INFINITY;
  int bi = INT_MAX;
  MS a{-INFINITY, 0.0f};
  scan_top1<kVec>(rp, beg, end, bv, bi, a);
  block_argmax(bv, bi);
  a = block_ms(a);

  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    ws.part3[row * plan.chunks + c] = make_float4(bv, __int_as_float(bi), a.m, a.s);
    __threadfence();
    const unsigned int prev = atomicAdd(ws.cnt1 + b, 1u);
    s_last = prev == static_cast<unsigned int>(2 * gamma * plan.chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int s_tok[2 * QSPEC_MAX_GAMMA];
  __shared__ float s_p1[2 * QSPEC_MAX_GAMMA];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = warp; k < 2 * gamma; k += kThreads / 32) {
    const int64_t r = k < gamma ? int64_t(b) * gamma + k : n_tgt + int64_t(b) * gamma + (k - gamma);
    float v = -INFINITY;
    int idx = INT_MAX;
    MS t{-INFINITY, 0.0f};
    for (int cc = lane; cc < plan.chunks; cc += 32) {
      const float4 pp = __ldcg(ws.part3 + r * plan.chunks + cc);
      argmax_take(v, idx, pp.x, __float_as_int(pp.y));
      t = ms_merge(t, MS{pp.z, pp.w});
    }
    warp_argmax(v, idx);
    t = warp_ms(t);
    if (lane == 0) {
      // the top-1 token's probability exp(max - m) / s (m: the running reference, not always the max)
      const float p1 = t.s > 0.0f ? __fdiv_rn(expf(v - t.m), t.s) : 0.0f;
      s_tok[k] = idx;
      s_p1[k] = p1;
      const int64_t o = int64_t(b) * gamma + (k < gamma ? k : k - gamma);
      if (k < gamma) {
        tgt_top1[o] = idx;
        if (tgt_p1) tgt_p1[o] = p1;
      } else {
        draft_top1[o] = idx;
        if (draft_p1) draft_p1[o] = p1;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (tally) {
      // positions, agree, both > high, agreeing among them, both <= high, agreeing among them,
      // sum of target top-1 probabilities, sum of draft top-1 probabilities
      double t[8] = {};
      for (int k = 0; k < gamma; ++k) {
        const bool agree = s_tok[k] == s_tok[gamma + k];
        const float pt = s_p1[k], pd = s_p1[gamma + k];
        t[0] += 1.0;
        t[1] += agree;
        if (pt > high && pd > high) { t[2] += 1.0; t[3] += agree; }
        if (pt <= high && pd <= high) { t[4] += 1.0; t[5] += agree; }
        t[6] += pt;
        t[7] += pd;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) atomicAdd(tally + e, t[e]);
    }
    ws.cnt1[b] = 0;
  }
}

// ------------------------------------------------------------------ tree verification (greedy)

// Candidates form a tree instead of a chain: node j holds a token and its parent (-1: the committed
// prefix, else an earlier node), target row 0 scores the token after the prefix and row j + 1 the
// token after node j.  Greedy: from the prefix, follow the child whose token equals the target's
// most likely token at the current row (the lowest-index child if several), as long as one exists;
// the target's token where the walk stops is emitted after the accepted path.
struct TreeLayout {
  Plan p;
  size_t err, cnt, part, total;
};

TreeLayout tree_layout(int B, int T, int V) {
  TreeLayout L;
  L.p = plan_rows(int64_t(B) * (T + 1), V);
  size_t off = 0;
  L.err = off;  off += 256;  // first: qspec_check_status reads the error word at the start
  L.cnt = off;  off = align256(off + sizeof(unsigned int) * B);
  L.part = off; off = align256(off + sizeof(float2) * size_t(B) * (T + 1) * L.p.chunks);
  L.total = off;
  return L;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) tree_kernel(const uint16_t* __restrict__ L,
                                                        const int32_t* __restrict__ tok,
                                                        const int32_t* __restrict__ parent, int T, int V,
                                                        Plan plan, unsigned int* __restrict__ err,
                                                        unsigned int* __restrict__ cnt, float2* __restrict__ part,
                                                        int32_t* __restrict__ accept_len,
                                                        int32_t* __restrict__ out_tok,
                                                        int32_t* __restrict__ accept_nodes) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x / plan.chunks;
  const int c = blockIdx.x % plan.chunks;
  const int beg = c * plan.chunk_len;
  const int end = min(V, beg + plan.chunk_len);
  float bv = -INFINITY;
  int bi = INT_MAX;
  scan_argmax<kVec>(L + row * V, beg, end, bv, bi);
  block_argmax(bv, bi);

  __shared__ bool s_last;
  const int R = T + 1;
  const int b = static_cast<int>(row / R);
  if (threadIdx.x == 0) {
    part[row * plan.chunks + c] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    const unsigned int prev = atomicAdd(cnt + b, 1u);
    s_last = prev == static_cast<unsigned int>(R * plan.chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int s_t[QSPEC_MAX_TREE + 1];
  __shared__ int s_tok[QSPEC_MAX_TREE], s_par[QSPEC_MAX_TREE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < R; i += kThreads / 32) {
    const int64_t r = int64_t(b) * R + i;
    float v = -INFINITY;
    int k = INT_MAX;
    for (int cc = lane; cc < plan.chunks; cc += 32) {
      const float2 pp = __ldcg(part + r * plan.chunks + cc);
      argmax_take(v, k, pp.x, __float_as_int(pp.y));
    }
    warp_argmax(v, k);
    if (lane == 0) s_t[i] = k;
  }
  for (int j = threadIdx.x; j < T; j += kThreads) {
    const int x = tok[int64_t(b) * T + j], p = parent[int64_t(b) * T + j];
    const bool ok = x >= 0 && x < V && p >= -1 && p < j;  // parents come before their children
    if (!ok) atomicOr(err, kErrBadToken);
    s_tok[j] = ok ? x : -1;  // an invalid node never matches
    s_par[j] = ok ? p : -2;
  }
  __syncthreads();
  if (warp == 0) {
    // walk: lanes test the nodes in parallel; the ballot's lowest set bit is the lowest-index child
    int cur = -1, r = 0, depth = 0;
    for (;;) {
      const int t = s_t[r];
      int found = -1;
      for (int j0 = 0; j0 < T && found < 0; j0 += 32) {
        const int j = j0 + lane;
        const bool hit = j < T && s_par[j] == cur && s_tok[j] == t;
        const unsigned int m = __ballot_sync(0xFFFFFFFFu, hit);
        if (m) found = j0 + __ffs(m) - 1;
      }
      if (found < 0) break;
      if (lane == 0) {
        out_tok[int64_t(b) * R + depth] = s_tok[found];
        if (accept_nodes) accept_nodes[int64_t(b) * T + depth] = found;
      }
      ++depth;
      cur = found;
      r = found + 1;
    }
    if (lane == 0) {
      accept_len[b] = depth;
      out_tok[int64_t(b) * R + depth] = s_t[r];
      cnt[b] = 0;
    }
    for (int k = depth + 1 + lane; k < R; k += 32) out_tok[int64_t(b) * R + k] = -1;
    if (accept_nodes)
      for (int k = depth + lane; k < T; k += 32) accept_nodes[int64_t(b) * T + k] = -1;
  }
}

qspec_status check_verify_args(const void* tgt, const int32_t* d, int B, int gamma, int V,
                               const int32_t* accept_len, const int32_t* out_tok, void* ws,
                               size_t ws_bytes) {
  if (!tgt || !d || !accept_len || !out_tok) return QSPEC_ERR_INVALID_ARG;
  if (B <= 0 || gamma <= 0 || V <= 0) return QSPEC_ERR_INVALID_ARG;
  if (gamma > QSPEC_MAX_GAMMA || V < 2 || V > QSPEC_MAX_V ||
      int64_t(B) * (2 * gamma + 1) * int64_t(V) >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(tgt) || !aligned16(d) || !aligned16(accept_len) || !aligned16(out_tok))
    return QSPEC_ERR_MISALIGNED;
  if (!ws || !aligned16(ws)) return ws ? QSPEC_ERR_MISALIGNED : QSPEC_ERR_WORKSPACE;
  if (ws_bytes < layout(B, gamma, V).total) return QSPEC_ERR_WORKSPACE;
  return QSPEC_OK;
}

}  // namespace

unsigned int* verify_error_word(void* ws) { return static_cast<unsigned int*>(ws); }

}  // namespace qspec

using namespace qspec;

extern "C" size_t qspec_verify_workspace_size(int32_t B, int32_t gamma, int32_t V) {
  if (B <= 0 || gamma <= 0 || gamma > QSPEC_MAX_GAMMA || V < 2 || V > QSPEC_MAX_V) return 0;
  return layout(B, gamma, V).total;
}

extern "C" qspec_status qspec_verify_greedy(const uint16_t* tgt_logits, const int32_t* draft_tok,
                                            int32_t B, int32_t gamma, int32_t V,
                                            int32_t* accept_len, int32_t* out_tok,
                                            int32_t* tgt_argmax, void* ws, size_t ws_bytes,
                                            qspec_stream_t stream) {
  qspec_status st = check_verify_args(tgt_logits, draft_tok, B, gamma, V, accept_len, out_tok, ws, ws_bytes);
  if (st != QSPEC_OK) return st;
  if (tgt_argmax && !aligned16(tgt_argmax)) return QSPEC_ERR_MISALIGNED;
  const Layout L = layout(B, gamma, V);
  const WS w = bind(ws, L);
  const int64_t blocks = int64_t(B) * (gamma + 1) * L.pg.chunks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (V % 8 == 0)
    return launch_pdl(greedy_kernel<true>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, draft_tok,
                      int(gamma), int(V), L.pg, w, accept_len, out_tok, tgt_argmax);
  return launch_pdl(greedy_kernel<false>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, draft_tok,
                    int(gamma), int(V), L.pg, w, accept_len, out_tok, tgt_argmax);
}

namespace qspec {
namespace {
// CTAs of sampling pass 2 that are resident at once on this device (occupancy x SMs; looked up once
// per device ordinal, the kernels being the same in every context).
int pass2_resident_ctas() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_pass2_kernel<true>, kThreads, 0) != cudaSuccess ||
      per_sm <= 0)
    return 0;
  const int r = per_sm * num_sms();
  if (dev < 64) cached[dev] = r;
  return r;
}
}  // namespace
}  // namespace qspec

extern "C" qspec_status qspec_verify_sample(const uint16_t* tgt_logits, const uint16_t* draft_logits,
                                            const int32_t* draft_tok, const float* u_accept,
                                            const float* u_resample, int32_t B, int32_t gamma,
                                            int32_t V, int32_t* accept_len, int32_t* out_tok,
                                            float* accept_prob, float* p_tok, float* q_tok, void* ws,
                                            size_t ws_bytes, qspec_stream_t stream) {
  qspec_status st = check_verify_args(tgt_logits, draft_tok, B, gamma, V, accept_len, out_tok, ws, ws_bytes);
  if (st != QSPEC_OK) return st;
  if (!draft_logits || !u_accept || !u_resample) return QSPEC_ERR_INVALID_ARG;
  if (!aligned16(draft_logits) || !aligned16(u_accept) || !aligned16(u_resample) ||
      (accept_prob && !aligned16(accept_prob)) || (p_tok && !aligned16(p_tok)) || (q_tok && !aligned16(q_tok)))
    return QSPEC_ERR_MISALIGNED;
  const Layout L = layout(B, gamma, V);
  const WS w = bind(ws, L);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t blocks1 = int64_t(B) * (2 * gamma + 1) * L.p1.chunks;
  const bool vec = V % 8 == 0;
  const qspec_status st1 =
      vec ? launch_pdl(sample_pass1_kernel<true>, dim3(unsigned(blocks1)), dim3(kThreads), 0, s, tgt_logits,
                       draft_logits, draft_tok, u_accept, int(B), int(gamma), int(V), L.p1, w, accept_len, out_tok,
                       accept_prob, p_tok, q_tok)
          : launch_pdl(sample_pass1_kernel<false>, dim3(unsigned(blocks1)), dim3(kThreads), 0, s, tgt_logits,
                       draft_logits, draft_tok, u_accept, int(B), int(gamma), int(V), L.p1, w, accept_len, out_tok,
                       accept_prob, p_tok, q_tok);
  if (st1 != QSPEC_OK) return st1;

  // Pass 2 with programmatic dependent launch: its CTAs are scheduled while pass 1 drains and
  // wait (griddepcontrol.wait) for pass 1 to complete before reading the workspace.
  // One resident wave: as many CTAs per sequence as fit the GPU at once (each loops over its share of
  // the chunk groups), so no second wave waits behind the first one's latency chain.
  const int groups2 = (L.chunks2 + kPass2Chunks - 1) / kPass2Chunks;
  const int resident = pass2_resident_ctas();
  if (resident <= 0) return QSPEC_ERR_CUDA;
  const int per_seq = std::max(1, std::min(groups2, resident / int(B)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(int64_t(B) * per_seq));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (vec)
    e = cudaLaunchKernelEx(&cfg, sample_pass2_kernel<true>, tgt_logits, draft_logits, u_resample, int(B),
                           int(gamma), int(V), L.chunks2, per_seq, w, out_tok);
  else
    e = cudaLaunchKernelEx(&cfg, sample_pass2_kernel<false>, tgt_logits, draft_logits, u_resample, int(B),
                           int(gamma), int(V), L.chunks2, per_seq, w, out_tok);
  return e == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

extern "C" qspec_status qspec_verify_top1(const uint16_t* tgt_logits, const uint16_t* draft_logits, int32_t B,
                                          int32_t gamma, int32_t V, int32_t* tgt_top1, int32_t* draft_top1,
                                          float* tgt_p1, float* draft_p1, float high, double* tally,
                                          void* ws, size_t ws_bytes, qspec_stream_t stream) {
  if (!tgt_logits || !draft_logits || !tgt_top1 || !draft_top1) return QSPEC_ERR_INVALID_ARG;
  if (B <= 0 || gamma <= 0 || V <= 0) return QSPEC_ERR_INVALID_ARG;
  if (gamma > QSPEC_MAX_GAMMA || V < 2 || V > QSPEC_MAX_V ||
      int64_t(B) * (2 * gamma + 1) * int64_t(V) >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(tgt_logits) || !aligned16(draft_logits) || !aligned16(tgt_top1) || !aligned16(draft_top1) ||
      (tgt_p1 && !aligned16(tgt_p1)) || (draft_p1 && !aligned16(draft_p1)) || (tally && !aligned16(tally)))
    return QSPEC_ERR_MISALIGNED;
  if (!(high == high)) return QSPEC_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws)) return ws ? QSPEC_ERR_MISALIGNED : QSPEC_ERR_WORKSPACE;
  const Layout L = layout(B, gamma, V);
  if (ws_bytes < L.total) return QSPEC_ERR_WORKSPACE;
  const WS w = bind(ws, L);
  const int64_t blocks = int64_t(B) * (2 * gamma) * L.pt.chunks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (V % 8 == 0)
    return launch_pdl(top1_kernel<true>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, draft_logits,
                      int(B), int(gamma), int(V), L.pt, w, tgt_top1, draft_top1, tgt_p1, draft_p1, high, tally);
  return launch_pdl(top1_kernel<false>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, draft_logits,
                    int(B), int(gamma), int(V), L.pt, w, tgt_top1, draft_top1, tgt_p1, draft_p1, high, tally);
}

extern "C" size_t qspec_verify_tree_workspace_size(int32_t B, int32_t T, int32_t V) {
  if (B <= 0 || T <= 0 || T > QSPEC_MAX_TREE || V < 2 || V > QSPEC_MAX_V) return 0;
  return tree_layout(B, T, V).total;
}

extern "C" qspec_status qspec_verify_tree_greedy(const uint16_t* tgt_logits, const int32_t* tree_tok,
                                                 const int32_t* tree_parent, int32_t B, int32_t T, int32_t V,
                                                 int32_t* accept_len, int32_t* out_tok, int32_t* accept_nodes,
                                                 void* ws, size_t ws_bytes, qspec_stream_t stream) {
  if (!tgt_logits || !tree_tok || !tree_parent || !accept_len || !out_tok) return QSPEC_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || V <= 0) return QSPEC_ERR_INVALID_ARG;
  if (T > QSPEC_MAX_TREE || V < 2 || V > QSPEC_MAX_V || int64_t(B) * (T + 1) * int64_t(V) >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(tgt_logits) || !aligned16(tree_tok) || !aligned16(tree_parent) || !aligned16(accept_len) ||
      !aligned16(out_tok) || (accept_nodes && !aligned16(accept_nodes)))
    return QSPEC_ERR_MISALIGNED;
  if (!ws || !aligned16(ws)) return ws ? QSPEC_ERR_MISALIGNED : QSPEC_ERR_WORKSPACE;
  const TreeLayout L = tree_layout(B, T, V);
  if (ws_bytes < L.total) return QSPEC_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  unsigned int* err = reinterpret_cast<unsigned int*>(w + L.err);
  unsigned int* cnt = reinterpret_cast<unsigned int*>(w + L.cnt);
  float2* part = reinterpret_cast<float2*>(w + L.part);
  const int64_t blocks = int64_t(B) * (T + 1) * L.p.chunks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (V % 8 == 0)
    return launch_pdl(tree_kernel<true>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, tree_tok,
                      tree_parent, int(T), int(V), L.p, err, cnt, part, accept_len, out_tok, accept_nodes);
  return launch_pdl(tree_kernel<false>, dim3(unsigned(blocks)), dim3(kThreads), 0, s, tgt_logits, tree_tok,
                    tree_parent, int(T), int(V), L.p, err, cnt, part, accept_len, out_tok, accept_nodes);
}

// ------------------------------------------------------------------ allocation-free greedy verify
//
// Some callers cannot allocate device memory at the point where they verify: plug-ins that execute
// inside another runtime's fixed memory plan (a serving engine that forbids allocation during a
// decode step), or plain C hosts without access to an allocator.  For them,
// qspec_verify_greedy_noalloc uses scratch memory that lives inside this library: a fixed array of
// device memory that every GPU loading the library holds until exit.  The pages have no counterpart
// of this; it is a deployment convenience only.

namespace {

constexpr size_t kNoAllocScratchBytes = QSPEC_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address belongs to the copy of this module loaded in one CUDA context, so the
// cache is keyed on the context's process-unique id (a context created after another was destroyed,
// e.g. after cudaDeviceReset, gets a new id, never a stale address).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

CtxFns ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

// Id of the context current on this thread; false if none is current or the driver cannot say.
bool current_ctx_id(unsigned long long* id) {
  const CtxFns f = ctx_fns();
  CUcontext ctx = nullptr;
  if (!f.get_current || !f.get_id || f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kNoAllocCacheSlots = 64;
std::mutex g_noalloc_mu;
unsigned long long g_noalloc_ctx[kNoAllocCacheSlots] = {};
void* g_noalloc_ptr[kNoAllocCacheSlots] = {};
int g_noalloc_used = 0;

// Device address of the scratch array in the current context.  cudaGetSymbolAddress runs once per
// context (normally once per device, in its primary context), with that context current, on the
// first call made there; later calls in that context take the cached address.
qspec_status noalloc_scratch(void** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = 0;
  bool have_id = current_ctx_id(&id);
  if (have_id) {
    for (int i = 0; i < g_noalloc_used; ++i)
      if (g_noalloc_ctx[i] == id) {
        *out = g_noalloc_ptr[i];
        return QSPEC_OK;
      }
  }
  // (the lookup also initialises the runtime's context on this thread's device if none was current)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QSPEC_ERR_CUDA;
  if (!have_id) have_id = current_ctx_id(&id);
  if (have_id && g_noalloc_used < kNoAllocCacheSlots) {  // (a full table only skips the caching)
    g_noalloc_ctx[g_noalloc_used] = id;
    g_noalloc_ptr[g_noalloc_used] = p;
    ++g_noalloc_used;
  }
  *out = p;
  return QSPEC_OK;
}

}  // namespace

extern "C" qspec_status qspec_verify_greedy_noalloc(const uint16_t* tgt_logits, const int32_t* draft_tok,
                                                    int32_t B, int32_t gamma, int32_t V,
                                                    int32_t* accept_len, int32_t* out_tok,
                                                    int32_t* tgt_argmax, qspec_stream_t stream) {
  if (!tgt_logits || !draft_tok || !accept_len || !out_tok) return QSPEC_ERR_INVALID_ARG;
  if (B <= 0 || gamma <= 0 || V <= 0) return QSPEC_ERR_INVALID_ARG;
  if (gamma > QSPEC_MAX_GAMMA || V < 2 || V > QSPEC_MAX_V ||
      int64_t(B) * (gamma + 1) * int64_t(V) >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(tgt_logits) || !aligned16(draft_tok) || !aligned16(accept_len) || !aligned16(out_tok) ||
      (tgt_argmax && !aligned16(tgt_argmax)))
    return QSPEC_ERR_MISALIGNED;
  // compact layout: error word, per-sequence tickets, per-(row, chunk) partial argmaxes
  const Plan plan = plan_rows(int64_t(B) * (gamma + 1), V);
  const size_t off_cnt = 256;
  const size_t off_part = align256(off_cnt + sizeof(unsigned int) * size_t(B));
  const size_t need = off_part + sizeof(float2) * size_t(B) * (gamma + 1) * plan.chunks;
  if (need > kNoAllocScratchBytes) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  void* base = nullptr;
  const qspec_status st = noalloc_scratch(&base);
  if (st != QSPEC_OK) return st;
  char* p = static_cast<char*>(base);
  WS w{};
  w.err = reinterpret_cast<unsigned int*>(p);
  w.cnt1 = reinterpret_cast<unsigned int*>(p + off_cnt);
  w.part1 = reinterpret_cast<float2*>(p + off_part);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the error word and the tickets must start at 0
  if (cudaMemsetAsync(p, 0, off_part, s) != cudaSuccess) return QSPEC_ERR_CUDA;
  const int64_t blocks = int64_t(B) * (gamma + 1) * plan.chunks;
  if (V % 8 == 0)
    greedy_kernel<true><<<unsigned(blocks), kThreads, 0, s>>>(tgt_logits, draft_tok, gamma, V, plan, w,
                                                              accept_len, out_tok, tgt_argmax);
  else
    greedy_kernel<false><<<unsigned(blocks), kThreads, 0, s>>>(tgt_logits, draft_tok, gamma, V, plan, w,
                                                               accept_len, out_tok, tgt_argmax);
  return launch_status();
}
