// Tensor-core (tcgen05) W4A16 linear for token counts beyond the GEMV's: the weights are
// dequantised on chip, and the accumulators of J weight tiles stay in TMEM for the whole K range of
// a work item.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": the W4A16 mode turns each 4-bit weight back into a 16-bit value (its code
// times its group's scale) while multiplying the 16-bit activations; section "QSpec の W4A4 モードと
// W4A16 モード": both modes read the same packed weights.
//
// Design (one CTA per SM, persistent):
//  * D[n, m] = sum_k W[n, k] x[m, k], computed transposed: 128 weight rows are the MMA's M side and
//    NM tokens (128 or 256) its N side; tcgen05.mma.cta_group::1.kind::f16 with fp16 operands and
//    fp32 accumulators in TMEM.
//  * A operand: eight converter warps turn the packed codes of a 128-row x 64-channel block into
//    fp16(code * s[n, g]) -- the exact code times the fp16 group scale, rounded once -- and store
//    the tile in TMEM (tcgen05.st), from where the MMA reads it.  (Kept in shared memory instead,
//    the MMA's operand reads, the TMA writes and the converters' stores together held the N = 256
//    MMAs to about half the tensor-core rate.)
//  * B operand: the activations in fp16, converted once per call (tokens_f16_kernel) with one
//    power-of-two factor per token, which is exact; TMA loads them with the 128-byte swizzle and the
//    epilogue multiplies the factor back.
//  * A work item is J consecutive 128-row tiles x NM tokens.  Its J accumulators stay in TMEM over
//    all of K, so an activation block is loaded once for J weight tiles; where TMEM allows, two
//    accumulator sets let the next item's MMAs run while the last one drains.
//  * Schedule: every CTA first takes whole items (the same number each), then an equal contiguous
//    share of the units (item, 64-channel block) of the items left over.  An item cut between CTAs
//    is finished by its last contributor (atomic ticket), which adds every contributor's partial
//    sums in CTA order, so the result does not depend on timing.
//  * Shared-memory rings: weight stages (J boxes of 128 rows x 256 channels -- 128 bytes a row;
//    TMA streams boxes 32 bytes wide at a fraction of the HBM rate) and activation blocks (NM
//    tokens x 64 channels); a TMEM ring of dequantised tiles.
//  * Warp roles: warp 0 loads the activation blocks; warp 1 loads each weight stage and stages its
//    group scales;
//    warps 2 .. J + 1 issue the MMAs of one tile each; eight converter warps dequantise; four
//    epilogue warps drain finished items.  Stages are handed over with mbarriers; every wait is
//    bounded, after which the CTA finishes in abort mode (no more work, in-flight copies waited for,
//    TMEM freed) and sets the timeout error bit.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "linear_internal.h"
#include "tc_ptx.cuh"

namespace qspec {
namespace dq {
using namespace ptx;

constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;  // one per TMEM lane quarter
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kFirstIssuer = 2;
constexpr int kQuad = 4;              // 64-channel blocks per weight stage (256 channels, 128 bytes a row)
constexpr int kWTile = 128 * 128;     // packed weights of one 128-row tile x 256 channels
constexpr int kSmemMax = 232448;      // dynamic shared memory one CTA may opt into
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s) before a wait gives up

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int ws_bad;
  int last;
};

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
// Accumulator sets in TMEM: two when they fit beside at least two units' dequantised tiles (32
// columns each).
__host__ __device__ constexpr int acc_sets(int NM, int J) { return 2 * J * NM + 2 * J * 32 <= 512 ? 2 : 1; }
// Ring depths: weight stages (J x 16.5 KB each: codes and scales), activation blocks (NM x 128 bytes
// each) and dequantised tiles (TMEM, the columns the accumulators leave).
struct RingCfg {
  int nw, nb, nat;
};
__host__ __device__ constexpr int w_stage_bytes(int J) { return J * (kWTile + 2 * 128 * 2); }
__host__ __device__ constexpr int nw_of(int J) { return cmax(2, cmin(8, (130 * 1024) / w_stage_bytes(J))); }
__host__ __device__ constexpr RingCfg ring_cfg(int NM, int J) {
  return RingCfg{nw_of(J), cmin(8, (220 * 1024 - nw_of(J) * w_stage_bytes(J)) / (NM * 128)),
                 cmin(16, (512 - acc_sets(NM, J) * J * NM) / 32)};
}
__host__ __device__ constexpr int first_conv(int J) { return kFirstIssuer + J; }
__host__ __device__ constexpr int first_epi(int J) { return kFirstIssuer + J + kConvWarps; }
__host__ __device__ constexpr int threads_of(int J) { return (first_epi(J) + kEpiWarps) * 32; }
__host__ __device__ constexpr int smem_of(int NM, int J) {
  return 1024 /* alignment slack */ + ring_cfg(NM, J).nw * w_stage_bytes(J) + ring_cfg(NM, J).nb * NM * 128 +
         (3 * ring_cfg(NM, J).nw + 2 * ring_cfg(NM, J).nb + 2 * ring_cfg(NM, J).nat + 5) * 8 +
         static_cast<int>(sizeof(Misc)) + 64;
}

struct DqArgs {
  int M, N, K, KB, T_m;
  uint32_t dp_items;      // whole items per CTA, taken first
  uint32_t sk_beg, sk_units;  // the units shared out afterwards: [sk_beg, sk_beg + sk_units)
  uint16_t* y;
  const __half* S;
  const float* pw;        // per-token power-of-two factors
  float* partial;         // [gridDim.x][2][NM][128 J]
  unsigned int* ticket;   // [items]
  unsigned int* err;      // the linear error word
  WsGuard guard;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimit) {
      *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// Ignores the abort flag (lets in-flight copies land before exit); bounded.
__device__ __forceinline__ void wait_bar_final(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimit) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// One CTA's units in order: its whole items [r1_beg, r1_end), then its share [r2_beg, r2_end) of the
// rest; a unit is one 64-channel block of one item.  A weight stage holds the (up to) four blocks of
// one 256-channel quad of an item that a range covers.
struct UnitIter {
  uint32_t u, seg_beg, seg_end, r2_beg, r2_end, KB, item, kb;
  bool in_r2;
  uint32_t cur_item, cur_kb, cur_seg_beg, cur_seg_end;
  bool cur_first, cur_last;  // first / last unit of cur_item within its range
  bool cur_wnew, cur_wlast;  // first / last unit of its weight stage
  __device__ UnitIter(uint32_t r1b, uint32_t r1e, uint32_t r2b, uint32_t r2e, uint32_t KB_)
      : u(r1b), seg_beg(r1b), seg_end(r1e), r2_beg(r2b), r2_end(r2e), KB(KB_), in_r2(false) {
    item = r1b / KB_;
    kb = r1b - item * KB_;
  }
  __device__ bool next() {
    if (u >= seg_end) {
      if (in_r2 || r2_beg >= r2_end) return false;
      in_r2 = true;
      u = seg_beg = r2_beg;
      seg_end = r2_end;
      item = u / KB;
      kb = u - item * KB;
    }
    cur_item = item;
    cur_kb = kb;
    cur_seg_beg = seg_beg;
    cur_seg_end = seg_end;
    cur_first = u == seg_beg || kb == 0;
    cur_last = u + 1 == seg_end || kb + 1 == KB;
    cur_wnew = u == seg_beg || (kb & (kQuad - 1)) == 0;
    cur_wlast = cur_last || (kb & (kQuad - 1)) == kQuad - 1;
    ++u;
    if (++kb == KB) {
      kb = 0;
      ++item;
    }
    return true;
  }
};

// The CTA whose share of the leftover units holds unit v (counted from the start of that region).
__device__ __forceinline__ uint32_t owner_of(uint32_t v, uint32_t R, uint32_t P) {
  return static_cast<uint32_t>(((static_cast<uint64_t>(v) + 1) * P - 1) / R);
}

// One packed word (channels k0..k7 of a row as two's complement nibbles in the order k0, k2, k4, k6,
// k1, k3, k5, k7) -> four fp16x2 words (k0,k1) .. (k6,k7) of code * s.  Nibble pair (i, i + 4) goes
// to bits 0..3 / 16..19 with its top bit flipped, under the exponent of fp16 1024: exactly 1032 +
// code; subtracting 1032 is exact, the product with s is rounded once.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, uint32_t* out) {
  const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x64086408u));
    const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&v), off);
    const __half2 p = __hmul2(c, s2);
    out[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
}

template <int NM, int J>
__global__ void __launch_bounds__(threads_of(J), 1)
    linear_dq_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const DqArgs a) {
  constexpr RingCfg R = ring_cfg(NM, J);
  constexpr int NW = R.nw, NB = R.nb, NAT = R.nat;
  constexpr int DB = acc_sets(NM, J);
  constexpr int WS = J * kWTile;  // one weight stage
  constexpr int BS = NM * 128;    // one activation block
  constexpr int BN = 128 * J;
  constexpr uint32_t kACol = static_cast<uint32_t>(DB * J * NM);  // first TMEM column of the A tiles
  constexpr uint32_t kCols = 512;
  static_assert(smem_of(NM, J) <= kSmemMax, "shared memory");
  static_assert(NW >= 2 && NB >= 2 && DB * J * NM <= 512, "configuration");
  static_assert(NAT >= 2 * J && kACol + 32 * NAT <= 512, "TMEM tiles");
  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned tiles (alignment of the shared-window offset)
  uint8_t* wring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* bring = wring + NW * WS;
  __half* sc = reinterpret_cast<__half*>(bring + NB * BS);  // [NW][J][2 groups][128 rows]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(sc + NW * J * 256);  // weight bytes of a stage landed
  uint64_t* sfull = wfull + NW;                                     // its scales staged
  uint64_t* wempty = sfull + NW;                                    // converters done with it
  uint64_t* bfull = wempty + NW;
  uint64_t* bempty = bfull + NB;
  uint64_t* afull = bempty + NB;
  uint64_t* afree = afull + NAT;
  uint64_t* dfull = afree + NAT;  // [DB]
  uint64_t* dfree = dfull + 2;    // [DB]
  uint64_t* done = dfree + 2;
  Misc* misc = reinterpret_cast<Misc*>(done + 1);
  volatile int* abort_flag = &misc->abort_flag;
  unsigned int* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(sfull + i, 1);
      mbar_init(wempty + i, kConvWarps);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(bfull + i, 1);
      mbar_init(bempty + i, J);
    }
    for (int i = 0; i < NAT; ++i) {
      mbar_init(afull + i, kConvWarps);
      mbar_init(afree + i, 1);
    }
    for (int i = 0; i < DB; ++i) {
      mbar_init(dfull + i, J);
      mbar_init(dfree + i, kEpiWarps);
    }
    mbar_init(done, J);
    misc->abort_flag = 0;
    misc->last = 0;
    // the workspace must hold this shape's layout (or none yet); the header only ever goes from 0
    // to a tag, so the claim may run before the dependency wait
    misc->ws_bad = ws_claim(a.guard) ? 0 : 1;
    fence_mbar_init();
  }
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmX);
    }
    tmem_alloc(&misc->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  if (misc->ws_bad) {  // (uniform over the CTA)
    if (warp == 0) tmem_dealloc(tmem, kCols);
    return;
  }

  grid_launch_dependents();
  grid_dependency_wait();

  const uint32_t P = gridDim.x, c = blockIdx.x;
  const uint32_t KB = static_cast<uint32_t>(a.KB), T_m = static_cast<uint32_t>(a.T_m);
  const uint32_t r1_beg = c * a.dp_items * KB, r1_end = (c + 1) * a.dp_items * KB;
  const uint32_t r2_beg = a.sk_beg + static_cast<uint32_t>(static_cast<uint64_t>(c) * a.sk_units / P);
  const uint32_t r2_end = a.sk_beg + static_cast<uint32_t>(static_cast<uint64_t>(c + 1) * a.sk_units / P);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      fence_proxy_async_global();  // the activations were written by the previous kernel
      UnitIter it(r1_beg, r1_end, r2_beg, r2_end, KB);
      int s = 0;
      while (it.next()) {
        const int b = s % NB;
        if (s >= NB) wait_bar(bempty + b, ((s / NB) - 1) & 1, abort_flag, err);
        if (*abort_flag) break;
        mbar_arrive_expect_tx(bfull + b, BS);
        tma_load_2d(bring + b * BS, &tmX, bfull + b, static_cast<int>(it.cur_kb) * 64,
                    static_cast<int>(it.cur_item % T_m) * NM);
        ++s;
      }
      // nothing may still be copying into shared memory when the CTA exits
      for (int t = (s > NB ? s - NB : 0); t < s; ++t) wait_bar_final(bfull + t % NB, (t / NB) & 1, err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ weight stages
    // Lane 0 issues each stage's weight TMA loads as soon as its slot is free (independently of the
    // activation blocks); lane l stages the group scales of rows 4l .. 4l + 3 of every tile, both
    // groups of the stage's quad.  The next stage's scale loads are in flight while the current one
    // waits for its slot and is stored.
    const int G = a.K / kGroup;
    UnitIter it(r1_beg, r1_end, r2_beg, r2_end, KB);
    int n0s[2] = {0, 0}, xs[2] = {0, 0};  // TMA coordinates of the fetched stages
    auto fetch = [&](__half (&v)[J][4][2], int slot) -> bool {
      bool found = false;
      while (!found && it.next()) found = it.cur_wnew;
      if (!found) return false;
      const int n0 = static_cast<int>(it.cur_item / T_m) * BN;
      const int g0 = static_cast<int>(it.cur_kb / kQuad) * 2;
      n0s[slot] = n0;
      xs[slot] = static_cast<int>(it.cur_kb / kQuad) * 128;
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = n0 + j * 128 + 4 * lane + i;
          const __half* srow = a.S + static_cast<long long>(n) * G;
          v[j][i][0] = n < a.N ? __ldg(srow + g0) : __ushort_as_half(0);
          v[j][i][1] = n < a.N && g0 + 1 < G ? __ldg(srow + g0 + 1) : __ushort_as_half(0);
        }
      return true;
    };
    __half va[J][4][2], vb[J][4][2];
    int ws = 0;
    int issued = 0;
    auto store = [&](const __half (&v)[J][4][2], int slot) {
      const int w = ws % NW;
      bool ok = true;
      if (ws >= NW) ok = wait_bar(wempty + w, ((ws / NW) - 1) & 1, abort_flag, err);
      if (lane == 0 && ok && !*abort_flag) {
        mbar_arrive_expect_tx(wfull + w, WS);
#pragma unroll
        for (int j = 0; j < J; ++j) tma_load_2d(wring + w * WS + j * kWTile, &tmW, wfull + w, xs[slot], n0s[slot] + j * 128);
        ++issued;
      }
      if (ok && !*abort_flag) {
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sc[((w * J + j) * 2 + 0) * 128 + 4 * lane + i] = v[j][i][0];
            sc[((w * J + j) * 2 + 1) * 128 + 4 * lane + i] = v[j][i][1];
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sfull + w);
      ++ws;
    };
    bool have_a = fetch(va, 0);
    while (have_a) {
      const bool have_b = fetch(vb, 1);
      store(va, 0);
      if (!have_b) break;
      have_a = fetch(va, 0);
      store(vb, 1);
    }
    // nothing may still be copying into shared memory when the CTA exits (stages issued in order)
    if (lane == 0)
      for (int t = (issued > NW ? issued - NW : 0); t < issued; ++t) wait_bar_final(wfull + t % NW, (t / NW) & 1, err);
  } else if (warp < first_conv(J)) {
    // ------------------------------------------------------------------ MMA issuer of tile j
    const int j = warp - kFirstIssuer;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, NM);
      UnitIter it(r1_beg, r1_end, r2_beg, r2_end, KB);
      int s = 0, item_i = 0;
      while (it.next()) {
        const int b = s % NB;
        const int ax = s * J + j, x = ax % NAT;
        const int db = item_i % DB;  // accumulator set of this item
        bool ok = wait_bar(bfull + b, (s / NB) & 1, abort_flag, err);
        ok = wait_bar(afull + x, (ax / NAT) & 1, abort_flag, err) && ok;
        if (it.cur_first && item_i >= DB) ok = wait_bar(dfree + db, ((item_i / DB) - 1) & 1, abort_flag, err) && ok;
        if (ok && !*abort_flag) {
          tc_fence_after();
          const uint32_t b_addr = smem_u32(bring + b * BS);
          const uint32_t d = tmem + static_cast<uint32_t>((db * J + j) * NM);
          const uint32_t a_col = tmem + kACol + static_cast<uint32_t>(x * 32);  // 8 columns per K step
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(d, a_col + kk * 8, smem_desc_sw128(b_addr + kk * 32), idesc,
                        (it.cur_first && kk == 0) ? 0u : 1u);
        }
        mma_commit(afree + x);
        mma_commit(bempty + b);
        if (it.cur_last) {
          mma_commit(dfull + db);
          ++item_i;
        }
        ++s;
      }
      mma_commit(done);
      wait_bar_final(done, 0, err);
    }
  } else if (warp < first_epi(J)) {
    // ------------------------------------------------------------------ converters
    const int cw = warp - first_conv(J);  // 0 .. 7
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // the row of the tile (a warp's rows are its TMEM lane quarter, which tcgen05.st requires) and
    // the 32-channel half of the 64-channel block this thread converts
    const int row = q * 32 + lane;
    const int hh = cw >> 2;
    UnitIter it(r1_beg, r1_end, r2_beg, r2_end, KB);
    int s = 0, ws = 0, w = 0;
    bool okw = true;
    while (it.next()) {
      if (it.cur_wnew) {
        w = ws % NW;
        okw = wait_bar(wfull + w, (ws / NW) & 1, abort_flag, err);
        okw = wait_bar(sfull + w, (ws / NW) & 1, abort_flag, err) && okw;
      }
      const int kq = static_cast<int>(it.cur_kb & (kQuad - 1));
      const int chunk = 2 * kq + hh;  // the row's 16-byte chunk holding this thread's 32 channels
      const uint8_t* wsrc = wring + w * WS + row * 128 + ((chunk ^ (row & 7)) << 4);
      const __half* ssrc = sc + (w * J * 2 + (kq >> 1)) * 128 + row;
      // all J tiles of the unit at once: one wait for their TMEM stores, one hand-over
      bool oku = okw;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int ax = s * J + j;
        if (ax >= NAT) oku = wait_bar(afree + ax % NAT, ((ax / NAT) - 1) & 1, abort_flag, err) && oku;
      }
      if (oku && !*abort_flag) {
        uint4 w4[J];
        __half2 s2[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
          w4[j] = *reinterpret_cast<const uint4*>(wsrc + j * kWTile);
          s2[j] = __half2half2(ssrc[j * 256]);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
          uint32_t o[16];
          dequant_word(w4[j].x, s2[j], o);
          dequant_word(w4[j].y, s2[j], o + 4);
          dequant_word(w4[j].z, s2[j], o + 8);
          dequant_word(w4[j].w, s2[j], o + 12);
          const int x = (s * J + j) % NAT;
          tmem_st16(tmem + lane_base + kACol + static_cast<uint32_t>(x * 32 + hh * 16), o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < J; ++j) mbar_arrive(afull + (s * J + j) % NAT);
      }
      if (it.cur_wlast) {
        __syncwarp();
        if (lane == 0) mbar_arrive(wempty + w);
        ++ws;
      }
      ++s;
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int et = (warp - first_epi(J)) * 32 + lane;  // 0 .. 127
    const int q = warp & 3;                             // TMEM lane quarter: rows 32 q .. 32 q + 31
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int M = a.M, N = a.N;
    const uint32_t R2 = a.sk_units;
    auto store_y = [&](int n, int m0, const float* v) {
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int m = m0 + t;
        if (m < M && n < N) a.y[static_cast<long long>(m) * N + n] = f32_to_bf16_bits(v[t] * __ldg(a.pw + m));
      }
    };
    UnitIter it(r1_beg, r1_end, r2_beg, r2_end, KB);
    int item_i = 0;
    while (it.next()) {
      if (!it.cur_last) continue;
      const uint32_t item = it.cur_item;
      const int db = item_i % DB;
      const bool ok = wait_bar(dfull + db, (item_i / DB) & 1, abort_flag, err);
      ++item_i;
      tc_fence_after();
      const int n0 = static_cast<int>(item / T_m) * BN;
      const int mt0 = static_cast<int>(item % T_m) * NM;
      const bool whole = item * KB >= it.cur_seg_beg && (item + 1) * KB <= it.cur_seg_end;
      const int slot = item == it.cur_seg_beg / KB ? 0 : 1;  // (a split item lies in the shared range)
      float* pt = a.partial + (static_cast<size_t>(c) * 2 + slot) * (BN * NM);
#pragma unroll 1
      for (int j = 0; j < J; ++j) {
        const int rr = j * 128 + q * 32 + lane;  // row within the item
#pragma unroll 1
        for (int col = 0; col < NM; col += 16) {
          float v[16];
          uint32_t raw[16];
          if (ok) {
            tmem_ld16(tmem + lane_base + static_cast<uint32_t>((db * J + j) * NM + col), raw);
            tmem_wait_ld();
          }
#pragma unroll
          for (int t = 0; t < 16; ++t) v[t] = ok ? __uint_as_float(raw[t]) : 0.0f;
          if (whole) {
            if (ok && !*abort_flag) store_y(n0 + rr, mt0 + col, v);
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) pt[(col + t) * BN + rr] = v[t];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dfree + db);
      if (whole) continue;
      // a split item: publish, take a ticket, and the last contributor adds all partials in CTA order
      const uint32_t c_first = owner_of(item * KB - a.sk_beg, R2, P);
      const uint32_t c_last = owner_of((item + 1) * KB - 1 - a.sk_beg, R2, P);
      __threadfence();
      named_bar_sync(1, kEpiThreads);
      if (et == 0) {
        const unsigned int prev = atomicAdd(a.ticket + item, 1u);
        misc->last = prev == c_last - c_first;
      }
      named_bar_sync(1, kEpiThreads);
      if (!misc->last) continue;
      __threadfence();
      // contributor c_first may have begun in an earlier item (this item is then its slot 1); every
      // later contributor begins inside this item (slot 0)
      const uint32_t first_beg = a.sk_beg + static_cast<uint32_t>(static_cast<uint64_t>(c_first) * R2 / P);
      const uint32_t first_slot = first_beg / KB == item ? 0u : 1u;
      // The partial tiles ([column][row] fp32) are summed as a stream of float4 (four rows of one
      // column) in CTA order; each thread has kU4 float4 of up to kCg contributors in flight, and
      // four outputs go out as one 8-byte store.
      constexpr int E4 = BN * NM / 4;
      constexpr int kU4 = 4, kCg = 4;
      const float4* p4 = reinterpret_cast<const float4*>(a.partial);
#pragma unroll 1
      for (int e0 = et; e0 < E4; e0 += kEpiThreads * kU4) {
        float4 acc[kU4];
#pragma unroll
        for (int u = 0; u < kU4; ++u) acc[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
        for (uint32_t c0 = c_first; c0 <= c_last; c0 += kCg) {
          float4 v[kCg][kU4];
#pragma unroll
          for (int g = 0; g < kCg; ++g) {
            const uint32_t cp = c0 + g;
            const uint32_t sl = cp == c_first ? first_slot : 0u;
            const float4* src = p4 + (static_cast<size_t>(cp) * 2 + sl) * E4;
#pragma unroll
            for (int u = 0; u < kU4; ++u) {
              const int e = e0 + u * kEpiThreads;
              v[g][u] = cp <= c_last && e < E4 ? __ldcg(src + e) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
          }
#pragma unroll
          for (int g = 0; g < kCg; ++g)  // in CTA order (absent contributors add zeros)
#pragma unroll
            for (int u = 0; u < kU4; ++u) {
              acc[u].x += v[g][u].x;
              acc[u].y += v[g][u].y;
              acc[u].z += v[g][u].z;
              acc[u].w += v[g][u].w;
            }
        }
        if (*abort_flag) continue;
#pragma unroll
        for (int u = 0; u < kU4; ++u) {
          const int e = e0 + u * kEpiThreads;
          if (e >= E4) continue;
          const int col = (e * 4) / BN, r = (e * 4) % BN;
          const int m = mt0 + col, n = n0 + r;
          if (m >= M || n >= N) continue;  // N is a multiple of 8, so n < N covers n .. n + 3
          const float f = __ldg(a.pw + m);
          const uint32_t lo = static_cast<uint32_t>(f32_to_bf16_bits(acc[u].x * f)) |
                              (static_cast<uint32_t>(f32_to_bf16_bits(acc[u].y * f)) << 16);
          const uint32_t hi = static_cast<uint32_t>(f32_to_bf16_bits(acc[u].z * f)) |
                              (static_cast<uint32_t>(f32_to_bf16_bits(acc[u].w * f)) << 16);
          *reinterpret_cast<uint2*>(a.y + static_cast<long long>(m) * N + n) = make_uint2(lo, hi);
        }
      }
      if (et == 0) a.ticket[item] = 0;
    }
  }
  // Lane 0 of the producer and issuer warps ran its role alone; reconverge every warp before the
  // CTA barrier, so TMEM is released only after every warp has finished with it.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <int NM, int J>
qspec_status launch(const CUtensorMap& tmW, const CUtensorMap& tmX, const DqArgs& args, int P, cudaStream_t stream) {
  auto kern = linear_dq_kernel<NM, J>;
  constexpr int smem = smem_of(NM, J);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return QSPEC_ERR_CUDA;
  return launch_pdl(kern, dim3(P), dim3(threads_of(J)), smem, stream, tmW, tmX, args);
}

}  // namespace dq

// Launches the instantiated kernels: NM = 128 with J = 1 or 2, NM = 256 with J = 1.
qspec_status dq_launch(int NM, int J, const CUtensorMap& tmW, const CUtensorMap& tmX, const dq::DqArgs& args, int P,
                       cudaStream_t stream);

}  // namespace qspec
