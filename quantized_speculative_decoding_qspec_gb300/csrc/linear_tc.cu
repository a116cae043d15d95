// Tensor-core (tcgen05) path of the W4A16 / W4A4 linears over the shared packed INT4 weights.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": W4A16 converts the 4-bit weights while multiplying 16-bit activations;
// W4A4 also quantises the activations to 4 bits (one fp32 scale per token here).  Section
// "QSpec の W4A4 モードと W4A16 モード": both modes read the same 4-bit weights.
//
// Design (one GB300 SM per CTA, persistent):
//  * The product is computed transposed, D[n, m] = sum_k W[n, k] x[m, k]: 128 weight rows form the
//    MMA's M = 128 side, the tokens (padded to NM = 16..64) its N side, so decode-sized M still
//    fills the tensor core.
//  * Work is split "stream-K": the (tile, 128-channel group) units of the whole problem are cut
//    into gridDim.x equal contiguous ranges, so every SM streams the same number of weight bytes.
//    A tile whose groups span several CTAs is finished by the last contributor (atomic ticket, no
//    spinning), which adds the partial sums in CTA order -- the result does not depend on timing.
//  * Warp roles: warp 0 issues TMA loads (packed weights, 128 rows x 256 channels per stage, and
//    the activation tile); warp 1 owns TMEM and issues tcgen05.mma; warp 2 stages the fp16 group
//    scales; warps 3..10 convert INT4 codes to bf16 (exact) straight into TMEM, where they are the
//    MMA's A operand, and drain the fp32 accumulator of every 128-channel group, scaling it by
//    s[n, g].  Stages are handed over with mbarriers; every wait is bounded.
//  * W4A4: the INT4 activation codes are carried as bf16 (exact), so both modes share one MMA
//    type; products and 128-term group sums are small integers, exact in the fp32 accumulator.
//    For M <= 4 the per-token quantiser is fused (each CTA computes the token amax itself and
//    converts the activation tile in shared memory); for larger M a small kernel quantises once
//    and the GEMM reads the codes.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "linear_internal.h"
#include "tc_ptx.cuh"

namespace qspec {

// Error bits of the linear kernels (read and cleared by qspec_check_status): kErrTimeout when a
// kernel gave up a bounded wait, kErrWorkspace when a workspace held another shape's layout.
__device__ unsigned int g_linear_error = 0;

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::mutex g_err_mu;
constexpr int kErrSlots = 64;
unsigned long long g_err_ctx[kErrSlots] = {};
unsigned int* g_err_ptr[kErrSlots] = {};
int g_err_used = 0;

bool ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

// The error word's address belongs to the module copy of one CUDA context: cached per context id
// (process-unique, so a context created after another was destroyed never sees a stale address).
unsigned int* linear_error_word() {
  std::lock_guard<std::mutex> lock(g_err_mu);
  unsigned long long id = 0;
  bool have_id = ctx_id(&id);
  if (have_id)
    for (int i = 0; i < g_err_used; ++i)
      if (g_err_ctx[i] == id) return g_err_ptr[i];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_linear_error) != cudaSuccess) return nullptr;
  if (!have_id) have_id = ctx_id(&id);
  if (have_id && g_err_used < kErrSlots) {
    g_err_ctx[g_err_used] = id;
    g_err_ptr[g_err_used] = static_cast<unsigned int*>(p);
    ++g_err_used;
  }
  return static_cast<unsigned int*>(p);
}

namespace {

using namespace ptx;

constexpr int kWorkerWarps = 8;
constexpr int kFirstWorker = 3;
constexpr int kFirstExtraIssuer = kFirstWorker + kWorkerWarps;
// Accumulator chains per 128-channel group: a stage's MMAs are spread over 2 * chains issuing
// warps with separate TMEM accumulators (one thread issuing back-to-back MMAs is latency-bound at
// these narrow N); the drain adds the chains.  TMEM: 256 columns of A + 2 x 2 x chains x NM of D.
__host__ __device__ constexpr int tc_chains(int NM) { return NM * 2 <= 64 ? 2 : 1; }
__host__ __device__ constexpr int tc_issuers(int NM) { return 2 * tc_chains(NM); }
__host__ __device__ constexpr int tc_threads(int NM) { return (kFirstExtraIssuer + tc_issuers(NM) - 1) * 32; }
constexpr int kWBytes = 128 * 128;           // one stage of packed weights: 128 rows x 256 channels
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s) before a wait gives up
constexpr int kFusedMaxM = 4;

enum Mode : int { kA16 = 0, kA4Fused = 1, kA4Codes = 2 };

__host__ __device__ constexpr int b_bytes(int NM) { return NM * 128 * 4; }  // 4 boxes of NM x 64 bf16
__host__ __device__ constexpr int stage_bytes(int NM) { return kWBytes + b_bytes(NM); }
__host__ __device__ constexpr int num_stages(int NM) {
  return NM <= 16 ? 8 : (NM <= 32 ? 6 : (NM <= 48 ? 5 : 4));
}

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int ws_bad;
  int last;
  unsigned int amax_bits[kFusedMaxM];
  float s_a[kFusedMaxM];
};

__host__ __device__ constexpr size_t smem_bytes(int NM) {
  return 1024 /* alignment slack */ + size_t(num_stages(NM)) * stage_bytes(NM) +
         size_t(num_stages(NM)) * 256 * sizeof(__half) + (2 * num_stages(NM) + 9) * sizeof(uint64_t) +
         sizeof(Misc) + 64;
}

struct TcArgs {
  int M, N, K, G, T_m, NMrows;
  long long U;
  uint16_t* y;
  const __half* S;
  float* partial;         // [gridDim.x][2][128][NM]
  unsigned int* ticket;   // [tiles]
  const float* s_a;       // kA4Codes: per-token scales
  const uint16_t* x;      // kA4Fused: activations for the amax prologue
  int32_t* acc_out;
  int8_t* xq_out;
  float* xs_out;
  WsGuard guard;          // the workspace's layout claim
};


// Bounded wait: false if it gave up (then the whole CTA runs in abort mode).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimit) {
      *abort_flag = 1;
      atomicOr(&g_linear_error, 1u);
      return false;
    }
  }
}

// Wait that ignores the abort flag (used to let in-flight copies land before exit); bounded.
__device__ __forceinline__ void wait_bar_final(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimit) {
      atomicOr(&g_linear_error, 1u);
      return;
    }
  }
}

// Stages of one CTA's unit range [u_beg, u_end): a stage is up to two consecutive groups of one
// tile.  Tiles are numbered n-major (tile = n_tile * T_m + m_tile); everything is advanced
// incrementally in 32-bit arithmetic (one division per CTA).
struct StageIter {
  uint32_t u, u_end, G, T_m;
  uint32_t tile, g, n_tile, m_tile;  // current position
  uint32_t cur_g, cur_ng, cur_tile, cur_n_tile, cur_m_tile;
  bool cur_last;
  __device__ StageIter(uint32_t ub, uint32_t ue, uint32_t G_, uint32_t T_m_) : u(ub), u_end(ue), G(G_), T_m(T_m_) {
    tile = ub / G_;
    g = ub - tile * G_;
    n_tile = tile / T_m_;
    m_tile = tile - n_tile * T_m_;
  }
  __device__ bool next() {
    if (u >= u_end) return false;
    cur_g = g;
    cur_tile = tile;
    cur_n_tile = n_tile;
    cur_m_tile = m_tile;
    const uint32_t left_tile = G - g, left_cta = u_end - u;
    const uint32_t left = left_tile < left_cta ? left_tile : left_cta;
    cur_ng = left < 2 ? left : 2;
    cur_last = cur_ng == left;
    u += cur_ng;
    g += cur_ng;
    if (g == G) {
      g = 0;
      ++tile;
      if (++m_tile == T_m) {
        m_tile = 0;
        ++n_tile;
      }
    }
    return true;
  }
};

__device__ __forceinline__ uint32_t owner_of(uint32_t u, uint32_t U, uint32_t P) {
  return static_cast<uint32_t>(((static_cast<uint64_t>(u) + 1) * P - 1) / U);
}

// One packed word (channels k0..k7 of a row as two's complement nibbles in the order k0, k2, k4,
// k6, k1, k3, k5, k7) -> 4 bf16x2 words holding (k0,k1), (k2,k3), (k4,k5), (k6,k7): nibble pair
// (i, i + 4) is shifted to bits 0..3 / 16..19 and its top bit flipped into the low mantissa bits of
// bf16 128.0, giving exactly 136 + code.  With OFFSET the words are left at 136 + code (a second
// MMA against a constant -136 operand removes the offset); otherwise 136 is subtracted here.
template <bool OFFSET>
__device__ __forceinline__ void codes_to_bf16x2(uint32_t w, uint32_t* out) {
  const __nv_bfloat162 off = __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43084308u));
    if constexpr (OFFSET) {
      out[i] = v;
    } else {
      const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
      out[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
}

// TMEM columns: 256 of A (two stage buffers), 2 x 2 x chains x NM of D, and, where they fit, 8 of a
// constant -136 A operand for the offset form of the weight conversion.
__host__ __device__ constexpr bool tc_offset(int NM) { return 256 + 4 * tc_chains(NM) * NM + 8 <= 512; }

template <int NM, int MODE>
__global__ void __launch_bounds__(tc_threads(NM), 1)
    linear_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const TcArgs a) {
  constexpr int NS = num_stages(NM);
  constexpr int SB = stage_bytes(NM);
  constexpr int HALF = NM / 2;
  constexpr int CH = tc_chains(NM);
  constexpr int NI = tc_issuers(NM);
  constexpr int DB = 2;  // accumulator (D) buffers in TMEM
  constexpr bool OFFSET = tc_offset(NM);
  constexpr uint32_t kConstCol = 256 + DB * 2 * CH * NM;  // the -136 operand (OFFSET only)
  static_assert(kConstCol + (OFFSET ? 8 : 0) <= kTmemCols, "TMEM columns");
  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned tiles (alignment of the shared-window offset)
  uint8_t* ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __half* sc = reinterpret_cast<__half*>(ring + NS * SB);  // [NS][2][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(sc + NS * 256);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;
  uint64_t* afree = afull + 2;
  uint64_t* dfull = afree + 2;
  uint64_t* dfree = dfull + DB;
  uint64_t* done = dfree + DB;
  Misc* misc = reinterpret_cast<Misc*>(done + 1);
  volatile int* abort_flag = &misc->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, 2);                  // producer (expect_tx) + scale warp
      mbar_init(empty + i, kWorkerWarps + NI);  // worker warps + one commit per issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(afull + i, kWorkerWarps);
      mbar_init(afree + i, NI);
    }
    for (int i = 0; i < DB; ++i) {
      mbar_init(dfull + i, NI);
      mbar_init(dfree + i, kWorkerWarps);
    }
    mbar_init(done, NI);
    misc->abort_flag = 0;
    misc->last = 0;
    for (int i = 0; i < kFusedMaxM; ++i) misc->amax_bits[i] = 0;
    // the workspace must hold this shape's layout (or none yet); otherwise nothing is touched.  The
    // claim may run before the dependency wait: the header only ever goes from 0 to a tag.
    misc->ws_bad = ws_claim(a.guard) ? 0 : 1;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&misc->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  if (misc->ws_bad) {  // (uniform over the CTA)
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }

  // Programmatic dependent launch: let the next kernel start launching; wait for the previous one
  // before touching global memory.
  grid_launch_dependents();
  grid_dependency_wait();

  const uint32_t P = gridDim.x, c = blockIdx.x;
  const uint32_t U = static_cast<uint32_t>(a.U);
  const uint32_t u_beg = static_cast<uint32_t>(static_cast<uint64_t>(c) * U / P);
  const uint32_t u_end = static_cast<uint32_t>(static_cast<uint64_t>(c + 1) * U / P);
  const int G = a.G;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      fence_proxy_async_global();
      StageIter it(u_beg, u_end, G, a.T_m);
      int s = 0, issued = 0;
      while (it.next()) {
        const int slot = s % NS;
        if (s >= NS) wait_bar(empty + slot, ((s / NS) - 1) & 1, abort_flag);
        if (!*abort_flag) {
          ++issued;
          uint8_t* st = ring + slot * SB;
          mbar_arrive_expect_tx(full + slot, SB);
          tma_load_2d(st, &tmW, full + slot, static_cast<int>(it.cur_g * 64), static_cast<int>(it.cur_n_tile * 128));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_2d(st + kWBytes + j * (NM * 128), &tmX, full + slot, static_cast<int>(it.cur_g * 128 + 64 * j),
                        static_cast<int>(it.cur_m_tile * a.NMrows));
        }
        ++s;
      }
      // nothing may still be copying into shared memory when the CTA exits
      for (int t = (issued > NS ? issued - NS : 0); t < issued; ++t) wait_bar_final(full + t % NS, (t / NS) & 1);
    }
  } else if (warp == 1 || warp >= kFirstExtraIssuer) {
    // ------------------------------------------------------------------ MMA issuers
    // issuer i handles group i / CH of each stage and the 16-channel steps kk = i % CH (mod CH)
    const int issuer = warp == 1 ? 0 : warp - kFirstExtraIssuer + 1;
    const int jg = issuer / CH, ch = issuer % CH;
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NM);
      StageIter it(u_beg, u_end, G, a.T_m);
      int s = 0;
      while (it.next()) {
        const int slot = s % NS, pa = s & 1, pd = s % DB;
        bool ok = wait_bar(afull + pa, (s >> 1) & 1, abort_flag);
        if (s >= DB) ok = wait_bar(dfree + pd, ((s / DB) - 1) & 1, abort_flag) && ok;
        ok = wait_bar(full + slot, (s / NS) & 1, abort_flag) && ok;
        if (ok && !*abort_flag && jg < static_cast<int>(it.cur_ng)) {
          tc_fence_after();
          const uint32_t a_base = tmem + pa * 128;
          const uint32_t b_base = smem_u32(ring + slot * SB + kWBytes);
          const uint32_t d = tmem + 256 + ((pd * 2 + jg) * CH + ch) * NM;
#pragma unroll
          for (int kk = ch; kk < 8; kk += CH) {
            const int kb = jg * 8 + kk;  // 16-channel step within the stage
            const uint64_t bd = smem_desc_sw128(b_base + (kb >> 2) * (NM * 128) + (kb & 3) * 32);
            mma_bf16_ts(d, a_base + kb * 8, bd, idesc, kk >= CH ? 1u : 0u);
            if constexpr (OFFSET) mma_bf16_ts(d, tmem + kConstCol, bd, idesc, 1u);
          }
        }
        mma_commit(empty + slot);
        mma_commit(afree + pa);
        mma_commit(dfull + pd);
        ++s;
      }
      mma_commit(done);
      wait_bar_final(done, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ group-scale stager
    // Lane l stages rows 4l..4l+3 of the tile (two groups each).  Loads run two batches of
    // kScaleBatch stages ahead of the stores so that their latency overlaps the weight stream.
    constexpr int kScaleBatch = 4;
    struct Batch {
      int n0[kScaleBatch], ng[kScaleBatch];
      int count;
      __half v[kScaleBatch][8];
    };
    StageIter it(u_beg, u_end, G, a.T_m);
    auto fetch = [&](Batch& b) {
      b.count = 0;
#pragma unroll
      for (int j = 0; j < kScaleBatch; ++j) {
        b.ng[j] = 0;
        b.n0[j] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) b.v[j][i] = __ushort_as_half(0);
        if (b.count == j && it.next()) {
          b.count = j + 1;
          b.ng[j] = static_cast<int>(it.cur_ng);
          b.n0[j] = static_cast<int>(it.cur_n_tile) * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = b.n0[j] + lane * 4 + i;
            if (n < a.N) {
              const __half* srow = a.S + static_cast<long long>(n) * G + it.cur_g;
              b.v[j][2 * i] = __ldg(srow);
              if (it.cur_ng == 2) b.v[j][2 * i + 1] = __ldg(srow + 1);
            }
          }
        }
      }
    };
    int s = 0;
    auto store = [&](const Batch& b) {
#pragma unroll
      for (int j = 0; j < kScaleBatch; ++j) {
        if (j < b.count) {
          const int slot = s % NS;
          if (s >= NS) wait_bar(empty + slot, ((s / NS) - 1) & 1, abort_flag);
          __half* dst = sc + slot * 256;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dst[lane * 4 + i] = b.v[j][2 * i];
            dst[128 + lane * 4 + i] = b.v[j][2 * i + 1];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(full + slot);
          ++s;
        }
      }
      return b.count == kScaleBatch;
    };
    Batch A, B;
    fetch(A);
    while (true) {
      fetch(B);
      if (!store(A)) break;
      fetch(A);
      if (!store(B)) break;
    }
  } else {
    // ------------------------------------------------------------------ workers: dequant + drain
    const int wi = warp - kFirstWorker;   // 0..7
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int h = wi >> 2;                // which group of a stage (dequant) / token half (drain)
    const int row = q * 32 + lane;        // output row within the tile = TMEM lane
    const int wt = wi * 32 + lane;        // 0..255 among the workers
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int M = a.M, N = a.N;

    if constexpr (MODE == kA4Fused) {
      // per-token amax over all of K (tokens < M <= 4), then s_a = amax / 7 in fp32
      for (int m = 0; m < M; ++m) {
        uint32_t mx = 0;
        const uint16_t* xr = a.x + static_cast<long long>(m) * a.K;
        for (int k8 = wt; k8 < a.K / 8; k8 += 256) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + k8);
          mx = max(mx, max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu)));
          mx = max(mx, max(max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu)));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if (lane == 0) atomicMax(&misc->amax_bits[m], mx);
      }
      named_bar_sync(1, kWorkerWarps * 32);
      if (wt < M) misc->s_a[wt] = __fdiv_rn(__uint_as_float(misc->amax_bits[wt] << 16), 7.0f);
      named_bar_sync(1, kWorkerWarps * 32);
      if (blockIdx.x == 0 && a.xs_out && wt < M) a.xs_out[wt] = misc->s_a[wt];
      if (a.xq_out) {  // this CTA's slice of the int8 codes
        const int k0 = static_cast<int>(c * a.K / P), k1 = static_cast<int>((c + 1) * a.K / P);
        for (int m = 0; m < M; ++m) {
          const float sa = misc->s_a[m];
          for (int k = k0 + wt; k < k1; k += 256) {
            const float xv = bf16_lo(a.x[static_cast<long long>(m) * a.K + k]);
            const float cq = sa == 0.0f ? 0.0f : fminf(fmaxf(rintf(__fdiv_rn(xv, sa)), -8.0f), 7.0f);
            a.xq_out[static_cast<long long>(m) * a.K + k] = static_cast<int8_t>(cq);
          }
        }
      }
    }

    if constexpr (OFFSET) {
      // the constant A operand: -136 (bf16 0xC308) in every element of this warp's 32 lanes
      if (h == 0) {
        const uint32_t neg136[8] = {0xC308C308u, 0xC308C308u, 0xC308C308u, 0xC308C308u,
                                    0xC308C308u, 0xC308C308u, 0xC308C308u, 0xC308C308u};
        tmem_st8(tmem + lane_base + kConstCol, neg136);
        tmem_wait_st();  // ordered before the MMAs by the first stage's afull hand-over
      }
    }

    float acc[HALF];
#pragma unroll
    for (int t = 0; t < HALF; ++t) acc[t] = 0.0f;

    struct Pending {
      int s, ng, g;
      uint32_t tile;
      int n_tile, m_tile;
      bool last;
      float s0, s1;
    };

    // Accumulator registers of one stage between issuing its TMEM loads and using them: chain 0
    // of each group in d0 / d1, the second chain (CH = 2) in e0 / e1.
    struct DrainRegs {
      uint32_t d0[HALF], d1[HALF], e0[CH > 1 ? HALF : 1], e1[CH > 1 ? HALF : 1];
    };

    // Waits for the stage's MMAs and issues its TMEM loads (not yet waited for).
    auto drain_issue = [&](const Pending& p, DrainRegs& r) -> bool {
      const int pd = p.s % DB;
      const bool ok = wait_bar(dfull + pd, (p.s / DB) & 1, abort_flag);
      tc_fence_after();
      if (ok) {
        const uint32_t dcol = tmem + lane_base + 256 + pd * 2 * CH * NM + h * HALF;
#pragma unroll
        for (int c8 = 0; c8 < HALF / 8; ++c8) {
          tmem_ld8(dcol + 8 * c8, r.d0 + 8 * c8);
          if constexpr (CH > 1) tmem_ld8(dcol + NM + 8 * c8, r.e0 + 8 * c8);
        }
        if (p.ng == 2) {
#pragma unroll
          for (int c8 = 0; c8 < HALF / 8; ++c8) {
            tmem_ld8(dcol + CH * NM + 8 * c8, r.d1 + 8 * c8);
            if constexpr (CH > 1) tmem_ld8(dcol + CH * NM + NM + 8 * c8, r.e1 + 8 * c8);
          }
        }
      }
      return ok;
    };

    // Completes the loads, releases the D buffer and adds s[n, g] * D into the running sums.
    auto drain_finish = [&](const Pending& p, DrainRegs& r, bool ok) {
      if (ok) {
        tmem_wait_ld();
        if constexpr (CH > 1) {
#pragma unroll
          for (int t = 0; t < HALF; ++t) {
            r.d0[t] = __float_as_uint(__uint_as_float(r.d0[t]) + __uint_as_float(r.e0[t]));
            if (p.ng == 2) r.d1[t] = __float_as_uint(__uint_as_float(r.d1[t]) + __uint_as_float(r.e1[t]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dfree + p.s % DB);
      if (!ok || *abort_flag) return;
#pragma unroll
      for (int t = 0; t < HALF; ++t) acc[t] = fmaf(p.s0, __uint_as_float(r.d0[t]), acc[t]);
      if (p.ng == 2) {
#pragma unroll
        for (int t = 0; t < HALF; ++t) acc[t] = fmaf(p.s1, __uint_as_float(r.d1[t]), acc[t]);
      }
      if constexpr (MODE != kA16) {
        if (a.acc_out) {
          const int n = p.n_tile * 128 + row;
          const int m0 = p.m_tile * a.NMrows + h * HALF;
#pragma unroll
          for (int t = 0; t < HALF; ++t) {
            const int m = m0 + t;
            if (m < M && n < N) {
              int32_t* dst = a.acc_out + (static_cast<long long>(m) * N + n) * G + p.g;
              dst[0] = static_cast<int32_t>(__uint_as_float(r.d0[t]));
              if (p.ng == 2) dst[1] = static_cast<int32_t>(__uint_as_float(r.d1[t]));
            }
          }
        }
      }
    };

    auto drain = [&](const Pending& p) {
      DrainRegs r;
      const bool ok = drain_issue(p, r);
      drain_finish(p, r, ok);
    };

    auto token_scale = [&](int m) -> float {
      if constexpr (MODE == kA4Fused) return misc->s_a[m];
      else if constexpr (MODE == kA4Codes) return __ldg(a.s_a + m);
      else return 1.0f;
    };

    auto store_y = [&](const Pending& p, const float* v) {
      const int n = p.n_tile * 128 + row;
      const int m0 = p.m_tile * a.NMrows + h * HALF;
#pragma unroll
      for (int t = 0; t < HALF; ++t) {
        const int m = m0 + t;
        if (m < M && n < N) {
          float o = v[t];
          if constexpr (MODE != kA16) o *= token_scale(m);
          a.y[static_cast<long long>(m) * N + n] = f32_to_bf16_bits(o);
        }
      }
    };

    auto epilogue = [&](const Pending& p) {
      const uint32_t tile = p.tile;
      const uint32_t c_first = owner_of(tile * G, U, P);
      const uint32_t c_last = owner_of((tile + 1) * G - 1, U, P);
      if (c_first == c_last) {
        if (!*abort_flag) store_y(p, acc);
      } else {
        // only the float4 columns of this warp's token half that hold real tokens travel
        constexpr int NV = HALF / 4;
        const int m_here = min(NM, M - p.m_tile * a.NMrows);
        const int nv = max(0, min(NV, (m_here - h * HALF + 3) / 4));
        const int my_slot = (tile == u_beg / G) ? 0 : 1;
        float* part = a.partial + ((static_cast<size_t>(c) * 2 + my_slot) * 128 + row) * NM + h * HALF;
#pragma unroll
        for (int t = 0; t < NV; ++t)
          if (t < nv)
            *reinterpret_cast<float4*>(part + 4 * t) = make_float4(acc[4 * t], acc[4 * t + 1], acc[4 * t + 2], acc[4 * t + 3]);
        __threadfence();
        named_bar_sync(1, kWorkerWarps * 32);
        if (wt == 0) {
          const unsigned int prevc = atomicAdd(a.ticket + tile, 1u);
          misc->last = prevc == static_cast<unsigned int>(c_last - c_first);
        }
        named_bar_sync(1, kWorkerWarps * 32);
        if (misc->last) {
          __threadfence();
          // Contributor c_first may have begun in an earlier tile (this tile is then its slot 1);
          // every later contributor begins inside this tile (slot 0): c * U / P > tile * G for
          // c > c_first, and it is at most the tile's last unit for c <= c_last.
          const uint32_t first_beg = static_cast<uint32_t>(static_cast<uint64_t>(c_first) * U / P);
          const uint32_t first_slot = first_beg / G == tile ? 0u : 1u;
          // acc is already published above, so it is reused as the running sum of all
          // contributors' partials, added in CTA order with kFixBatch contributors' loads in flight
#pragma unroll
          for (int t = 0; t < HALF; ++t) acc[t] = 0.0f;
          constexpr int kFixBatch = NM == 16 ? 8 : 1;
          const float* pbase = a.partial + static_cast<size_t>(row) * NM + h * HALF;
          for (uint32_t c0 = c_first; c0 <= c_last; c0 += kFixBatch) {
            float4 v[kFixBatch][NV];
#pragma unroll
            for (int j = 0; j < kFixBatch; ++j) {
              const uint32_t cc = c0 + j;
              const uint32_t sl = cc == c_first ? first_slot : 0u;
              const float4* src = reinterpret_cast<const float4*>(pbase + (static_cast<size_t>(cc) * 2 + sl) * 128 * NM);
#pragma unroll
              for (int t = 0; t < NV; ++t)
                v[j][t] = (cc <= c_last && t < nv) ? __ldcg(src + t) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int j = 0; j < kFixBatch; ++j) {
              if (c0 + j <= c_last) {
#pragma unroll
                for (int t = 0; t < NV; ++t) {
                  acc[4 * t] += v[j][t].x;
                  acc[4 * t + 1] += v[j][t].y;
                  acc[4 * t + 2] += v[j][t].z;
                  acc[4 * t + 3] += v[j][t].w;
                }
              }
            }
          }
          if (!*abort_flag) store_y(p, acc);
          if (wt == 0) a.ticket[tile] = 0;
        }
      }
#pragma unroll
      for (int t = 0; t < HALF; ++t) acc[t] = 0.0f;
    };

    Pending prev{};
    bool has_prev = false;

    StageIter it(u_beg, u_end, G, a.T_m);
    int s = 0;
    while (it.next()) {
      const int slot = s % NS, pa = s & 1;
      bool ok = wait_bar(full + slot, (s / NS) & 1, abort_flag);
      if (s >= 2) ok = wait_bar(afree + pa, ((s >> 1) - 1) & 1, abort_flag) && ok;
      Pending cur{s, static_cast<int>(it.cur_ng), static_cast<int>(it.cur_g), it.cur_tile,
                  static_cast<int>(it.cur_n_tile), static_cast<int>(it.cur_m_tile), it.cur_last, 0.0f, 0.0f};
      const bool work = ok && !*abort_flag;
      const bool convert = work && h < static_cast<int>(it.cur_ng);
      uint8_t* st = ring + slot * SB;
      const uint8_t* wrow = st + row * 128;  // this warp's 128 codes: one group of 32 rows
      if (work) {
        cur.s0 = __half2float(sc[slot * 256 + row]);
        cur.s1 = __half2float(sc[slot * 256 + 128 + row]);
        if constexpr (MODE == kA4Fused) {
          // activation tile -> INT4 codes (as exact bf16) in place, rows m < M
          uint8_t* bst = st + kWBytes;
          for (int m = 0; m < M; ++m) {
            const int k = wt;  // 0..255 within the stage
            const int j = k >> 6, kin = k & 63;
            uint16_t* p = reinterpret_cast<uint16_t*>(bst + j * (NM * 128) + (m >> 3) * 1024 + (m & 7) * 128 +
                                                      ((((kin >> 3) ^ (m & 7))) << 4) + (kin & 7) * 2);
            const float sa = misc->s_a[m];
            const float cq = sa == 0.0f ? 0.0f : fminf(fmaxf(rintf(__fdiv_rn(bf16_lo(*p), sa)), -8.0f), 7.0f);
            *p = f32_to_bf16_bits(cq);
          }
          fence_proxy_async_smem();
        }
        if (convert) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((((4 * h + cc) ^ (row & 7))) << 4));
            uint32_t out[16];
            codes_to_bf16x2<OFFSET>(v.x, out);
            codes_to_bf16x2<OFFSET>(v.y, out + 4);
            codes_to_bf16x2<OFFSET>(v.z, out + 8);
            codes_to_bf16x2<OFFSET>(v.w, out + 12);
            tmem_st16(tmem + lane_base + pa * 128 + h * 64 + cc * 16, out);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(afull + pa);
        mbar_arrive(empty + slot);
      }
      if (has_prev) {
        drain(prev);
        if (prev.last) epilogue(prev);
      }
      prev = cur;
      has_prev = true;
      ++s;
    }
    if (has_prev) {
      drain(prev);
      if (prev.last) epilogue(prev);
    }
  }
  // Lane 0 of the producer and issuer warps ran its role alone; reconverge every warp before the
  // CTA barrier (a partially arrived warp must not count as arrived), so TMEM is released only
  // after every worker has finished reading it.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

}  // namespace

// A 2-D tensor map (dims {inner, outer}, row pitch row_bytes, box {box_inner, box_outer}); rows or
// columns outside the tensor read as zeros.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_map_2d(map, dt, base, inner, outer, row_bytes, box_inner, box_outer, true);
}

// The fused kernel quantises W4A4 tokens itself (M <= 4); other quantised cases (W4A4 at larger M,
// every W4A8) are quantised once by the quantiser kernel (quant.cu) and multiply codes.
bool fused_mode(int abits, int M) { return abits == 4 && M <= kFusedMaxM; }
bool codes_mode_of(int abits, int M) { return abits != 16 && !fused_mode(abits, M); }

int pick_nm(int abits, int M) {
  if (fused_mode(abits, M)) return 16;
  return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 48 ? 48 : 64));
}

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t ticket, partial, codes, s_a, total;
};

// Stream-K grid: P CTAs share U = tiles x groups units.  A CTA costs about its units plus, for
// the last contributor of a split tile, one read of every other contributor's partial tile
// (NM >= 32: one contributor's loads in flight at a time, about 1.5 units each; NM = 16: eight
// in flight).  Few tiles over many CTAs make many contributors per tile, so the grid is the P that
// minimises ceil(U / P) + (contributors per tile) x fixup cost, ties to the wider grid.
int pick_ctas(int NM, long long U, int G, int sms) {
  const double fix = NM == 16 ? 0.25 : 1.5;
  int best = 1;
  double best_cost = 0.0;
  const int p_max = static_cast<int>(std::min<long long>(U, sms));
  for (int P = 1; P <= p_max; ++P) {
    const long long per = (U + P - 1) / P;
    const long long contrib = (static_cast<long long>(G) * P + U - 1) / U + 1;
    const double cost = static_cast<double>(per) + (P > 1 ? fix * static_cast<double>(contrib) : 0.0);
    if (P == 1 || cost <= best_cost) {
      best = P;
      best_cost = cost;
    }
  }
  return best;
}

WsLayout ws_layout(int abits, int M, int N, int K, int P) {
  const int NM = pick_nm(abits, M);  // tiles of NM >= 16 tokens: at most tc_ticket_count tickets
  WsLayout L;
  size_t off = kWsHeader;  // the layout header comes first
  L.ticket = off;  off = al256(off + sizeof(unsigned int) * tc_ticket_count(M, N));
  L.partial = off; off = al256(off + sizeof(float) * size_t(P) * 2 * 128 * NM);
  // quantised codes and scales: used by the codes mode here, and by the GEMV when it quantises
  // the tokens in a separate kernel
  const bool codes = abits != 16;
  L.codes = off;   off = al256(off + (codes ? sizeof(uint16_t) * size_t(M) * K : 0));
  L.s_a = off;     off = al256(off + (codes ? sizeof(float) * size_t(M) : 0));
  L.total = off;
  return L;
}

template <int NM, int MODE>
qspec_status launch_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const TcArgs& args, int P,
                       cudaStream_t stream) {
  auto kern = linear_tc_kernel<NM, MODE>;
  const size_t smem = smem_bytes(NM);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return QSPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P);
  cfg.blockDim = dim3(tc_threads(NM));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, args) == cudaSuccess ? QSPEC_OK : QSPEC_ERR_CUDA;
}

}  // namespace

bool linear_tc_supported(int abits, int M, int N, int K) {
  if (abits == 16 && linear_dq_supported(M, N, K)) return true;
  if (M < 1 || M > QSPEC_MAX_M || N < 8 || K < kGroup) return false;
  const int NM = pick_nm(abits, M);
  const long long U = (static_cast<long long>(N) + 127) / 128 * ((M + NM - 1) / NM) * (K / kGroup);
  return U < (1LL << 31);  // the device side counts units in 32 bits
}

size_t linear_tc_workspace_size(int abits, int M, int N, int K) {
  if (abits == 16 && linear_dq_supported(M, N, K)) return linear_dq_workspace_size(M, N, K);
  return ws_layout(abits, M, N, K, num_sms()).total;
}

qspec_status linear_tc(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K,
                       uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws, size_t ws_bytes,
                       const WsGuard& guard, cudaStream_t stream) {
  if (abits == 16 && linear_dq_supported(M, N, K)) return linear_dq(x, Wp, S, M, N, K, y, ws, ws_bytes, guard, stream);
  const int NM = pick_nm(abits, M);
  const int T_m = (M + NM - 1) / NM;
  const long long T = (static_cast<long long>(N) + 127) / 128 * T_m;
  const int G = K / kGroup;
  const long long U = T * G;
  const int P = pick_ctas(NM, U, G, num_sms());
  const WsLayout L = ws_layout(abits, M, N, K, num_sms());
  if (!ws || ws_bytes < L.total) return QSPEC_ERR_WORKSPACE;
  char* wsb = static_cast<char*>(ws);

  const bool codes_mode = codes_mode_of(abits, M);
  uint16_t* codes = reinterpret_cast<uint16_t*>(wsb + L.codes);
  float* s_a = reinterpret_cast<float*>(wsb + L.s_a);

  CUtensorMap tmW, tmX;
  if (!make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wp, static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N),
                   static_cast<uint64_t>(K) / 2, 128, 128))
    return QSPEC_ERR_CUDA;
  const void* bsrc = codes_mode ? static_cast<const void*>(codes) : static_cast<const void*>(x);
  if (!make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, bsrc, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K) * 2, 64, static_cast<uint32_t>(NM)))
    return QSPEC_ERR_CUDA;

  if (codes_mode) {
    const qspec_status st = quantise_tokens(abits, x, M, K, false, codes, s_a, xq_out, xs_out, guard, stream);
    if (st != QSPEC_OK) return st;
  }

  TcArgs args;
  args.M = M;
  args.N = N;
  args.K = K;
  args.G = G;
  args.T_m = T_m;
  args.NMrows = NM;
  args.U = U;
  args.y = y;
  args.S = reinterpret_cast<const __half*>(S);
  args.partial = reinterpret_cast<float*>(wsb + L.partial);
  args.ticket = reinterpret_cast<unsigned int*>(wsb + L.ticket);
  args.s_a = s_a;
  args.x = x;
  args.acc_out = acc_out;
  args.xq_out = xq_out;
  args.xs_out = xs_out;
  args.guard = guard;

  if (abits == 16) {
    switch (NM) {
      case 16: return launch_tc<16, kA16>(tmW, tmX, args, P, stream);
      case 32: return launch_tc<32, kA16>(tmW, tmX, args, P, stream);
      case 48: return launch_tc<48, kA16>(tmW, tmX, args, P, stream);
      default: return launch_tc<64, kA16>(tmW, tmX, args, P, stream);
    }
  }
  if (!codes_mode) return launch_tc<16, kA4Fused>(tmW, tmX, args, P, stream);
  switch (NM) {
    case 16: return launch_tc<16, kA4Codes>(tmW, tmX, args, P, stream);
    case 32: return launch_tc<32, kA4Codes>(tmW, tmX, args, P, stream);
    case 48: return launch_tc<48, kA4Codes>(tmW, tmX, args, P, stream);
    default: return launch_tc<64, kA4Codes>(tmW, tmX, args, P, stream);
  }
}

size_t linear_tc_workspace_size_all(int M, int N, int K) {
  size_t n = 0;
  for (int abits : {16, 4, 8}) n = std::max(n, linear_tc_workspace_size(abits, M, N, K));
  return n;
}

bool ws_codes(int abits, int M, int N, int K, void* ws, uint16_t** codes, float** s_a) {
  if (abits == 16 || !ws) return false;
  const WsLayout L = ws_layout(abits, M, N, K, num_sms());
  *codes = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + L.codes);
  *s_a = reinterpret_cast<float*>(static_cast<char*>(ws) + L.s_a);
  return true;
}

qspec_status read_and_clear_linear_error(cudaStream_t stream, unsigned int* bits) {
  *bits = 0;
  if (cudaMemcpyFromSymbolAsync(bits, g_linear_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return QSPEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QSPEC_ERR_CUDA;
  if (*bits) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_linear_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return QSPEC_ERR_CUDA;
  }
  return QSPEC_OK;
}

}  // namespace qspec
