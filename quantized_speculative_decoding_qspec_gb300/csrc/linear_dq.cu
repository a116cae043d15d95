// Host side of the tensor-core W4A16 linear (dq_impl.cuh): the activation conversion kernel, the
// workspace layout and the launch plan (tokens per tile, tiles per item, CTAs).
#include <algorithm>

#include "dq_impl.cuh"

namespace qspec {
namespace {

using dq::DqArgs;

constexpr int kPThreads = 256;

// Tokens -> fp16 with one power-of-two factor per token (the B operand of the kernel).  The factor
// 2^e puts the token's largest magnitude in [2^14, 2^15): every bf16 value of the token that is not
// below 2^-28 of it becomes an fp16 normal number with the same significand, so the conversion is
// exact there; pw[m] = 2^e undoes it in the epilogue.
__global__ void __launch_bounds__(kPThreads) tokens_f16_kernel(const uint16_t* __restrict__ x, int K,
                                                              uint16_t* __restrict__ xh, float* __restrict__ pw,
                                                              WsGuard guard) {
  __shared__ unsigned int s_max[kPThreads / 32];
  __shared__ int s_ok;
  if (threadIdx.x == 0) s_ok = ws_claim(guard) ? 1 : 0;
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  __syncthreads();
  if (!s_ok) return;
  const int m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K);
  unsigned int mx = 0;
  for (int i = threadIdx.x; i < K / 8; i += kPThreads) {
    const uint4 v = __ldg(xr + i);
    mx = max(mx, max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu)));
    mx = max(mx, max(max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu)));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
#pragma unroll
  for (int w = 0; w < kPThreads / 32; ++w) mx = max(mx, s_max[w]);
  // floor(log2(amax)) from the bf16 exponent field (subnormals: from the position of the top bit)
  int e = 0;
  if (mx != 0) {
    const int field = static_cast<int>(mx >> 7);
    const int E = field != 0 ? field - 127 : -126 - (7 - (31 - __clz(mx & 0x7Fu)));
    e = E - 14;
  }
  // 2^-e as two normal fp32 factors (-e lies in [-113, 147])
  const int h1 = (-e) / 2, h2 = -e - h1;
  const float f1 = __uint_as_float(static_cast<uint32_t>(h1 + 127) << 23);
  const float f2 = __uint_as_float(static_cast<uint32_t>(h2 + 127) << 23);
  if (threadIdx.x == 0)
    pw[m] = e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(1u << (e + 149));
  uint4* dst = reinterpret_cast<uint4*>(xh + static_cast<size_t>(m) * K);
  for (int i = threadIdx.x; i < K / 8; i += kPThreads) {
    const uint4 v = __ldg(xr + i);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const __half lo = __float2half_rn(bf16_lo(in[p]) * f1 * f2);
      const __half hi = __float2half_rn(bf16_hi(in[p]) * f1 * f2);
      out[p] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
    dst[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

int pick_nm(int M) { return M <= 128 ? 128 : 256; }
int max_j(int NM) { return NM == 128 ? 2 : 1; }

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct Plan {
  int NM, J, T_m, KB, P;
  long long items;
  uint32_t dp, sk_beg, sk_units;  // whole items per CTA; the units shared out after them
};

// Model of one CTA's time, in clock cycles.  A unit (one 64-channel block of J tiles) costs the
// largest of: its weight bytes at the per-SM share of HBM bandwidth, its dequantisation (about 170
// cycles a tile plus a hand-over) and its MMAs (about 0.6 NM cycles each on the tensor core).  With
// one accumulator set in TMEM every item's drain stalls the MMAs; an item cut between CTAs costs its
// last contributor a read of every contributor's partial tile.  (The constants were set by timing
// the Llama-2-70B layers at 128 and 256 tokens; raising the partial-tile cost moved those to J = 1
// and made them up to 35% slower.)
double plan_cost(int NM, int J, int KB, int P, uint32_t dp, uint32_t sk_units) {
  const double hbm = J * (dq::kWTile / dq::kQuad) / 21.0;
  const double conv = J * 170.0 + 150.0;
  const double mma = J * 4 * 0.6 * NM + 100.0;
  const double unit = std::max(std::max(hbm, mma), conv);
  const double per = static_cast<double>(dp) * KB + static_cast<double>((sk_units + P - 1) / P);
  double cost = per * unit;
  if (dq::acc_sets(NM, J) == 1) cost += (dp + (sk_units > 0 ? 2.0 : 0.0)) * (1500.0 + 6.0 * J * NM);
  const bool split = sk_units > 0 && !(sk_units % P == 0 && (sk_units / P) % KB == 0);
  if (split) {
    const double contrib = static_cast<double>((static_cast<uint64_t>(KB) * P + sk_units - 1) / sk_units + 1);
    cost += contrib * (800.0 + 3.0 * J * NM);
  }
  return cost;
}

// The whole items per CTA and the shared-out units of P CTAs: every CTA gets at least one shared
// unit or none (so each contributor of a split item has written its partial tile); false if P CTAs
// cannot be given work that way.
bool split_work(long long items, int KB, int P, uint32_t* dp, uint32_t* sk_units) {
  long long d = items / P;
  long long r = (items - d * P) * KB;
  if (r > 0 && r < P) {
    if (d == 0) return false;
    --d;
    r += static_cast<long long>(P) * KB;
  }
  *dp = static_cast<uint32_t>(d);
  *sk_units = static_cast<uint32_t>(r);
  return true;
}

Plan make_plan(int M, int N, int K, int sms) {
  Plan pl{};
  pl.NM = pick_nm(M);
  pl.T_m = (M + pl.NM - 1) / pl.NM;
  pl.KB = K / 64;
  double best = -1.0;
  for (int J = 1; J <= max_j(pl.NM); J *= 2) {
    const long long items = (static_cast<long long>(N) + 128 * J - 1) / (128 * J) * pl.T_m;
    const long long U = items * pl.KB;
    const int p_max = static_cast<int>(std::min<long long>(U, sms));
    for (int P = 1; P <= p_max; ++P) {
      uint32_t dp = 0, sk = 0;
      if (!split_work(items, pl.KB, P, &dp, &sk)) continue;
      const double cost = plan_cost(pl.NM, J, pl.KB, P, dp, sk);
      if (best < 0.0 || cost < best) {
        best = cost;
        pl.J = J;
        pl.P = P;
        pl.items = items;
        pl.dp = dp;
        pl.sk_units = sk;
        pl.sk_beg = static_cast<uint32_t>(static_cast<long long>(dp) * P * pl.KB);
      }
    }
  }
  return pl;
}

struct Layout {
  size_t ticket, partial, xh, pw, total;
};

// Regions after the header: the tickets shared with the exact-code kernel (at least one per item of
// any plan), then the partial tiles, sized for the largest J over grids of up to `sms` CTAs.
Layout layout_of(int M, int N, int K, int sms) {
  const int NM = pick_nm(M);
  Layout L;
  size_t off = kWsHeader;
  L.ticket = off;  off = al256(off + sizeof(unsigned int) * tc_ticket_count(M, N));
  L.partial = off; off = al256(off + sizeof(float) * size_t(sms) * 2 * 128 * max_j(NM) * NM);
  L.xh = off;      off = al256(off + sizeof(uint16_t) * size_t(M) * K);
  L.pw = off;      off = al256(off + sizeof(float) * size_t(M));
  L.total = off;
  return L;
}

}  // namespace

bool linear_dq_supported(int M, int N, int K) {
  if (M < kDqMinTokens || M > QSPEC_MAX_M || N < 8 || K < kGroup) return false;
  const int NM = pick_nm(M);
  const long long items = (static_cast<long long>(N) + 127) / 128 * ((M + NM - 1) / NM);
  return items * (K / 64) < (1LL << 31);  // the device side counts units in 32 bits
}

size_t linear_dq_workspace_size(int M, int N, int K) { return layout_of(M, N, K, num_sms()).total; }

qspec_status linear_dq(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K, uint16_t* y,
                       void* ws, size_t ws_bytes, const WsGuard& guard, cudaStream_t stream) {
  const int sms = num_sms();
  const Layout L = layout_of(M, N, K, sms);
  if (!ws || ws_bytes < L.total) return QSPEC_ERR_WORKSPACE;
  const Plan pl = make_plan(M, N, K, sms);
  char* wsb = static_cast<char*>(ws);
  uint16_t* xh = reinterpret_cast<uint16_t*>(wsb + L.xh);
  float* pw = reinterpret_cast<float*>(wsb + L.pw);

  CUtensorMap tmW, tmX;
  // weight boxes of 128 bytes (256 channels) x 128 rows: narrower boxes stream far below the HBM rate
  if (!encode_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wp, static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N),
                     static_cast<uint64_t>(K) / 2, 128, 128, true))
    return QSPEC_ERR_CUDA;
  if (!encode_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                     static_cast<uint64_t>(K) * 2, 64, static_cast<uint32_t>(pl.NM), true))
    return QSPEC_ERR_CUDA;

  qspec_status st = launch_pdl(tokens_f16_kernel, dim3(M), dim3(kPThreads), 0, stream, x, K, xh, pw, guard);
  if (st != QSPEC_OK) return st;

  DqArgs args;
  args.M = M;
  args.N = N;
  args.K = K;
  args.KB = pl.KB;
  args.T_m = pl.T_m;
  args.dp_items = pl.dp;
  args.sk_beg = pl.sk_beg;
  args.sk_units = pl.sk_units;
  args.y = y;
  args.S = reinterpret_cast<const __half*>(S);
  args.pw = pw;
  args.partial = reinterpret_cast<float*>(wsb + L.partial);
  args.ticket = reinterpret_cast<unsigned int*>(wsb + L.ticket);
  args.err = guard.err;
  args.guard = guard;
  return dq_launch(pl.NM, pl.J, tmW, tmX, args, pl.P, stream);
}

}  // namespace qspec
