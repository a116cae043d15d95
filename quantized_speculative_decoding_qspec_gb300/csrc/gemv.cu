// Entry of the decode-size GEMV (both linear modes and W4A8): shape checks, K chunking, the
// separate quantiser for many tokens, and dispatch to the per-mode launchers (gemv_impl.cuh, one
// translation unit per activation mode).
#include "gemv_impl.cuh"

namespace qspec {
using namespace gemv_impl;

// Token slots for M tokens: the smallest staged width that holds them.
int token_slots(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32; }

bool gemv_supported(int M, int N, int K) {
  if (M < 1 || M > kMaxTokens || N < 1 || K % kGroup != 0) return false;
  const int kc = pick_kc(token_slots(M), K / kGroup);
  // 17..32 tokens: only up to 4 K chunks (measured on Llama-2-70B shapes at M = 32: with 4 chunks
  // the GEMV beats the tcgen05 kernel on q/o, k/v and gate/up and loses 6% on lm_head; with 14, on
  // down at K = 28672, it loses 50%)
  if (M > 16) return kc > 0 && kc <= 4;
  return kc > 0;
}

size_t gemv_workspace_bytes(int M, int N, int K) {
  if (!gemv_supported(M, N, K)) return 0;
  const int MT = token_slots(M), G = K / kGroup;
  return chunk_ws_bytes(MT, N, G, plan_kc(MT, N, G));
}

namespace {
// The GEMV over the parts of P (N = 16 x their tiles, the row count that the planners and the
// workspace see; the workspace belongs to that (M, N, K)).
qspec_status gemv_parts(int abits, const uint16_t* x, const Parts& P, int M, int N, int K, int8_t* xq_out,
                        float* xs_out, int32_t* acc_out, void* ws, const WsGuard& guard, cudaStream_t stream) {
  const int MT = token_slots(M), G = K / kGroup;
  const int KC = plan_kc(MT, N, G);
  if (KC == 0) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  Outs o{xq_out, xs_out, acc_out, nullptr, nullptr, nullptr, guard};
  if (KC > 1) {  // chunk partials and tickets live after the tensor-core path's regions
    char* base = static_cast<char*>(ws) + al256(linear_tc_workspace_size_all(M, N, K));
    const size_t tiles = (static_cast<size_t>(N) + 15) / 16;
    o.part = reinterpret_cast<float*>(base);
    o.tick = reinterpret_cast<unsigned int*>(base + al256(static_cast<size_t>(KC) * tiles * ((MT + 7) / 8) * 512));
  }
  int qb = abits == 16 ? 0 : abits;
  // Four or more tokens, or tokens that take several staging batches, would be quantised by every
  // CTA again; there the quantiser runs once, in its own kernel, and the GEMV stages the codes
  // (measured: 70B W4A4 down at M = 4, 50.5 -> 41.7 us; q/o at M = 8, 21.2 -> 16.3 us; 8B q at
  // M = 4, 8.4 -> 7.0 us; a single token is faster quantised in every CTA, 4.2 vs 5.4 us on k).
  // More than 16 tokens always take this path (the 32-slot kernel does not quantise).
  uint16_t* codes = nullptr;
  float* s_a = nullptr;
  if (qb != 0 && (M >= 4 || static_cast<long long>(M) * K > 8LL * kStageU * kThreads)) {
    if (!ws_codes(abits, M, N, K, ws, &codes, &s_a)) return QSPEC_ERR_WORKSPACE;
    const qspec_status st = quantise_tokens(abits, x, M, K, true, codes, s_a, xq_out, xs_out, guard, stream);
    if (st != QSPEC_OK) return st;
    x = codes;
    o.xq = nullptr;
    o.xs = nullptr;
    o.s_in = s_a;
    qb = 1;
  }
  switch (qb) {
    case 4: return launch_mode<4>(MT, x, P, M, N, K, o, KC, stream);
    case 8: return launch_mode<8>(MT, x, P, M, N, K, o, KC, stream);
    case 1: return launch_mode<1>(MT, x, P, M, N, K, o, KC, stream);
    default: return launch_mode<0>(MT, x, P, M, N, K, o, KC, stream);
  }
}
}  // namespace

qspec_status gemv(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K,
                  uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws, const WsGuard& guard,
                  cudaStream_t stream) {
  Parts P{};
  P.n = 1;
  P.tile_end[0] = (N + 15) / 16;
  P.N[0] = N;
  P.Wp[0] = Wp;
  P.S[0] = reinterpret_cast<const __half*>(S);
  P.y[0] = y;
  return gemv_parts(abits, x, P, M, N, K, xq_out, xs_out, acc_out, ws, guard, stream);
}

static_assert(kMaxParts == QSPEC_GROUP_MAX_PARTS && kPartsMaxMT == QSPEC_GROUP_MAX_M, "group limits");

int gemv_group_rows(const int64_t* N, int n) {
  long long tiles = 0;
  for (int i = 0; i < n; ++i) tiles += (N[i] + 15) / 16;
  return static_cast<int>(tiles * 16);
}

qspec_status gemv_group(int abits, const uint16_t* x, int M, int K, const GroupPart* parts, int n, void* ws,
                        const WsGuard& guard, cudaStream_t stream) {
  if (n < 1 || n > kMaxParts || token_slots(M) > kPartsMaxMT) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  Parts P{};
  P.n = n;
  int tiles = 0;
  for (int i = 0; i < n; ++i) {
    tiles += static_cast<int>((parts[i].N + 15) / 16);
    P.tile_end[i] = tiles;
    P.N[i] = static_cast<int>(parts[i].N);
    P.Wp[i] = parts[i].Wp;
    P.S[i] = reinterpret_cast<const __half*>(parts[i].S);
    P.y[i] = parts[i].y;
  }
  return gemv_parts(abits, x, P, M, tiles * 16, K, nullptr, nullptr, nullptr, ws, guard, stream);
}

}  // namespace qspec
