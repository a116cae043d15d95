// Steps a2 (W4A16 linear), a3 (per-token activation quantiser) and a4 (W4A4 linear) over the one
// shared packed INT4 weight tensor.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる"), section
// "W4A4 と W4A16 量子化": W4A16 converts 4-bit weights while multiplying 16-bit activations; W4A4
// quantises the activations to 4 bits as well.  Section "QSpec の W4A4 モードと W4A16 モード":
// both modes read the same 4-bit weights.
//
// This file holds the argument checks and the entry points.  Decode sizes run on the register-
// fragment GEMV (gemv.cu), larger token counts on the tcgen05 kernel (linear_tc.cu); there is no
// third path: a shape neither serves is refused with a status.
#include "common.cuh"
#include "linear_internal.h"

namespace qspec {

// Layout tag of a workspace used by (M, N, K) calls: M - 1 in bits 0..11, K / 128 - 1 in bits
// 12..34, N / 8 - 1 in bits 35..61 and bit 63 set (never 0, the value of a fresh workspace).
unsigned long long ws_tag(int M, int N, int K) {
  return (1ull << 63) | static_cast<unsigned long long>(M - 1) |
         (static_cast<unsigned long long>(K / kGroup - 1) << 12) | (static_cast<unsigned long long>(N / 8 - 1) << 35);
}

namespace {
bool make_guard(int M, int N, int K, void* ws, WsGuard* g) {
  g->hdr = static_cast<unsigned long long*>(ws);
  g->tag = ws_tag(M, N, K);
  g->err = linear_error_word();
  return g->err != nullptr;
}
}  // namespace
}  // namespace qspec

namespace {
qspec_status check_linear_args(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                               int64_t N, int64_t K, const uint16_t* y) {
  using namespace qspec;
  if (!x || !Wp || !S || !y) return QSPEC_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return QSPEC_ERR_INVALID_ARG;
  if (M > QSPEC_MAX_M || N % 8 != 0 || K % kGroup != 0 || N > (int64_t(1) << 30) ||
      K > (int64_t(1) << 30) || N * K >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(Wp) || !aligned16(S) || !aligned16(y)) return QSPEC_ERR_MISALIGNED;
  return QSPEC_OK;
}
}  // namespace

extern "C" size_t qspec_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > QSPEC_MAX_M || N % 8 != 0 || K % qspec::kGroup != 0 ||
      N > (int64_t(1) << 30) || K > (int64_t(1) << 30))
    return 0;
  // the header is the first kWsHeader bytes of the tensor-core layout
  const size_t tc = qspec::linear_tc_workspace_size_all(int(M), int(N), int(K));
  return ((tc + 255) & ~size_t(255)) + qspec::gemv_workspace_bytes(int(M), int(N), int(K));
}

extern "C" qspec_status qspec_linear_w4a16(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                           int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                           size_t ws_bytes, qspec_stream_t stream) {
  const qspec_status st = check_linear_args(x, Wp, S, M, N, K, y);
  if (st != QSPEC_OK) return st;
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!qspec::aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_workspace_size(M, N, K)) return QSPEC_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  qspec::WsGuard guard;
  if (!qspec::make_guard(int(M), int(N), int(K), ws, &guard)) return QSPEC_ERR_CUDA;
  if (qspec::gemv_supported(int(M), int(N), int(K)))
    return qspec::gemv(16, x, Wp, S, int(M), int(N), int(K), y, nullptr, nullptr, nullptr, ws, guard, s);
  if (qspec::linear_tc_supported(16, int(M), int(N), int(K)))
    return qspec::linear_tc(16, x, Wp, S, int(M), int(N), int(K), y, nullptr, nullptr, nullptr, ws, ws_bytes, guard,
                            s);
  return QSPEC_ERR_UNSUPPORTED_SHAPE;
}

namespace {
// The quantised-activation linears (steps a3 + a4, and the W4A8 variant): abits = 4 or 8.
qspec_status linear_quantised(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                              int64_t N, int64_t K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                              void* ws, size_t ws_bytes, qspec_stream_t stream) {
  const qspec_status st = check_linear_args(x, Wp, S, M, N, K, y);
  if (st != QSPEC_OK) return st;
  if ((xq_out && !qspec::aligned16(xq_out)) || (xs_out && !qspec::aligned16(xs_out)) ||
      (acc_out && !qspec::aligned16(acc_out)))
    return QSPEC_ERR_MISALIGNED;
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!qspec::aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_workspace_size(M, N, K)) return QSPEC_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  qspec::WsGuard guard;
  if (!qspec::make_guard(int(M), int(N), int(K), ws, &guard)) return QSPEC_ERR_CUDA;
  if (qspec::gemv_supported(int(M), int(N), int(K)))
    return qspec::gemv(abits, x, Wp, S, int(M), int(N), int(K), y, xq_out, xs_out, acc_out, ws, guard, s);
  if (qspec::linear_tc_supported(abits, int(M), int(N), int(K)))
    return qspec::linear_tc(abits, x, Wp, S, int(M), int(N), int(K), y, xq_out, xs_out, acc_out, ws, ws_bytes, guard,
                            s);
  return QSPEC_ERR_UNSUPPORTED_SHAPE;
}
}  // namespace

extern "C" qspec_status qspec_linear_w4a4(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                          int64_t M, int64_t N, int64_t K, uint16_t* y,
                                          int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws,
                                          size_t ws_bytes, qspec_stream_t stream) {
  return linear_quantised(4, x, Wp, S, M, N, K, y, xq_out, xs_out, acc_out, ws, ws_bytes, stream);
}

extern "C" qspec_status qspec_linear_w4a8(const uint16_t* x, const uint8_t* Wp, const uint16_t* S,
                                          int64_t M, int64_t N, int64_t K, uint16_t* y,
                                          int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws,
                                          size_t ws_bytes, qspec_stream_t stream) {
  return linear_quantised(8, x, Wp, S, M, N, K, y, xq_out, xs_out, acc_out, ws, ws_bytes, stream);
}

namespace {
// 16 x the parts' 16-row tiles, or -1 if a part is invalid; *st gets the status of the first
// invalid part.
int64_t group_rows(const qspec_linear_part* parts, int32_t n, int64_t K, qspec_status* st) {
  using namespace qspec;
  *st = QSPEC_OK;
  int64_t tiles = 0;
  for (int32_t i = 0; i < n; ++i) {
    const qspec_linear_part& p = parts[i];
    if (!p.Wp || !p.S || !p.y || p.N <= 0) { *st = QSPEC_ERR_INVALID_ARG; return -1; }
    if (p.N % 8 != 0 || p.N > (int64_t(1) << 30) || p.N * K >= (int64_t(1) << 40)) {
      *st = QSPEC_ERR_UNSUPPORTED_SHAPE;
      return -1;
    }
    if (!aligned16(p.Wp) || !aligned16(p.S) || !aligned16(p.y)) { *st = QSPEC_ERR_MISALIGNED; return -1; }
    tiles += (p.N + 15) / 16;
  }
  if (tiles * 16 > (int64_t(1) << 30)) { *st = QSPEC_ERR_UNSUPPORTED_SHAPE; return -1; }
  return tiles * 16;
}
}  // namespace

extern "C" size_t qspec_linear_group_workspace_size(int64_t M, const qspec_linear_part* parts, int32_t n_parts,
                                                    int64_t K) {
  if (!parts || n_parts < 1 || n_parts > QSPEC_GROUP_MAX_PARTS || M < 1 || M > QSPEC_GROUP_MAX_M || K <= 0 ||
      K % qspec::kGroup != 0)
    return 0;
  qspec_status st;
  const int64_t R = group_rows(parts, n_parts, K, &st);
  if (R < 0) return 0;
  return qspec_linear_workspace_size(M, R, K);
}

extern "C" qspec_status qspec_linear_group(int32_t abits, const uint16_t* x, int64_t M, int64_t K,
                                           const qspec_linear_part* parts, int32_t n_parts, void* ws,
                                           size_t ws_bytes, qspec_stream_t stream) {
  using namespace qspec;
  if (!x || !parts || n_parts < 1 || M <= 0 || K <= 0) return QSPEC_ERR_INVALID_ARG;
  if (abits != 4 && abits != 8 && abits != 16) return QSPEC_ERR_INVALID_ARG;
  if (n_parts > QSPEC_GROUP_MAX_PARTS || M > QSPEC_GROUP_MAX_M || K % kGroup != 0 || K > (int64_t(1) << 30))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  qspec_status st;
  const int64_t R = group_rows(parts, n_parts, K, &st);
  if (R < 0) return st;
  if (!aligned16(x)) return QSPEC_ERR_MISALIGNED;
  if (!gemv_supported(int(M), int(R), int(K))) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_workspace_size(M, R, K)) return QSPEC_ERR_WORKSPACE;
  WsGuard guard;
  if (!make_guard(int(M), int(R), int(K), ws, &guard)) return QSPEC_ERR_CUDA;
  GroupPart gp[QSPEC_GROUP_MAX_PARTS];
  for (int32_t i = 0; i < n_parts; ++i) gp[i] = GroupPart{parts[i].Wp, parts[i].S, parts[i].y, parts[i].N};
  return gemv_group(abits, x, int(M), int(K), gp, n_parts, ws, guard, reinterpret_cast<cudaStream_t>(stream));
}
