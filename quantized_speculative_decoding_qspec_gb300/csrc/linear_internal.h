// Internal interface between the linear entry points and their kernel families.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qspec.h"

namespace qspec {

// abits: activation width of the mode -- 16 (W4A16), 4 (W4A4) or 8 (W4A8).

// The linear workspace starts with a header of kWsHeader bytes.  Its first 64-bit word records the
// layout (M, N, K) of the calls that use the workspace's regions: a kernel that writes tickets,
// partial sums or codes there first claims the word (0 -> tag, or already tag) and, when it holds
// another shape's tag, skips all its work and sets kErrWorkspace in the error word.
constexpr size_t kWsHeader = 256;
struct WsGuard {
  unsigned long long* hdr;  // device address of the header word
  unsigned long long tag;   // this call's layout tag (never 0)
  unsigned int* err;        // device address of the linear error word (current context)
};
enum : unsigned int { kErrTimeout = 1u, kErrWorkspace = 2u };
// The tickets of the tensor-core kernels (split tiles) follow the header.  They must read zero when a
// kernel starts (each kernel resets the ones it used), so both kernels keep them in one region of
// this many words -- enough for 128-row tiles of 16 tokens, the finest split either kernel uses --
// and place their other regions after it.
inline long long tc_ticket_count(int M, int N) {
  return (static_cast<long long>(N) + 127) / 128 * ((static_cast<long long>(M) + 15) / 16);
}
unsigned long long ws_tag(int M, int N, int K);
// Device address of the linear error word in the current CUDA context (looked up once per context).
unsigned int* linear_error_word();

// Claims the workspace for this call's layout (one thread); true if the call may use it.
__device__ __forceinline__ bool ws_claim(const WsGuard& g) {
  const unsigned long long old = atomicCAS(g.hdr, 0ull, g.tag);
  if (old == 0ull || old == g.tag) return true;
  atomicOr(g.err, kErrWorkspace);
  return false;
}

// Tensor-core W4A16 kernel that dequantises the weights on chip (linear_dq.cu), for kDqMinTokens
// tokens or more (fewer run on the exact-code kernel, which measured faster there): the shapes for
// which linear_dq_supported() is true.
constexpr int kDqMinTokens = 65;
bool linear_dq_supported(int M, int N, int K);
size_t linear_dq_workspace_size(int M, int N, int K);
qspec_status linear_dq(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K, uint16_t* y,
                       void* ws, size_t ws_bytes, const WsGuard& guard, cudaStream_t stream);

// Tensor-core (tcgen05) kernels: the shapes for which linear_tc_supported() is true (W4A16 from
// kDqMinTokens tokens on runs on linear_dq, everything else on the exact-code kernel of
// linear_tc.cu).
bool linear_tc_supported(int abits, int M, int N, int K);
size_t linear_tc_workspace_size(int abits, int M, int N, int K);
qspec_status linear_tc(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M,
                       int N, int K, uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out,
                       void* ws, size_t ws_bytes, const WsGuard& guard, cudaStream_t stream);

// The per-token quantiser as its own kernel (one CTA per token): codes [M, K] and fp32 scales [M],
// plus the optional int8 codes and scales out.  The codes are bf16 for the tensor-core path; with
// gemv_layout they are the GEMV's staged fp16 chunks (elements 2, 3, 6, 7 of each 8 divided by 16).  ws_codes gives the workspace's code and scale
// buffers for a quantised mode (false for W4A16).
qspec_status quantise_tokens(int abits, const uint16_t* x, int M, int K, bool gemv_layout, uint16_t* codes,
                             float* s_a, int8_t* xq_out, float* xs_out, const WsGuard& guard, cudaStream_t stream);
bool ws_codes(int abits, int M, int N, int K, void* ws, uint16_t** codes, float** s_a);

// The largest tensor-core workspace over the three modes for one shape (the GEMV's own regions
// follow it).
size_t linear_tc_workspace_size_all(int M, int N, int K);

// Register-fragment MMA GEMV for every mode at decode sizes (M <= 32; K is split into chunks
// across CTAs when the staged activations of all K do not fit shared memory).
bool gemv_supported(int M, int N, int K);
size_t gemv_workspace_bytes(int M, int N, int K);  // beyond linear_tc_workspace_size_all
qspec_status gemv(int abits, const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int M, int N, int K,
                  uint16_t* y, int8_t* xq_out, float* xs_out, int32_t* acc_out, void* ws, const WsGuard& guard,
                  cudaStream_t stream);

// One weight matrix of a group that reads the same activations (qspec_linear_group).
struct GroupPart {
  const uint8_t* Wp;
  const uint16_t* S;
  uint16_t* y;
  int64_t N;
};
// The GEMV over a group of parts as one run of 16-row tiles; the planners and the workspace see
// gemv_group_rows(N, n) rows (16 x the parts' tiles).
int gemv_group_rows(const int64_t* N, int n);
qspec_status gemv_group(int abits, const uint16_t* x, int M, int K, const GroupPart* parts, int n, void* ws,
                        const WsGuard& guard, cudaStream_t stream);

// A 2-D tensor map for TMA loads (dims {inner, outer} elements of type dt, row pitch row_bytes, box
// {box_inner, box_outer}, 128-byte swizzle or none); out-of-range boxes read as zeros.  False if the
// driver offers no encoder or rejects the arguments.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

// Reads (synchronously) and clears the error bits the linear kernels set on the current device.
qspec_status read_and_clear_linear_error(cudaStream_t stream, unsigned int* bits);

}  // namespace qspec
