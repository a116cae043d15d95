// Step a1: symmetric per-group INT4 weight quantiser and packer.
//
// QSpec article ("QSpec実行時の2つの量子化による推論の一致率を調べる", section
// "QSpec の W4A4 モードと W4A16 モード"): one 4-bit weight set is shared by the draft (W4A4) and
// the verify (W4A16) mode.  The quantiser is the plain symmetric one, per group of 128 input
// channels: s = fp16(amax / 7), code = clamp(rint(w / s), -8, 7), codes 0 when s == 0.
//
// Packed layout: each 32-bit little-endian word holds 8 consecutive channels k = 8t..8t+7 as two's
// complement nibbles, the even channels (8t+0, 2, 4, 6) in nibbles 0..3 and the odd ones
// (8t+1, 3, 5, 7) in nibbles 4..7, so that a shift and a mask bring any (even, odd) channel pair to
// the low bits of the two half-words (the pages fix no bit order; this one suits the converters).
//
// Launch shape: a half-warp per group (8 bf16 = one 16-byte load per lane), two groups per warp.
// A row of W is K contiguous bf16 and K % 128 == 0, so group q covers the flat elements
// [128q, 128q + 128) of W, the flat bytes [64q, 64q + 64) of Wp and the flat entry q of S.
// HBM-bound: 2 bytes read and 0.5 + 1/64 bytes written per weight.
#include "common.cuh"

namespace qspec {
namespace {

__global__ void __launch_bounds__(256) pack_weights_kernel(const uint16_t* __restrict__ W,
                                                           uint8_t* __restrict__ Wp,
                                                           __half* __restrict__ S,
                                                           int64_t n_groups) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t q = warp * 2 + (lane >> 4);
  const int j = lane & 15;
  const bool valid = q < n_groups;

  uint4 v = make_uint4(0, 0, 0, 0);
  if (valid) v = ld_stream_v4(W + q * kGroup + 8 * j);
  const uint32_t w[8] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16,
                         v.z & 0xFFFFu, v.z >> 16, v.w & 0xFFFFu, v.w >> 16};

  // amax over the group: for non-negative floats the bit pattern orders like the value.
  uint32_t amax_bits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax_bits = max(amax_bits, w[i] & 0x7FFFu);
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1)
    amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, off));

  const float amax = __uint_as_float(amax_bits << 16);
  const __half s = __float2half_rn(__fdiv_rn(amax, 7.0f));
  const float sf = __half2float(s);

  uint32_t packed = 0;
  if (sf != 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float c = rintf(__fdiv_rn(__uint_as_float(w[i] << 16), sf));
      c = fminf(fmaxf(c, -8.0f), 7.0f);
      // channel 8j + i goes to nibble (i >> 1) + 4 (i & 1): even channels in the low half-word
      packed |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xFu) << (4 * ((i >> 1) + 4 * (i & 1)));
    }
  }
  if (valid) {
    reinterpret_cast<uint32_t*>(Wp + q * (kGroup / 2))[j] = packed;
    if (j == 0) S[q] = s;
  }
}

}  // namespace
}  // namespace qspec

extern "C" qspec_status qspec_pack_weights(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wp,
                                           uint16_t* S, qspec_stream_t stream) {
  using namespace qspec;
  if (!W || !Wp || !S) return QSPEC_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0) return QSPEC_ERR_INVALID_ARG;
  if (K % kGroup != 0 || N * K >= (int64_t(1) << 40)) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W) || !aligned16(Wp) || !aligned16(S)) return QSPEC_ERR_MISALIGNED;
  const int64_t n_groups = N * (K / kGroup);
  const int64_t blocks = (n_groups + 15) / 16;  // 8 warps x 2 groups per block
  pack_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      W, Wp, reinterpret_cast<__half*>(S), n_groups);
  return launch_status();
}
