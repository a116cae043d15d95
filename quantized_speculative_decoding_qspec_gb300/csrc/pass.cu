// Entry point of the linear pass (pass_impl.cuh): argument checks and the launch plan -- warps per
// tile and rounds of every layer, the rotation of the CTA order, and where each layer's staged
// activations live in the shared-memory ring.
#include "pass_impl.cuh"

namespace qspec {
using namespace pass_impl;

namespace {

constexpr int kArenaChunks = kArenaBytes / 16;
constexpr int kSegChunks = 64 * 1024 / 16;  // staged activations of one segment (unless one layer needs more)

int pass_slots(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }

// Warps per tile (K split among them): the fewest rounds x (groups per slice + fixed cost) over the
// whole grid, ties to the smaller split; slices must hold a multiple of D groups.
int pick_ks(int tiles, int G, int P, int D) {
  int best_ks = 0;
  long long best = -1;
  for (int ks = 1; ks <= kWarps; ks *= 2) {
    if (G % ks != 0 || (G / ks) % D != 0) continue;
    const long long slots = static_cast<long long>(P) * (kWarps / ks);
    const long long rounds = (tiles + slots - 1) / slots;
    const long long cost = rounds * (G / ks + 2);
    if (best < 0 || cost < best) {
      best = cost;
      best_ks = ks;
    }
  }
  return best_ks;
}

// One CTA per SM (the kernel's shared memory admits no second one), and every CTA must be resident
// at once: the grid barrier waits for all of them.
int pass_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
  return sms;
}

qspec_status check_layer(const qspec_pass_layer& d, int MT) {
  if (!d.x || !d.Wp || !d.S || !d.y) return QSPEC_ERR_INVALID_ARG;
  if (d.N <= 0 || d.K <= 0 || d.reserved != 0) return QSPEC_ERR_INVALID_ARG;
  if (d.N % 8 != 0 || d.K % kGroup != 0 || d.N > (int64_t(1) << 30) || d.N * d.K >= (int64_t(1) << 40))
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(MT) * d.K / 8 > kArenaChunks) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(d.x) || !aligned16(d.Wp) || !aligned16(d.S) || !aligned16(d.y)) return QSPEC_ERR_MISALIGNED;
  return QSPEC_OK;
}

}  // namespace
}  // namespace qspec

extern "C" size_t qspec_linear_pass_workspace_size(void) { return 256; }

extern "C" qspec_status qspec_linear_pass(int32_t abits, int64_t M, const qspec_pass_layer* layers, int32_t n_layers,
                                          void* ws, size_t ws_bytes, qspec_stream_t stream) {
  using namespace qspec;
  if (!layers || n_layers <= 0 || M <= 0) return QSPEC_ERR_INVALID_ARG;
  if (abits != 4 && abits != 8 && abits != 16) return QSPEC_ERR_INVALID_ARG;
  if (n_layers > QSPEC_PASS_MAX_LAYERS || M > QSPEC_PASS_MAX_M) return QSPEC_ERR_UNSUPPORTED_SHAPE;
  const int MT = pass_slots(static_cast<int>(M));
  for (int l = 0; l < n_layers; ++l) {
    const qspec_status st = check_layer(layers[l], MT);
    if (st != QSPEC_OK) return st;
  }
  if (!ws) return QSPEC_ERR_WORKSPACE;
  if (!aligned16(ws)) return QSPEC_ERR_MISALIGNED;
  if (ws_bytes < qspec_linear_pass_workspace_size()) return QSPEC_ERR_WORKSPACE;
  const int P = pass_ctas();
  if (P <= 0) return QSPEC_ERR_CUDA;

  // four groups in flight per warp when every layer's group count allows it, else one
  int D = 4;
  for (int l = 0; l < n_layers; ++l)
    if ((layers[l].K / kGroup) % 4 != 0) D = 1;

  Params prm = {};
  prm.M = static_cast<int>(M);
  prm.bar = static_cast<unsigned int*>(ws);
  prm.err = linear_error_word();
  if (!prm.err) return QSPEC_ERR_CUDA;
  // Segments: runs of consecutive layers with the same K, no barrier inside and at most
  // kSegChunks of staged activations (a single larger layer is a segment of its own).
  int n_seg = 0;
  for (int l = 0; l < n_layers; ++l) {
    const qspec_pass_layer& d = layers[l];
    const int len = MT * static_cast<int>(d.K) / 8;
    Segment* S = n_seg > 0 ? &prm.Sg[n_seg - 1] : nullptr;
    const bool join = S && !d.after && S->K == static_cast<int>(d.K) && (S->nl + 1) * len <= kSegChunks;
    if (!join) {
      S = &prm.Sg[n_seg++];
      *S = Segment{};
      S->l0 = l;
      S->K = static_cast<int>(d.K);
      S->flags = d.after ? kFlagBarrier : 0;
    }
    Layer& L = prm.L[l];
    L.x = d.x;
    L.Wp = d.Wp;
    L.S = reinterpret_cast<const __half*>(d.S);
    L.y = d.y;
    L.N = static_cast<int>(d.N);
    L.K = static_cast<int>(d.K);
    L.vt0 = S->tiles;
    L.act_len = len;
    S->tiles += (L.N + 15) / 16;
    ++S->nl;
  }
  prm.n_seg = n_seg;
  // The staged activations: a ring just large enough for every segment and for each pair of
  // consecutive segments that may be staged together (no barrier between them); consecutive
  // segments sit at opposite ends of it, so the next segment's copy never lands on the one read.
  auto seg_len = [&](const Segment& S) { return S.nl * MT * S.K / 8; };
  int arena = 0;
  for (int i = 0; i < n_seg; ++i) {
    arena = std::max(arena, seg_len(prm.Sg[i]));
    if (i > 0 && !(prm.Sg[i].flags & kFlagBarrier)) {
      const int pair = seg_len(prm.Sg[i]) + seg_len(prm.Sg[i - 1]);
      if (pair <= kArenaChunks) arena = std::max(arena, pair);
    }
  }
  prm.arena_chunks = arena;
  prm.corr_floats = 0;
  for (int i = 0; i < n_seg; ++i)
    prm.corr_floats = std::max(prm.corr_floats, prm.Sg[i].nl * (prm.Sg[i].K / kGroup) * MT);
  int rot = 0;
  for (int i = 0; i < n_seg; ++i) {
    Segment& S = prm.Sg[i];
    const int G = S.K / kGroup;
    S.KS = pick_ks(S.tiles, G, P, D);
    if (S.KS == 0) return QSPEC_ERR_UNSUPPORTED_SHAPE;
    S.gs = G / S.KS;
    const int per_cta = kWarps / S.KS;
    S.rounds = (S.tiles + P * per_cta - 1) / (P * per_cta);
    // after a barrier every CTA starts together; otherwise start on the CTAs the previous one left
    if (S.flags & kFlagBarrier) rot = 0;
    S.rot = rot;
    const int busy = static_cast<int>(std::min<long long>(P, (S.tiles + per_cta - 1) / per_cta));
    rot = ((rot - busy) % P + P) % P;
    int off = (i % 2 == 0) ? 0 : arena - seg_len(S);
    for (int l = S.l0; l < S.l0 + S.nl; ++l) {
      prm.L[l].act_off = off;
      off += prm.L[l].act_len;
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (abits) {
    case 4: return pass_impl::launch_pass_mode<4>(MT, D, prm, P, s);
    case 8: return pass_impl::launch_pass_mode<8>(MT, D, prm, P, s);
    default: return pass_impl::launch_pass_mode<0>(MT, D, prm, P, s);
  }
}
