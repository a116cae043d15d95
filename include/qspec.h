/*
 * qspec.h -- C ABI of libqspec.so, the GB300 (sm_103a) hot path of QSpec-style quantized
 * speculative decoding.
 *
 * The method (QSpec, as described in "QSpec実行時の2つの量子化による推論の一致率を調べる",
 * qiita.com/joule, sections "W4A4 と W4A16 量子化" and "QSpec の W4A4 モードと W4A16 モード"):
 * one set of 4-bit weights serves two modes.  The draft mode (W4A4) also quantises activations
 * to 4 bits; the verify mode (W4A16) keeps 16-bit activations and converts the 4-bit weights while
 * multiplying.  Drafted tokens are then checked against the verify-mode distribution with the
 * standard speculative-decoding rules ("Speculative Decodingとは？LLM生成を速くする方法",
 * kasblo.com, sections "greedy decodingでは一致するprefixを採用する" and
 * "samplingでもtargetの確率分布を保つ", eqs. a(x) and p'(x)).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major and contiguous.
 *    bfloat16 and float16 tensors are passed as uint16_t bit patterns.
 *  - Every base pointer must be 16-byte aligned (QSPEC_ERR_MISALIGNED otherwise).
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default stream).  No entry point
 *    synchronises except qspec_check_status, and none allocates or frees device memory.
 *  - Argument checks happen on the host before anything is enqueued; on failure nothing is
 *    enqueued and the status says why.  Launch failures return QSPEC_ERR_CUDA.
 *  - Outputs must not alias inputs.
 *  - Calls are thread-safe.  Calls that share a verify workspace must not overlap on the GPU.
 */
#ifndef QSPEC_H_
#define QSPEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* same type as cudaStream_t */
typedef struct CUstream_st* qspec_stream_t;

typedef enum {
  QSPEC_OK = 0,
  QSPEC_ERR_INVALID_ARG = 1,        /* null pointer, negative or zero size, bad token id        */
  QSPEC_ERR_UNSUPPORTED_SHAPE = 2,  /* size outside the documented limits                        */
  QSPEC_ERR_MISALIGNED = 3,         /* a base pointer is not 16-byte aligned                     */
  QSPEC_ERR_WORKSPACE = 4,          /* workspace missing, too small, or laid out for another shape */
  QSPEC_ERR_CUDA = 5,               /* a CUDA runtime/driver call or a launch failed             */
  QSPEC_ERR_TIMEOUT = 6             /* a kernel gave up a bounded wait and returned early        */
} qspec_status;

/* Limits checked by every call. */
#define QSPEC_GROUP 128             /* input channels per weight scale                           */
#define QSPEC_MAX_M 4096            /* tokens per linear call                                    */
#define QSPEC_MAX_GAMMA 16          /* draft length                                              */
#define QSPEC_MAX_V (1 << 24)       /* vocabulary                                                */
#define QSPEC_MAX_TREE 64           /* candidate nodes of a verification tree                    */

/*
 * qspec_pack_weights -- symmetric per-group INT4 weight quantiser and packer (step a1).
 *
 * The pages fix only "4-bit weights shared by both modes" (QSpec article, section
 * "QSpec の W4A4 モードと W4A16 モード"); the quantiser is the plain symmetric one:
 * for each row n and group g of 128 consecutive input channels,
 *     s[n,g]    = fp16( amax_g |W| / 7 )                   (fp32 IEEE division, round to fp16)
 *     code[n,k] = clamp( rint( W[n,k] / float(s[n,g]) ), -8, 7 )   (fp32 IEEE division, ties even)
 * with all codes 0 when s == 0.  Codes are two's complement nibbles; the 32-bit little-endian word
 * t of row n (bytes Wp[n, 4t..4t+3]) holds channels k = 8t..8t+7 with the even channels
 * 8t+0, 2, 4, 6 in nibbles 0..3 (bits 0..15) and the odd channels 8t+1, 3, 5, 7 in nibbles 4..7
 * (bits 16..31).  This packed format is the format both linear calls read.
 *
 *   W   [N, K] bf16 (input), K % 128 == 0, 1 <= N, N*K < 2^40
 *   Wp  [N, K/2] uint8 (output)
 *   S   [N, K/128] fp16 (output)
 * The result is bit-exact (independent of launch configuration).
 */
qspec_status qspec_pack_weights(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wp, uint16_t* S,
                                qspec_stream_t stream);

/*
 * qspec_linear_w4a16 -- verify-mode linear (step a2): y = x . dequant(Wp, S)^T.
 *
 * QSpec article, section "W4A16: 重みのみを 4-bit に量子化": 4-bit weights are converted to
 * 16-bit values during the product with 16-bit activations.
 *     y[m,n] = sum_k x[m,k] * code[n,k] * s[n, k/128]
 * The codes are converted to bf16 exactly, products of each 128-channel group are summed in fp32
 * and scaled by s[n,g]; y is rounded to bf16 once.
 *
 *   x  [M, K] bf16, Wp [N, K/2] uint8, S [N, K/128] fp16 (from qspec_pack_weights)
 *   y  [M, N] bf16 (output)
 *   ws, ws_bytes  device workspace, >= qspec_linear_workspace_size(M, N, K), zero-filled before its
 *                 first use; it holds the per-tile tickets and partial sums of output tiles whose K
 *                 range is split between SMs, and the W4A4 activation codes.  A call leaves the
 *                 workspace ready for the next call OF THE SAME (M, N, K); its layout depends on the
 *                 shape, so calls of different shapes (for instance the layers of a model) need
 *                 workspaces of their own, or a zero-fill in between.  The workspace's header records
 *                 the (M, N, K) of the first call that uses its regions; a later call of another shape
 *                 that would use them touches neither the workspace nor y and makes the next
 *                 qspec_check_status return QSPEC_ERR_WORKSPACE.  (Calls whose kernels use no region,
 *                 such as one to three tokens on the decode-size path when K fits on chip, run on
 *                 any large-enough workspace.)
 *   1 <= M <= 4096, N % 8 == 0, K % 128 == 0; QSPEC_ERR_UNSUPPORTED_SHAPE for the (very large)
 *   shapes whose tensor-core work units would not fit 32-bit counters, and QSPEC_ERR_CUDA if the
 *   driver offers no tensor-map encoder (there is no other path).
 * The fp32 summation order depends on the device's SM count, so results are reproducible on one
 * device but may differ in the last bits between devices.
 */
qspec_status qspec_linear_w4a16(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                                int64_t N, int64_t K, uint16_t* y, void* ws, size_t ws_bytes,
                                qspec_stream_t stream);

/*
 * qspec_linear_w4a4 -- draft-mode linear (steps a3 + a4) with the activation quantiser fused.
 *
 * QSpec article, section "W4A4 : 重みと活性値の両方を 4-bit に量子化": activations are also
 * quantised to 4 bits, so the product runs on 4-bit operands.  Per token m (all of K):
 *     s_a[m]    = amax_k |x[m,k]| / 7                     (fp32 IEEE division, kept in fp32)
 *     qa[m,k]   = clamp( rint( x[m,k] / s_a[m] ), -8, 7 ) (fp32 IEEE division, ties even; 0 if s_a==0)
 *     acc[m,n,g]= sum_{k in group g} qa[m,k] * code[n,k]  (exact integer)
 *     y[m,n]    = s_a[m] * sum_g float(s[n,g]) * acc[m,n,g]   (fp32, rounded to bf16 once)
 *
 *   x, Wp, S, y, M, N, K, ws, ws_bytes as for qspec_linear_w4a16 (the SAME Wp and S serve both modes).
 *   xq_out  [M, K] int8 codes qa, or NULL              (bit-exact)
 *   xs_out  [M] fp32 scales s_a, or NULL               (bit-exact)
 *   acc_out [M, N, K/128] int32 group sums, or NULL    (bit-exact; debugging aid)
 */
qspec_status qspec_linear_w4a4(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                               int64_t N, int64_t K, uint16_t* y, int8_t* xq_out, float* xs_out,
                               int32_t* acc_out, void* ws, size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_linear_w4a8 -- the W4A8 configuration (step f3): qspec_linear_w4a4 with 8-bit activations.
 *
 * The speculative-decoding-with-quantisation summary (aibr.jp), section "中核となる技術的要素",
 * names W4A8 beside W4A16 as a weight/activation configuration; it gives no quantiser, so this one
 * is the W4A4 quantiser at 8 bits, on the same packed 4-bit weights:
 *     s_a[m]    = amax_k |x[m,k]| / 127                     (fp32 IEEE division, kept in fp32)
 *     qa[m,k]   = clamp( rint( x[m,k] / s_a[m] ), -128, 127 ) (fp32 IEEE division, ties even)
 *     acc, y    as for qspec_linear_w4a4 (|acc| <= 131072: exact)
 *   Arguments, outputs and limits as qspec_linear_w4a4.
 */
qspec_status qspec_linear_w4a8(const uint16_t* x, const uint8_t* Wp, const uint16_t* S, int64_t M,
                               int64_t N, int64_t K, uint16_t* y, int8_t* xq_out, float* xs_out,
                               int32_t* acc_out, void* ws, size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_linear_group -- several linears that read the same activations, in one launch and one mode
 * (steps a2, a3 + a4, or the W4A8 configuration of f3): e.g. the q, k and v projections of a
 * decoder layer, or its gate and up projections.
 *
 * QSpec article, section "QSpec の W4A4 モードと W4A16 モード": both modes read the same packed weights.
 * Part i computes exactly what qspec_linear_w4a16 / _w4a4 / _w4a8 compute for (x, Wp_i, S_i):
 *     y_i = x . dequant(Wp_i, S_i)^T          (abits = 16)
 *     y_i = s_a . sum_g s . acc               (abits = 4 or 8, x quantised once per token)
 * with the same definitions and tolerances (the fp32 summation order may differ in the last bits).
 * The parts' rows stream as one run of 16-row tiles, so the launch, the activation staging and the
 * per-token quantisation are paid once for the group.
 *
 *   abits     16 (W4A16), 4 (W4A4) or 8 (W4A8)
 *   x         [M, K] bf16, 1 <= M <= QSPEC_GROUP_MAX_M, K % 128 == 0
 *   parts     HOST array of n_parts descriptors, 1 <= n_parts <= QSPEC_GROUP_MAX_PARTS; each:
 *               Wp [N, K/2] uint8, S [N, K/128] fp16 (from qspec_pack_weights), y [M, N] bf16
 *               (output), N % 8 == 0; read during the call
 *   ws, ws_bytes  device workspace, >= qspec_linear_group_workspace_size(M, parts, n_parts, K),
 *             zero-filled before its first use; its header records the layout as (M, R, K), R = 16
 *             x the parts' 16-row tiles (QSPEC_ERR_WORKSPACE for a workspace laid out otherwise)
 * Shapes the decode-size kernel does not serve return QSPEC_ERR_UNSUPPORTED_SHAPE (call the parts
 * one by one then).
 */
#define QSPEC_GROUP_MAX_PARTS 4
#define QSPEC_GROUP_MAX_M 4
typedef struct {
  const uint8_t* Wp;
  const uint16_t* S;
  uint16_t* y;
  int64_t N;
} qspec_linear_part;
size_t qspec_linear_group_workspace_size(int64_t M, const qspec_linear_part* parts, int32_t n_parts, int64_t K);
qspec_status qspec_linear_group(int32_t abits, const uint16_t* x, int64_t M, int64_t K, const qspec_linear_part* parts,
                                int32_t n_parts, void* ws, size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_linear_pass -- one launch for a pass of decode-size linears in one mode (steps a2, a3 + a4,
 * or the W4A8 configuration of f3), e.g. every linear of a decoder layer and the lm_head.
 *
 * QSpec article, section "QSpec の W4A4 モードと W4A16 モード": a draft pass runs every linear of
 * the model in W4A4 mode and a verify pass runs them in W4A16 mode, over the same packed weights.
 * Each layer l of the pass computes exactly what qspec_linear_w4a16 / _w4a4 / _w4a8 compute for it
 * (same definitions, same tolerances; the fp32 summation order may differ in the last bits):
 *     y_l = x_l . dequant(Wp_l, S_l)^T          (abits = 16)
 *     y_l = s_a . sum_g s . acc                  (abits = 4 or 8, x_l quantised per token)
 * The layers run in order on one persistent grid (one CTA per SM): the weight stream continues
 * across layer boundaries and the next layer's activations are copied on chip while the current
 * layer streams.  A layer with `after` set reads what earlier layers of the pass wrote: every CTA
 * finishes the earlier layers and waits for all others (a grid-wide barrier with an iteration limit;
 * if it expires, the pass stops and qspec_check_status returns QSPEC_ERR_TIMEOUT).  Without `after`,
 * a layer's x must not be the y of an earlier layer of the same pass.
 *
 *   abits     16 (W4A16), 4 (W4A4) or 8 (W4A8)
 *   M         tokens, 1 <= M <= QSPEC_PASS_MAX_M (the same for every layer)
 *   layers    HOST array of n_layers descriptors, 1 <= n_layers <= QSPEC_PASS_MAX_LAYERS; each:
 *               x [M, K] bf16, Wp [N, K/2] uint8, S [N, K/128] fp16 (from qspec_pack_weights),
 *               y [M, N] bf16 (output); N % 8 == 0, K % 128 == 0, and the staged activations must
 *               fit on chip: slots(M) * K <= 102400 with slots(M) = 1, 2, 4 for M = 1, 2, 3..4
 *               (K <= 25600 at M = 4); `reserved` must be 0
 *   ws, ws_bytes  device workspace of >= qspec_linear_pass_workspace_size() bytes, zero-filled
 *             before its first use (it holds the grid barrier's counters, which every pass leaves
 *             ready for the next); passes that share a workspace must not overlap on the GPU
 * The descriptors are read during the call (they may be reused or freed when it returns).
 */
#define QSPEC_PASS_MAX_LAYERS 16
#define QSPEC_PASS_MAX_M 4
typedef struct {
  const uint16_t* x;
  const uint8_t* Wp;
  const uint16_t* S;
  uint16_t* y;
  int64_t N, K;
  int32_t after;     /* nonzero: this layer reads outputs of earlier layers of the pass */
  int32_t reserved;  /* must be 0 */
} qspec_pass_layer;
size_t qspec_linear_pass_workspace_size(void);
qspec_status qspec_linear_pass(int32_t abits, int64_t M, const qspec_pass_layer* layers, int32_t n_layers,
                               void* ws, size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_linear_workspace_size -- bytes of device workspace the linear calls need for an [M, K] x
 * [N, K] product on the CURRENT device (the size depends on its SM count).  0 for invalid sizes.
 */
size_t qspec_linear_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * qspec_verify_workspace_size -- bytes of device workspace that the verify calls need for the
 * given shape.  The workspace must be zero-filled before its first use (e.g. one cudaMemset
 * after allocation); every call leaves it ready for the next call.  Returns 0 for invalid sizes.
 */
size_t qspec_verify_workspace_size(int32_t B, int32_t gamma, int32_t V);

/*
 * qspec_verify_greedy -- greedy verification (steps a5 + a6).
 *
 * Tutorial, section "greedy decodingでは一致するprefixを採用する": draft tokens are compared left
 * to right with the target's most likely token; the matching prefix is accepted, the first
 * mismatching position takes the target's token instead, and when every draft token matches the
 * target's token for the following position is added (at most gamma+1 tokens per call).
 *     t[b,i] = argmax_j tgt_logits[b,i,j]    (lowest index among equal maxima; +0 == -0)
 *     n[b]   = largest k <= gamma with d[b,i] == t[b,i] for all i < k
 *     out[b] = (d[b,0..n-1], t[b,n], -1, ...)
 *
 *   tgt_logits [B, gamma+1, V] bf16   target logits at the gamma draft positions and the next one
 *   draft_tok  [B, gamma] int32       draft tokens; ids outside [0, V) never match and raise
 *                                     QSPEC_ERR_INVALID_ARG at the next qspec_check_status
 *   accept_len [B] int32 (output)     n
 *   out_tok    [B, gamma+1] int32 (output)
 *   tgt_argmax [B, gamma+1] int32 (output) or NULL
 *   ws, ws_bytes                      device workspace, >= qspec_verify_workspace_size(B,gamma,V)
 *   1 <= B, 1 <= gamma <= 16, 2 <= V <= 2^24, B*(gamma+1)*V < 2^40.  Bit-exact.
 */
qspec_status qspec_verify_greedy(const uint16_t* tgt_logits, const int32_t* draft_tok, int32_t B,
                                 int32_t gamma, int32_t V, int32_t* accept_len, int32_t* out_tok,
                                 int32_t* tgt_argmax, void* ws, size_t ws_bytes,
                                 qspec_stream_t stream);

/*
 * qspec_verify_sample -- sampling verification (steps a5, a7, a8).
 *
 * Tutorial, section "samplingでもtargetの確率分布を保つ": with p the target distribution and q the
 * draft distribution (softmax of the logits, temperature 1, computed in fp32), draft token x at
 * position i is accepted with probability a(x) = min(1, p(x)/q(x)) (eq. a(x)); at the first
 * rejection n the emitted token is drawn from the residual max(0, p - q) / sum(...) (eq. p'(x));
 * when all gamma are accepted a bonus token is drawn from the target distribution at position
 * gamma.  The library draws no random numbers; the uniforms are inputs:
 *     accept position i      iff  u_accept[b,i] < a_i          (a_i = 1 when q(x) == 0)
 *     n[b]                   = first rejected position, or gamma
 *     j*                     = smallest j with sum_{i<=j} r_i > u_resample[b,n] * sum(r)
 *                              (r = residual of row n, or p of row gamma; r = p if sum is 0)
 *     out[b]                 = (d[b,0..n-1], j*, -1, ...)
 *
 *   tgt_logits   [B, gamma+1, V] bf16;  draft_logits [B, gamma, V] bf16;  draft_tok [B, gamma]
 *   u_accept     [B, gamma] fp32 in [0,1);  u_resample [B, gamma+1] fp32 in [0,1)
 *   accept_len [B], out_tok [B, gamma+1] int32 (outputs)
 *   accept_prob, p_tok, q_tok  [B, gamma] fp32 (outputs) or NULL: a_i, p_i(d_i), q_i(d_i) at every
 *                              draft position (also those after the first rejection)
 *   ws, ws_bytes as for qspec_verify_greedy.  Same size limits.
 */
qspec_status qspec_verify_sample(const uint16_t* tgt_logits, const uint16_t* draft_logits,
                                 const int32_t* draft_tok, const float* u_accept,
                                 const float* u_resample, int32_t B, int32_t gamma, int32_t V,
                                 int32_t* accept_len, int32_t* out_tok, float* accept_prob,
                                 float* p_tok, float* q_tok, void* ws, size_t ws_bytes,
                                 qspec_stream_t stream);

/*
 * qspec_verify_top1 -- top-1 statistics of the two modes at every draft position (step f2).
 *
 * Article "QSpec実行時の2つの量子化による推論の一致率を調べる", sections "実験：W4A4 と W4A16 の
 * Top-1 一致率を調べる" and "結果": at each draft position the W4A4 (draft) and W4A16 (target) modes
 * each have a most likely token and a probability for it (their own top-1; the two may differ).
 * The article reports how often the two tokens agree, each mode's mean top-1 probability, and the
 * agreement inside the region where both probabilities exceed 0.8 and where both are at most 0.8.
 *     tgt_top1[b,i]   = argmax_j tgt_logits[b,i,j]     (i < gamma; lowest index among equal maxima)
 *     draft_top1[b,i] = argmax_j draft_logits[b,i,j]
 *     tgt_p1[b,i]     = 1 / sum_j exp(tgt_logits[b,i,j] - max_j tgt_logits[b,i,j])   (fp32 softmax)
 *     draft_p1[b,i]   likewise for the draft row
 *
 *   tgt_logits   [B, gamma+1, V] bf16 (row gamma is not read);  draft_logits [B, gamma, V] bf16
 *   tgt_top1, draft_top1 [B, gamma] int32 (outputs)
 *   tgt_p1, draft_p1     [B, gamma] fp32 (outputs) or NULL
 *   high                 threshold of the high-confidence region (the article uses 0.8); not NaN
 *   tally                [8] fp64 or NULL: ACCUMULATED (added to, never cleared) over calls, so a
 *                        decode loop can keep one running tally on the device:
 *                        [0] positions, [1] agreeing positions, [2] positions with both p1 > high,
 *                        [3] agreeing among [2], [4] positions with both p1 <= high, [5] agreeing
 *                        among [4], [6] sum of tgt_p1, [7] sum of draft_p1.  Counts are exact; the
 *                        sums are fp64 sums of the fp32 probabilities in an unspecified order.
 *   ws, ws_bytes as for qspec_verify_greedy.  Same size limits.  Token ids are bit-exact;
 *   probabilities carry the fp32 softmax's rounding (within 1e-5 absolute of the exact value).
 */
qspec_status qspec_verify_top1(const uint16_t* tgt_logits, const uint16_t* draft_logits, int32_t B,
                               int32_t gamma, int32_t V, int32_t* tgt_top1, int32_t* draft_top1,
                               float* tgt_p1, float* draft_p1, float high, double* tally, void* ws,
                               size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_verify_tree_greedy -- greedy verification of a tree of candidates (step f4).
 *
 * The speculative-decoding-with-quantisation summary (aibr.jp), sections "先行研究との差別化
 * ポイント" and "中核となる技術的要素", names tree-style verification (candidates expanded as a tree;
 * its cost grows exponentially with the tree) without giving an algorithm.  This is the greedy rule
 * of qspec_verify_greedy carried over from a chain to a tree: node j (j < T) holds token
 * tree_tok[b,j] and parent tree_parent[b,j] (-1: the committed prefix; otherwise an earlier node,
 * parent < j).  Target row 0 scores the token after the prefix, row j + 1 the token after node j.
 *     t[r]  = argmax_v tgt_logits[b,r,v]                 (lowest index among equal maxima)
 *     walk: cur = prefix (row 0); while some child j of cur has tree_tok[b,j] == t[row of cur]:
 *           accept the lowest-index such j, cur = j (row j + 1)
 *     out[b] = (tokens of the accepted path, t[row where the walk stopped], -1, ...)
 * A chain (parent j - 1) reproduces qspec_verify_greedy.
 *
 *   tgt_logits   [B, T+1, V] bf16;  tree_tok, tree_parent [B, T] int32
 *   accept_len   [B] int32 (output) -- accepted nodes (depth of the path)
 *   out_tok      [B, T+1] int32 (output);  accept_nodes [B, T] int32 (output, node ids, -1 fill) or NULL
 *   ws, ws_bytes device workspace, >= qspec_verify_tree_workspace_size(B, T, V), zero-filled once;
 *                qspec_check_status(ws) reports invalid nodes (token outside [0, V) or a parent not in
 *                [-1, j-1]) as QSPEC_ERR_INVALID_ARG; such nodes never match.
 *   1 <= B, 1 <= T <= QSPEC_MAX_TREE, 2 <= V <= 2^24, B*(T+1)*V < 2^40.  Bit-exact.
 */
size_t qspec_verify_tree_workspace_size(int32_t B, int32_t T, int32_t V);
qspec_status qspec_verify_tree_greedy(const uint16_t* tgt_logits, const int32_t* tree_tok,
                                      const int32_t* tree_parent, int32_t B, int32_t T, int32_t V,
                                      int32_t* accept_len, int32_t* out_tok, int32_t* accept_nodes,
                                      void* ws, size_t ws_bytes, qspec_stream_t stream);

/*
 * qspec_verify_greedy_noalloc -- qspec_verify_greedy for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point.  Some callers cannot call cudaMalloc where they
 * verify: plug-ins executing inside another runtime's fixed memory plan (a serving engine that
 * forbids allocation during a decode step), or C hosts with no allocator at hand.  This variant takes
 * no workspace: its scratch (error word, per-sequence tickets, per-chunk partial argmaxes) is a fixed
 * array of QSPEC_NOALLOC_SCRATCH_BYTES of device memory inside the library, which every GPU that
 * loads the library holds until the process exits.  It allocates nothing and calls no allocating
 * routine.
 *
 *   Arguments and results as qspec_verify_greedy (bit-identical outputs), without ws / ws_bytes.
 *   Size limit: with R = B*(gamma+1) rows and C chunks per row (C = 1 once R >= 1216, otherwise at
 *   most ceil(1216 / R) and at most ceil(V / 2048)), the call needs
 *       256 + round_up_256(4*B) + 8*R*C  <=  QSPEC_NOALLOC_SCRATCH_BYTES
 *   bytes; that is up to about 26 000 rows at gamma = 1 and 31 700 at gamma = 15.  Larger shapes are
 *   rejected with QSPEC_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
 *   The first call in a CUDA context (normally once per device, in its primary context) looks up the
 *   array's device address with that context current and caches it for the context; make that first
 *   call before any stream capture.
 *   Every call shares the one array and clears its error word and tickets on `stream` first, so
 *   calls that overlap on the GPU (different streams, or concurrent graphs) race and must not be
 *   issued.  Draft-token range errors are not reported by qspec_check_status for this variant;
 *   out-of-range tokens simply never match.
 */
#define QSPEC_NOALLOC_SCRATCH_BYTES (256 * 1024)
qspec_status qspec_verify_greedy_noalloc(const uint16_t* tgt_logits, const int32_t* draft_tok,
                                         int32_t B, int32_t gamma, int32_t V, int32_t* accept_len,
                                         int32_t* out_tok, int32_t* tgt_argmax, qspec_stream_t stream);

/*
 * qspec_gather_rows -- dst[m, :] = src[idx[m], :] for m < n (step f1: embedding lookup of the tokens
 * a decode step feeds the model, and reordering of logits rows between [gamma, B] and [B, gamma]).
 *
 * Tutorial "Speculative Decodingとは？LLM生成を速くする方法", section "draft modelとtarget modelの
 * 処理フロー": each draft step feeds the token just chosen back into the model.
 *   src  [n_src, row_bytes] device;  idx [n] int32 device;  dst [n, row_bytes] device (no overlap
 *   with src).  row_bytes a multiple of 4; src, dst and idx 4-byte aligned, and src and dst 16-byte
 *   aligned when row_bytes is a multiple of 16 and at least 1024 (one CTA per row, 16-byte copies;
 *   shorter rows such as token ids take one thread per row); n <= 2^31 - 1.
 *   An id outside [0, n_src) writes a zero row and makes the next qspec_check_status return
 *   QSPEC_ERR_INVALID_ARG.
 */
qspec_status qspec_gather_rows(const void* src, int64_t n_src, int64_t row_bytes, const int32_t* idx,
                               int64_t n, void* dst, qspec_stream_t stream);

/*
 * qspec_select_tokens -- the next token of each of R logits rows (step f1: how a draft step, or a
 * plain target-only decode step, picks its token).
 *
 * Same section: the draft proposes its most likely token when decoding greedily and a draw from its
 * distribution q when sampling (temperature 1, fp32 softmax, inverse CDF in index order as in the
 * sampling verify):
 *     u == NULL:  tok[r] = argmax_j logits[r, j]    (lowest index among equal maxima; bit-exact)
 *     otherwise:  tok[r] = smallest j with sum_{i<=j} exp(l_i - m) > u[r] * sum_i exp(l_i - m)
 *                 (m = max_j l_j; if rounding leaves no such j, the last j with a nonzero term)
 *   logits [R, V] bf16 (16-byte aligned);  u [R] fp32 in [0,1) or NULL;  tok [R] int32 (output);
 *   u and tok 4-byte aligned.  One CTA per row.  2 <= V <= 2^24.  A row of only -inf gives token 0.
 */
qspec_status qspec_select_tokens(const uint16_t* logits, int32_t R, int32_t V, const float* u, int32_t* tok,
                                 qspec_stream_t stream);

/*
 * qspec_copy -- move `bytes` from src to dst with one kernel on the SMs (no copy engine).
 *
 * For a decode step's small per-step transfers (a few tokens' activations in, the verify results
 * out), where a copy-engine transfer is mostly fixed latency and the kernel after it cannot begin
 * until it ends.  Either pointer may be device memory or pinned (page-locked, host-allocated or
 * registered) host memory, which the kernel reads or writes through its device mapping over the
 * host link; pageable host memory is refused.  Launched with programmatic dependent launch: the
 * next kernel's prologue overlaps the copy; the copy writes dst only after the previous kernel in
 * the stream has finished, and reads a device-memory src only then too (a host src earlier).
 *
 *   dst, src  16-byte aligned, not overlapping; bytes > 0, a multiple of 16.
 * Returns QSPEC_ERR_INVALID_ARG for a null pointer, zero bytes or memory the GPU cannot address,
 * QSPEC_ERR_MISALIGNED for an address or size that is not a multiple of 16.
 */
qspec_status qspec_copy(void* dst, const void* src, size_t bytes, qspec_stream_t stream);

/*
 * qspec_check_status -- synchronises `stream`, then reports (and clears) the error words that the
 * kernels set on the device: the verify workspace's word when `ws` is not NULL, and the library's
 * own words for the linear and decode-loop kernels of the current device.  QSPEC_ERR_TIMEOUT if a
 * kernel gave up a bounded wait, QSPEC_ERR_WORKSPACE if a linear call found its workspace laid out
 * for another shape, QSPEC_ERR_INVALID_ARG if a draft token id or a gather id was out of range,
 * QSPEC_ERR_CUDA if the stream reported an error, QSPEC_OK otherwise.
 */
qspec_status qspec_check_status(void* ws, qspec_stream_t stream);

/* qspec_status_string -- a static, human-readable name for a status code. */
const char* qspec_status_string(qspec_status status);

#ifdef __cplusplus
}
#endif

#endif /* QSPEC_H_ */
