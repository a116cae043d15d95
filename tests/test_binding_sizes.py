"""The Python binding refuses buffers smaller than the call reads or writes, before any launch (CPU).

The C ABI takes plain pointers and sizes, so it cannot see a short buffer; the binding knows each
tensor's element count and raises ValueError instead of letting a kernel run past its end.  These
checks run before the library is touched, so CPU tensors suffice here.
"""
import pytest
import torch

from quantized_speculative_decoding_qspec_gb300 import qspec as q

bf16, u8, f16, i32, f32, f64 = torch.bfloat16, torch.uint8, torch.float16, torch.int32, torch.float32, torch.float64
LINEARS = (q.qspec_linear_w4a16, q.qspec_linear_w4a4, q.qspec_linear_w4a8)


def z(*shape, dtype):
    return torch.zeros(*shape, dtype=dtype)


def linear_args(M=2, N=16, K=256):
    return z(M, K, dtype=bf16), z(N, K // 2, dtype=u8), z(N, K // 128, dtype=f16), z(M, N, dtype=bf16), z(64, dtype=u8)


@pytest.mark.parametrize("fn", LINEARS, ids=lambda f: f.__name__)
def test_linear_short_output_or_scales(fn):
    x, Wp, S, y, ws = linear_args()
    with pytest.raises(ValueError, match="y holds 31 elements, the call needs 32"):
        fn(x, Wp, S, y.view(-1)[:31], ws)
    with pytest.raises(ValueError, match="S holds"):
        fn(x, Wp, S.view(-1)[:-1], y, ws)


@pytest.mark.parametrize("fn", LINEARS[1:], ids=lambda f: f.__name__)
def test_linear_short_optional_outputs(fn):
    x, Wp, S, y, ws = linear_args()
    with pytest.raises(ValueError, match="xq_out holds"):
        fn(x, Wp, S, y, ws, xq_out=z(2, 255, dtype=torch.int8))
    with pytest.raises(ValueError, match="xs_out holds"):
        fn(x, Wp, S, y, ws, xs_out=z(1, dtype=f32))
    with pytest.raises(ValueError, match="acc_out holds"):
        fn(x, Wp, S, y, ws, acc_out=z(2, 16, 1, dtype=i32))


def test_exact_sizes_pass_the_checks():
    M, N, K = 3, 24, 384
    x, Wp, S, y, _ = linear_args(M, N, K)
    q._need_linear(M, N, K, Wp, S, y, z(M, K, dtype=torch.int8), z(M, dtype=f32), z(M, N, K // 128, dtype=i32))
    q._need_greedy(4, 5, z(4, 4, dtype=i32), z(4, dtype=i32), z(4, 5, dtype=i32), z(4, 5, dtype=i32))


def test_pack_short_outputs():
    W = z(16, 256, dtype=bf16)
    with pytest.raises(ValueError, match="Wp holds"):
        q.qspec_pack_weights(W, z(16, 127, dtype=u8), z(16, 2, dtype=f16))
    with pytest.raises(ValueError, match="S holds"):
        q.qspec_pack_weights(W, z(16, 128, dtype=u8), z(16, 1, dtype=f16))


def test_verify_short_buffers():
    B, g, V = 2, 3, 100
    tgt, drf = z(B, g + 1, V, dtype=bf16), z(B, g, V, dtype=bf16)
    d, n, out, ws = z(B, g, dtype=i32), z(B, dtype=i32), z(B, g + 1, dtype=i32), z(64, dtype=u8)
    with pytest.raises(ValueError, match="out_tok holds"):
        q.qspec_verify_greedy(tgt, d, n, out[:, :g], ws)
    with pytest.raises(ValueError, match="draft_tok holds"):
        q.qspec_verify_greedy_noalloc(tgt, d[:, :1], n, out)
    with pytest.raises(ValueError, match="tgt_argmax holds"):
        q.qspec_verify_greedy(tgt, d, n, out, ws, tgt_argmax=z(B, g, dtype=i32))
    ua, ur = z(B, g, dtype=f32), z(B, g + 1, dtype=f32)
    with pytest.raises(ValueError, match="u_resample holds"):
        q.qspec_verify_sample(tgt, drf, d, ua, ur[:, :g], n, out, ws)
    with pytest.raises(ValueError, match="draft_logits holds"):
        q.qspec_verify_sample(tgt, drf[:, :1], d, ua, ur, n, out, ws)
    with pytest.raises(ValueError, match="q_tok holds"):
        q.qspec_verify_sample(tgt, drf, d, ua, ur, n, out, ws, q_tok=z(B, dtype=f32))
    with pytest.raises(ValueError, match="draft_p1 holds"):
        q.qspec_verify_top1(tgt, drf, d, d.clone(), ws, draft_p1=z(B, g - 1, dtype=f32))


def test_select_and_tree_short_buffers():
    with pytest.raises(ValueError, match="tok holds"):
        q.qspec_select_tokens(z(4, 50, dtype=bf16), z(3, dtype=i32))
    with pytest.raises(ValueError, match="u holds"):
        q.qspec_select_tokens(z(4, 50, dtype=bf16), z(4, dtype=i32), u=z(2, dtype=f32))
    B, T, V = 2, 5, 64
    tgt, tok, par = z(B, T + 1, V, dtype=bf16), z(B, T, dtype=i32), z(B, T, dtype=i32)
    n, out, ws = z(B, dtype=i32), z(B, T + 1, dtype=i32), z(64, dtype=u8)
    with pytest.raises(ValueError, match="accept_nodes holds"):
        q.qspec_verify_tree_greedy(tgt, tok, par, n, out, ws, accept_nodes=z(B, T - 1, dtype=i32))
    with pytest.raises(ValueError, match="out_tok holds"):
        q.qspec_verify_tree_greedy(tgt, tok, par, n, out[:, :T], ws)
