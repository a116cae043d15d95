"""The C-ABI library loads and exports every entry point of include/qspec.h; host-side argument
checks reject bad calls before anything reaches a GPU (no compute is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qspec.h")


def declared_symbols():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qspec_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    return q.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["qspec_pack_weights", "qspec_linear_w4a16", "qspec_linear_w4a4", "qspec_linear_workspace_size",
                 "qspec_verify_greedy",
                 "qspec_verify_sample", "qspec_verify_workspace_size", "qspec_check_status",
                 "qspec_status_string"]:
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    for name in declared_symbols():
        assert name in q.SIGNATURES, name
        assert callable(getattr(q, name, None)), name


def test_status_strings(lib):
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    for code, name in q.STATUS.items():
        assert lib.qspec_status_string(code).decode() == name
    assert lib.qspec_status_string(99).decode() == "QSPEC_ERR_UNKNOWN"


FAKE = 1 << 20          # a 16-byte-aligned stand-in address; never dereferenced (checks fail first)


def test_pack_argument_checks(lib):
    assert lib.qspec_pack_weights(None, 8, 128, FAKE, FAKE, None) == 1
    assert lib.qspec_pack_weights(FAKE, 0, 128, FAKE, FAKE, None) == 1
    assert lib.qspec_pack_weights(FAKE, 8, 100, FAKE, FAKE, None) == 2
    assert lib.qspec_pack_weights(FAKE + 8, 8, 128, FAKE, FAKE, None) == 3


def test_linear_argument_checks(lib):
    f16, f4 = lib.qspec_linear_w4a16, lib.qspec_linear_w4a4
    W = 1 << 16
    assert f16(FAKE, FAKE, FAKE, 4, 512, 256, None, FAKE, W, None) == 1
    assert f16(FAKE, FAKE, FAKE, 0, 512, 256, FAKE, FAKE, W, None) == 1
    assert f16(FAKE, FAKE, FAKE, 4097, 512, 256, FAKE, FAKE, W, None) == 2    # M above the limit
    assert f16(FAKE, FAKE, FAKE, 4, 510, 256, FAKE, FAKE, W, None) == 2       # N % 8 != 0
    assert f16(FAKE, FAKE, FAKE, 4, 512, 200, FAKE, FAKE, W, None) == 2       # K % 128 != 0
    assert f16(FAKE, FAKE + 4, FAKE, 4, 512, 256, FAKE, FAKE, W, None) == 3
    assert f16(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, None, W, None) == 4       # no workspace
    assert f16(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, FAKE + 8, W, None) == 3
    assert f4(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, FAKE + 1, None, None, FAKE, W, None) == 3
    assert f4(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, None, None, FAKE + 2, FAKE, W, None) == 3
    assert f4(FAKE, FAKE, FAKE, 4, 512, 384 + 1, FAKE, None, None, None, FAKE, W, None) == 2
    assert f4(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, None, None, None, None, W, None) == 4
    need = lib.qspec_linear_workspace_size(16, 264, 8192)                      # a K-chunked GEMV shape
    assert f16(FAKE, FAKE, FAKE, 16, 264, 8192, FAKE, FAKE, need - 256, None) == 4
    assert f4(FAKE, FAKE, FAKE, 16, 264, 8192, FAKE, None, None, None, FAKE, need - 256, None) == 4


def test_linear_workspace_size_rejects_bad_shapes(lib):
    assert lib.qspec_linear_workspace_size(0, 512, 256) == 0
    assert lib.qspec_linear_workspace_size(4, 510, 256) == 0
    assert lib.qspec_linear_workspace_size(4, 512, 200) == 0
    assert lib.qspec_linear_workspace_size(4097, 512, 256) == 0


def test_verify_workspace_size(lib):
    assert lib.qspec_verify_workspace_size(0, 3, 1024) == 0
    assert lib.qspec_verify_workspace_size(1, 0, 1024) == 0
    assert lib.qspec_verify_workspace_size(1, 17, 1024) == 0
    assert lib.qspec_verify_workspace_size(1, 3, 1) == 0
    small = lib.qspec_verify_workspace_size(1, 3, 1024)
    big = lib.qspec_verify_workspace_size(64, 7, 152064)
    assert 0 < small < big and small % 256 == 0 and big % 256 == 0


def test_verify_argument_checks(lib):
    g = lib.qspec_verify_greedy
    need = lib.qspec_verify_workspace_size(2, 3, 1024)
    assert g(FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, FAKE, need - 1, None) == 4
    assert g(FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, need, None) == 4
    assert g(FAKE, FAKE, 2, 17, 1024, FAKE, FAKE, None, FAKE, need, None) == 2
    assert g(FAKE, FAKE, 2, 3, 1, FAKE, FAKE, None, FAKE, need, None) == 2
    assert g(None, FAKE, 2, 3, 1024, FAKE, FAKE, None, FAKE, need, None) == 1
    assert g(FAKE, FAKE, 2, 3, 1024, FAKE + 4, FAKE, None, FAKE, need, None) == 3
    s = lib.qspec_verify_sample
    assert s(FAKE, None, FAKE, FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, None, FAKE, need, None) == 1
    assert s(FAKE, FAKE, FAKE, FAKE + 8, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, None, FAKE, need, None) == 3
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, None, FAKE, 16, None) == 4


def test_w4a8_argument_checks(lib):
    f8 = lib.qspec_linear_w4a8
    W = 1 << 16
    assert f8(FAKE, FAKE, FAKE, 4, 512, 256, None, None, None, None, FAKE, W, None) == 1
    assert f8(FAKE, FAKE, FAKE, 4097, 512, 256, FAKE, None, None, None, FAKE, W, None) == 2
    assert f8(FAKE, FAKE, FAKE, 4, 512, 200, FAKE, None, None, None, FAKE, W, None) == 2
    assert f8(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, FAKE + 1, None, None, FAKE, W, None) == 3
    assert f8(FAKE, FAKE, FAKE, 4, 512, 256, FAKE, None, None, None, None, W, None) == 4


def test_top1_argument_checks(lib):
    t = lib.qspec_verify_top1
    need = lib.qspec_verify_workspace_size(2, 3, 1024)
    ok = (FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, 0.8, None)
    assert t(*ok, FAKE, need - 1, None) == 4                                     # workspace too small
    assert t(None, *ok[1:], FAKE, need, None) == 1                               # no target logits
    assert t(FAKE, FAKE, 2, 17, 1024, FAKE, FAKE, None, None, 0.8, None, FAKE, need, None) == 2
    assert t(FAKE, FAKE, 2, 3, 1, FAKE, FAKE, None, None, 0.8, None, FAKE, need, None) == 2
    assert t(FAKE, FAKE, 2, 3, 1024, FAKE + 4, FAKE, None, None, 0.8, None, FAKE, need, None) == 3
    assert t(FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, float("nan"), None, FAKE, need, None) == 1
    assert t(FAKE, FAKE, 2, 3, 1024, FAKE, FAKE, None, None, 0.8, FAKE + 8, FAKE, need, None) == 3


def test_decode_loop_argument_checks(lib):
    g, sel = lib.qspec_gather_rows, lib.qspec_select_tokens
    assert g(None, 8, 64, FAKE, 4, FAKE, None) == 1
    assert g(FAKE, 0, 64, FAKE, 4, FAKE, None) == 1
    assert g(FAKE, 8, 6, FAKE, 4, FAKE, None) == 2                               # rows of 6 bytes
    assert g(FAKE, 8, 64, FAKE + 2, 4, FAKE, None) == 3                          # misaligned ids
    assert g(FAKE + 4, 8, 2048, FAKE, 4, FAKE, None) == 3                        # 16-byte rows need 16-byte bases
    assert sel(None, 4, 1024, None, FAKE, None) == 1
    assert sel(FAKE, 0, 1024, None, FAKE, None) == 1
    assert sel(FAKE, 4, 1, None, FAKE, None) == 2
    assert sel(FAKE + 8, 4, 1024, None, FAKE, None) == 3
    assert sel(FAKE, 4, 1024, FAKE + 1, FAKE, None) == 3


def test_tree_argument_checks(lib):
    t = lib.qspec_verify_tree_greedy
    need = lib.qspec_verify_tree_workspace_size(2, 7, 1024)
    assert need > 0 and lib.qspec_verify_tree_workspace_size(2, 65, 1024) == 0
    assert lib.qspec_verify_tree_workspace_size(0, 7, 1024) == 0
    assert t(FAKE, FAKE, FAKE, 2, 7, 1024, FAKE, FAKE, None, FAKE, need - 1, None) == 4
    assert t(FAKE, None, FAKE, 2, 7, 1024, FAKE, FAKE, None, FAKE, need, None) == 1
    assert t(FAKE, FAKE, FAKE, 2, 65, 1024, FAKE, FAKE, None, FAKE, need, None) == 2
    assert t(FAKE, FAKE, FAKE + 4, 2, 7, 1024, FAKE, FAKE, None, FAKE, need, None) == 3
    assert t(FAKE, FAKE, FAKE, 2, 7, 1024, FAKE, FAKE, FAKE + 8, FAKE, need, None) == 3


def test_product_path_has_no_fallback():
    """The binding never imports the oracle and fails loudly without the library."""
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    src = open(q.__file__, encoding="utf-8").read()
    assert "oracle" not in src.replace("no fallback", "")
    with pytest.raises(RuntimeError):
        q.load(os.path.join(ROOT, "does_not_exist.so"))


def test_linear_pass_argument_checks(lib):
    from quantized_speculative_decoding_qspec_gb300 import qspec as q

    def layers(*specs):
        arr = (q.PassLayer * len(specs))()
        for i, (x, N, K, after, res) in enumerate(specs):
            arr[i] = q.PassLayer(x, FAKE, FAKE, FAKE, N, K, after, res)
        return arr

    f = lib.qspec_linear_pass
    ok = layers((FAKE, 512, 256, 0, 0), (FAKE, 64, 4096, 1, 0))
    W = lib.qspec_linear_pass_workspace_size()
    assert W >= 8
    assert f(4, 1, None, 2, FAKE, W, None) == 1                 # no descriptors
    assert f(4, 1, ok, 0, FAKE, W, None) == 1                   # no layers
    assert f(4, 0, ok, 2, FAKE, W, None) == 1                   # no tokens
    assert f(5, 1, ok, 2, FAKE, W, None) == 1                   # no such mode
    assert f(16, 5, ok, 2, FAKE, W, None) == 2                  # M above QSPEC_PASS_MAX_M
    assert f(16, 1, layers(*[(FAKE, 512, 256, 0, 0)] * 17), 17, FAKE, W, None) == 2   # too many layers
    assert f(16, 4, layers((FAKE, 512, 25600 + 128, 0, 0)), 1, FAKE, W, None) == 2    # staging does not fit
    assert f(16, 1, layers((FAKE, 510, 256, 0, 0)), 1, FAKE, W, None) == 2           # N % 8
    assert f(16, 1, layers((FAKE, 512, 200, 0, 0)), 1, FAKE, W, None) == 2           # K % 128
    assert f(16, 1, layers((None, 512, 256, 0, 0)), 1, FAKE, W, None) == 1           # null pointer
    assert f(16, 1, layers((FAKE, 512, 256, 0, 7)), 1, FAKE, W, None) == 1           # reserved not 0
    assert f(16, 1, layers((FAKE + 8, 512, 256, 0, 0)), 1, FAKE, W, None) == 3       # misaligned x
    assert f(16, 1, ok, 2, None, W, None) == 4                  # no workspace
    assert f(16, 1, ok, 2, FAKE + 8, W, None) == 3              # misaligned workspace
    assert f(16, 1, ok, 2, FAKE, W - 1, None) == 4              # workspace too small


def test_linear_group_argument_checks(lib):
    from quantized_speculative_decoding_qspec_gb300 import qspec as q

    def parts(*specs):
        arr = (q.LinearPart * len(specs))()
        for i, (wp, N) in enumerate(specs):
            arr[i] = q.LinearPart(wp, FAKE, FAKE, N)
        return arr

    f, wsz = lib.qspec_linear_group, lib.qspec_linear_group_workspace_size
    qkv = parts((FAKE, 4096), (FAKE, 1024), (FAKE, 1024))
    W = wsz(1, qkv, 3, 4096)
    assert W > 0 and W == wsz(1, parts((FAKE, 6144)), 1, 4096)  # the parts' rows as one run of tiles
    assert wsz(5, qkv, 3, 4096) == 0                             # M above QSPEC_GROUP_MAX_M
    assert wsz(1, qkv, 5, 4096) == 0 and wsz(1, qkv, 0, 4096) == 0
    assert wsz(1, parts((FAKE, 100)), 1, 4096) == 0              # N % 8
    assert f(4, None, 1, 4096, qkv, 3, FAKE, W, None) == 1       # no activations
    assert f(4, FAKE, 1, 4096, None, 3, FAKE, W, None) == 1      # no parts
    assert f(4, FAKE, 1, 4096, qkv, 0, FAKE, W, None) == 1       # zero parts
    assert f(5, FAKE, 1, 4096, qkv, 3, FAKE, W, None) == 1       # no such mode
    assert f(16, FAKE, 5, 4096, qkv, 3, FAKE, W, None) == 2      # M above QSPEC_GROUP_MAX_M
    assert f(16, FAKE, 1, 4096, parts(*[(FAKE, 64)] * 5), 5, FAKE, W, None) == 2   # too many parts
    assert f(16, FAKE, 1, 200, qkv, 3, FAKE, W, None) == 2       # K % 128
    assert f(16, FAKE, 1, 4096, parts((FAKE, 64), (FAKE, 60)), 2, FAKE, W, None) == 2  # N % 8
    assert f(16, FAKE, 1, 4096, parts((None, 64)), 1, FAKE, W, None) == 1          # null weights
    assert f(16, FAKE, 1, 4096, parts((FAKE + 8, 64)), 1, FAKE, W, None) == 3      # misaligned weights
    assert f(16, FAKE + 8, 1, 4096, qkv, 3, FAKE, W, None) == 3  # misaligned x
    assert f(16, FAKE, 1, 4096, qkv, 3, None, W, None) == 4      # no workspace
    assert f(16, FAKE, 1, 4096, qkv, 3, FAKE + 8, W, None) == 3  # misaligned workspace
    assert f(16, FAKE, 1, 4096, qkv, 3, FAKE, W - 1, None) == 4  # workspace too small


def test_copy_argument_checks(lib):
    # refused on the host before any CUDA call: null pointers, zero bytes, 16-byte alignment of both
    # addresses and of the size
    assert lib.qspec_copy(None, ctypes.c_void_p(64), 64, None) == 1
    assert lib.qspec_copy(ctypes.c_void_p(64), None, 64, None) == 1
    assert lib.qspec_copy(ctypes.c_void_p(64), ctypes.c_void_p(128), 0, None) == 1
    assert lib.qspec_copy(ctypes.c_void_p(72), ctypes.c_void_p(128), 64, None) == 3
    assert lib.qspec_copy(ctypes.c_void_p(64), ctypes.c_void_p(136), 64, None) == 3
    assert lib.qspec_copy(ctypes.c_void_p(64), ctypes.c_void_p(128), 40, None) == 3
