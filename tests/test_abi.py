"""CPU-side checks of the C ABI: the library builds, loads without a GPU, exports
every function include/te_attn.h declares, and its host-only helpers answer."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "te_attn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(te_attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import bwd_packed_varlen_gb300 as ta
    if not os.path.exists(ta.library_path()):
        from bwd_packed_varlen_gb300 import build
        build.build()
    return ta.library()


def test_header_declares_the_two_entry_points():
    names = _declared()
    assert "te_attn_fwd_thd" in names and "te_attn_bwd_thd" in names
    assert len(names) >= 7


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_host_helpers(lib):
    import bwd_packed_varlen_gb300 as ta
    assert ta.version() >= 10000
    assert ta.fwd_workspace_size(7, 32960, 32960, 32, 8, 128) > 0
    # backward workspace holds D = rowsum(dO * O): fp32 [total_q, hq]
    assert (ta.bwd_workspace_size(7, 32960, 32960, 32, 8, 128)
            - ta.fwd_workspace_size(7, 32960, 32960, 32, 8, 128)) >= 32960 * 32 * 4
    assert ta.fwd_workspace_size(0, 10, 10, 2, 1, 64) == 0
    assert lib.te_attn_last_error() is not None


def test_no_cpu_path():
    """The binding refuses CPU tensors instead of computing anything on the host."""
    import torch
    import bwd_packed_varlen_gb300 as ta
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises((ValueError, RuntimeError)):
        ta.fwd(q, q, q, cu, cu, cu, cu, 0.1, 1)


def _param_counts():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(te_attn_\w+)\s*\(([^)]*)\)\s*;", src):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else len(args.split(","))
    return out


def test_binding_signatures_match_header(lib):
    """Every ctypes prototype has as many parameters as the C declaration."""
    counts = _param_counts()
    for name, n in counts.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == n, (name, n, fn.argtypes)


def test_autograd_wrapper_has_no_cpu_path():
    """The DotProductAttention-like wrapper refuses CPU tensors and unsupported
    layouts before any compute; the mask aliases map to the C ABI's three masks."""
    import torch
    import bwd_packed_varlen_gb300 as ta
    from bwd_packed_varlen_gb300 import autograd as ag
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    kv = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError):
        ta.dot_product_attention(q, kv, kv, cu, cu)
    with pytest.raises(ValueError):
        ta.DotProductAttention(2, 64, 1)(q, kv, kv, cu, cu)
    with pytest.raises(NotImplementedError):
        ta.dot_product_attention(q, kv, kv, cu, cu, qkv_format="hbsd")
    q4, kv4 = q.view(4, 1, 2, 64), kv.view(4, 1, 1, 64)
    with pytest.raises(ValueError):
        ta.dot_product_attention(q4, kv4, kv4, cu, cu, qkv_format="sbhd")
    with pytest.raises(ValueError):
        ta.fwd_sbhd(q4, kv4, kv4, cu, cu, 0.1)
    with pytest.raises(ValueError):
        ta.DotProductAttention(3, 64, 2)
    assert {ag._mask_name(m) for m in ("causal", "padding_causal")} == {"padding_causal"}
    assert ag._mask_name("causal_bottom_right") == "padding_causal_bottom_right"
    assert ag._mask_name("no_mask") == "padding"
    assert ta._binding._mask("padding_causal_bottom_right") == 3


def test_host_checked_errors_launch_nothing(lib):
    """Argument errors the host can see return their code before any device work,
    so they are checked here without a GPU (the pointers are placeholders that the
    library never dereferences on these paths)."""
    import ctypes
    P = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never touched
    cu = ctypes.c_void_p(1 << 21)
    big = ctypes.c_size_t(1 << 40)

    def fwd(**kw):
        a = dict(batch=2, tq=64, tk=64, hq=4, hkv=2, d=64, scale=0.1, mask=1, dtype=1, ws=P, wsb=big)
        a.update(kw)
        return lib.te_attn_fwd_thd(P, P, P, P, P, cu, cu, cu, cu, a["batch"], a["tq"], a["tk"], 0, 0,
                                   a["hq"], a["hkv"], a["d"], a["scale"], a["mask"], a["dtype"],
                                   a["ws"], a["wsb"], None)
    assert fwd(mask=4) == -2                      # unknown mask type
    assert fwd(hq=3) == -1                        # hq not a multiple of hkv
    assert fwd(d=12) == -2                        # head dim not a multiple of 8
    assert fwd(d=264) == -2                       # head dim above 256
    assert fwd(batch=0) == -1
    assert fwd(dtype=7) == -2
    assert fwd(scale=float("inf")) == -1
    assert fwd(ws=None) == -1
    assert fwd(wsb=ctypes.c_size_t(16)) == -3     # workspace too small
    assert lib.te_attn_last_error()

    def e4m3(d=64, descale=1.0, wsb=big):
        return lib.te_attn_fwd_thd_e4m3(P, P, P, P, P, cu, cu, cu, cu, 2, 64, 64, 0, 0, 4, 2, d,
                                        0.1, descale, 1.0, 1.0, 1, P, wsb, None)
    assert e4m3(d=40) == -2                       # e4m3 needs d % 16 == 0
    assert e4m3(d=144) == -2                      # and d <= 128
    assert e4m3(descale=0.0) == -1
    assert e4m3(descale=float("nan")) == -1
    assert e4m3(wsb=ctypes.c_size_t(lib.te_attn_fwd_workspace_size(2, 64, 64, 4, 2, 64))) == -3
    assert (lib.te_attn_fwd_e4m3_workspace_size(2, 64, 64, 4, 2, 64)
            == lib.te_attn_fwd_workspace_size(2, 64, 64, 4, 2, 64) + 64 * 2 * 64 * 2)

    assert lib.te_attn_fwd_sbhd(P, P, P, P, P, cu, cu, 0, 8, 8, 4, 2, 64, 0.1, 1, 1, P, big,
                                None) == -1       # batch < 1
    assert lib.te_attn_bwd_sbhd(P, P, P, P, P, P, P, P, P, cu, cu, 2, -1, 8, 4, 2, 64, 0.1, 1, 1,
                                P, big, None) == -1  # negative length
    assert lib.te_attn_fwd_sbhd(P, P, P, P, P, cu, cu, 2, 1 << 30, 8, 4, 2, 64, 0.1, 1, 1, P, big,
                                None) == -1       # rows overflow int


def test_misaligned_tensor_pointers_are_refused(lib):
    """A tensor pointer off a 16-byte boundary is answered with TE_ERR_INVALID_ARG
    before any launch, on the forward and on every backward tensor (placeholder
    pointers that the library never dereferences on this path)."""
    import ctypes
    P = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 8)
    cu = ctypes.c_void_p(1 << 21)
    big = ctypes.c_size_t(1 << 40)
    args = (cu, cu, cu, cu, 2, 64, 64, 0, 0, 4, 2, 64, 0.1, 1, 1, P, big, None)
    for i in (0, 1, 2, 3):                        # q, k, v, out
        ptrs = [P] * 5
        ptrs[i] = bad
        assert lib.te_attn_fwd_thd(*ptrs, *args) == -1, i
        assert b"aligned" in lib.te_attn_last_error()
    for i in (0, 1, 2, 3, 4, 6, 7, 8):            # q, k, v, out, dout, dq, dk, dv
        ptrs = [P] * 9
        ptrs[i] = bad
        assert lib.te_attn_bwd_thd(*ptrs, *args) == -1, i
        assert b"aligned" in lib.te_attn_last_error()


def test_debug_build_exports_the_same_symbols(lib):
    """The bounds-checking build exports every declared function too."""
    import bwd_packed_varlen_gb300 as ta
    dbg = ta.library(debug=True)
    for name in _declared():
        assert hasattr(dbg, name), name
    assert dbg.te_attn_version() == lib.te_attn_version()


def test_noalloc_checks_arguments_before_sizes(lib):
    """te_attn_bwd_thd_noalloc answers a bad argument with te_attn_bwd_thd's own code
    and message, before it compares the problem with its built-in scratch size, and
    launches nothing in either case (placeholder pointers, no GPU needed)."""
    P = ctypes.c_void_p(1 << 20)
    cu = ctypes.c_void_p(1 << 21)

    def call(batch=2, tq=64, tk=64, hq=4, hkv=2, d=64, mask=1, dtype=1, lse=P):
        return lib.te_attn_bwd_thd_noalloc(P, P, P, P, P, lse, P, P, P, cu, cu, cu, cu, batch, tq,
                                           tk, 0, 0, hq, hkv, d, 0.1, mask, dtype, None)
    huge = 1 << 22  # a problem whose workspace exceeds the built-in scratch
    assert call(tq=huge, hq=3) == -1                  # hq not a multiple of hkv wins
    assert b"multiple of hkv" in lib.te_attn_last_error()
    assert call(tq=huge, d=12) == -2                  # unsupported head dim wins
    assert call(tq=huge, batch=0) == -1
    assert call(tq=huge, mask=9) == -2
    assert call(tq=huge, lse=None) == -1              # NULL lse
    assert call(tq=huge) == -3                        # valid arguments, too large
    assert b"more than the built-in" in lib.te_attn_last_error()


def test_selftest_and_status_reads_check_arguments(lib):
    """Host-side argument errors of the self-test and status entry points (no launch)."""
    assert lib.te_attn_selftest_wait_timeout(None, 256, 10, None) == -1
    P = ctypes.c_void_p(1 << 20)
    assert lib.te_attn_selftest_wait_timeout(P, 64, 10, None) == -3
    assert lib.te_attn_selftest_wait_timeout(P, 256, 0, None) == -1
    assert lib.te_attn_selftest_wait_timeout(P, 256, 2_000_000, None) == -1
    assert lib.te_attn_read_status_noalloc(None, None) == -1
    assert lib.te_attn_read_status(None, None, None) == -1


def test_backward_workspace_sizes(lib):
    """The fused backward's workspace adds its dQ accumulator (one 128-row fp32 tile
    of 64 or 128 columns per query tile and head), a counter per tile and its
    work-item list to the two-kernel backward's; it has none for d = 256."""
    B, T, hq, hkv = 7, 32960, 32, 8
    cap_q = T // 128 + B + 1
    cap_k = T // 128 + B + 1
    for d, cols in ((128, 128), (96, 128), (64, 64), (8, 64)):
        full = lib.te_attn_bwd_fused_workspace_size(B, T, T, hq, hkv, d)
        small = lib.te_attn_bwd_workspace_size(B, T, T, hq, hkv, d)
        extra = cap_q * hq * 128 * cols * 4 + cap_q * hq * 4 + cap_k * hkv * 16
        assert extra <= full - small <= extra + 512, (d, full - small, extra)
    assert lib.te_attn_bwd_fused_workspace_size(B, T, T, hq, hkv, 256) == 0
    P = ctypes.c_void_p(1 << 20)
    cu = ctypes.c_void_p(1 << 21)
    big = ctypes.c_size_t(1 << 40)
    # head dim above 128: unsupported, before any launch
    assert lib.te_attn_bwd_thd_fused(P, P, P, P, P, P, P, P, P, cu, cu, cu, cu, 2, 64, 64, 0, 0, 4,
                                     2, 256, 0.1, 1, 1, P, big, None) == -2
    # the two-kernel backward's workspace is too small for the fused one
    small = lib.te_attn_bwd_workspace_size(2, 64, 64, 4, 2, 128)
    assert lib.te_attn_bwd_thd_fused(P, P, P, P, P, P, P, P, P, cu, cu, cu, cu, 2, 64, 64, 0, 0, 4,
                                     2, 128, 0.1, 1, 1, P, ctypes.c_size_t(small), None) == -3
