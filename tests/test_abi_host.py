"""The C ABI on the host: the library loads, exports every symbol of include/cfc.h, and rejects
bad arguments with the documented status codes before it touches a GPU (no kernel runs)."""
import ctypes
import os
import re
import subprocess

import pytest

from recurrent_cfc_cell_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cfc.h")

OK, INVALID_DIM, NULL_PTR, MISALIGNED, WS_TOO_SMALL, UNSUPPORTED = 0, -1, -2, -3, -4, -5
INVALID_ARG = -8


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_documented_entry_points():
    assert set(declared_functions()) == set(_lib.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_error_strings(lib):
    for code in (OK, INVALID_DIM, NULL_PTR, MISALIGNED, WS_TOO_SMALL, UNSUPPORTED, -6, -7,
                 INVALID_ARG, -9, 12345):
        s = lib.cfc_error_string(code)
        assert isinstance(s, bytes) and len(s) > 0


def ws_bytes(lib, B, K, C, n_x, mode=0):
    out = ctypes.c_size_t(0)
    rc = lib.cfc_workspace_bytes(B, K, C, n_x, mode, ctypes.byref(out))
    return rc, out.value


@pytest.mark.parametrize("B,K,C,n_x", [(4, 8, 32, 16), (32, 64, 128, 48), (32, 64, 256, 64),
                                        (256, 64, 128, 48), (2048, 128, 256, 64), (1, 1, 1, 1),
                                        (3, 5, 40, 5)])
def test_workspace_holds_d_pre(lib, B, K, C, n_x):
    rc, n = ws_bytes(lib, B, K, C, n_x)
    assert rc == OK
    assert n >= K * B * 4 * C * 4


@pytest.mark.parametrize("B,K,C,n_x", [(0, 8, 32, 16), (4, 0, 32, 16), (4, 8, 0, 16),
                                        (4, 8, 32, 0), (4, 8, 257, 16), (4, 8, 256, 513),
                                        (-1, 8, 32, 16)])
def test_invalid_dims(lib, B, K, C, n_x):
    assert ws_bytes(lib, B, K, C, n_x)[0] == INVALID_DIM
    fake = ctypes.c_void_p(0x10000)
    rc = lib.cfc_forward(fake, fake, fake, fake, fake, B, K, C, n_x, fake, fake, None, 0,
                         None)
    assert rc == INVALID_DIM


def test_invalid_dw_mode(lib):
    assert ws_bytes(lib, 4, 8, 32, 16, mode=7)[0] == INVALID_ARG
    f = ctypes.c_void_p(0x10000)
    rc = lib.cfc_backward(f, f, f, f, f, f, f, 4, 8, 32, 16, f, f, f, f, f, 1 << 30, 7, None)
    assert rc == INVALID_ARG


def test_null_and_misaligned_pointers(lib):
    f = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    args = [f] * 5
    for k in range(5):
        a = list(args)
        a[k] = None
        assert lib.cfc_forward(*a, 4, 8, 32, 16, f, f, None, 0, None) == NULL_PTR
        a[k] = odd
        assert lib.cfc_forward(*a, 4, 8, 32, 16, f, f, None, 0, None) == MISALIGNED
    assert lib.cfc_forward(*args, 4, 8, 32, 16, None, f, None, 0, None) == NULL_PTR
    assert lib.cfc_forward(*args, 4, 8, 32, 16, f, odd, None, 0, None) == MISALIGNED
    # backward: du may be NULL, everything else may not
    b7 = [f] * 7
    outs = [f, f, f, f, f]  # dW, db, du, dh0, ws
    for k in (0, 1, 3, 4):
        o = list(outs)
        o[k] = None
        assert lib.cfc_backward(*b7, 4, 8, 32, 16, *o, 1 << 30, 0, None) == NULL_PTR
    o = list(outs)
    o[4] = odd
    assert lib.cfc_backward(*b7, 4, 8, 32, 16, *o, 1 << 30, 0, None) == MISALIGNED
    assert lib.reduce_axis0(None, 4, 4, f, None) == NULL_PTR
    assert lib.reduce_axis0(ctypes.c_void_p(0x10002), 4, 4, f, None) == MISALIGNED
    assert lib.reduce_axis0(f, 0, 4, f, None) == INVALID_DIM
    assert lib.reduce_axis0(f, 4, -3, f, None) == INVALID_DIM


def test_forward_backward_checks_every_argument_before_launching(lib):
    """The one-call training step rejects a bad argument of either half before it launches
    the forward (no GPU is touched on these paths)."""
    f = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    rc, need = ws_bytes(lib, 4, 8, 32, 16)
    assert rc == OK
    ins = [f] * 6                   # u, h0, W, b, ts, dH
    outs = [f] * 7                  # H, cache, dW, db, du, dh0, ws
    def call(i, o, dims=(4, 8, 32, 16), nbytes=need, mode=0):
        return lib.cfc_forward_backward(*i, *dims, *o, nbytes, mode, None)
    for k in range(6):
        a = list(ins)
        a[k] = None
        assert call(a, outs) == NULL_PTR
        a[k] = odd
        assert call(a, outs) == MISALIGNED
    for k in (0, 1, 2, 3, 5, 6):    # du (index 4) may be NULL
        o = list(outs)
        o[k] = None
        assert call(ins, o) == NULL_PTR
        o[k] = odd
        assert call(ins, o) == MISALIGNED
    assert call(ins, outs, dims=(4, 8, 257, 16)) == INVALID_DIM
    assert call(ins, outs, mode=7) == INVALID_ARG
    assert call(ins, outs, nbytes=need - 1) == WS_TOO_SMALL


def test_short_workspace(lib):
    f = ctypes.c_void_p(0x10000)
    rc, need = ws_bytes(lib, 4, 8, 32, 16)
    assert rc == OK
    assert lib.cfc_backward(*([f] * 7), 4, 8, 32, 16, f, f, f, f, f, need - 1, 0,
                            None) == WS_TOO_SMALL


def test_no_device_is_reported_not_crashed(lib):
    """On a machine without a GPU a well-formed call reports UNSUPPORTED_DEVICE."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    f = ctypes.c_void_p(0x10000)
    assert lib.cfc_forward(*([f] * 5), 4, 8, 32, 16, f, f, None, 0, None) == UNSUPPORTED
    st = ctypes.c_int(0)
    assert lib.cfc_device_status(ctypes.byref(st)) == UNSUPPORTED


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "libcfc.so"))


def _l2x_bytes(B, C):
    """The tensor-core BPTT's workspace: per CTA of a C / 32 cluster, the W_h^T slice as two fp16
    terms (C x 128 entries each: C * 512 bytes) and C output scales (fp32), 256-byte aligned;
    then per cluster two step-parities of C/32 x C/32 exchange blocks of [rows x 32] fp32, for
    the larger of the two row tiles (128 or 144 rows per cluster) rounded up over B."""
    cs = C // 32
    image = -(-(cs * C * 512 + cs * C * 4) // 256) * 256
    rows = max(-(-B // nr) * nr for nr in (128, 144))
    return image + rows * 2 * cs * cs * 32 * 4


@pytest.mark.parametrize("B,C,expect", [(32, 128, 0), (128, 256, 0), (129, 256, _l2x_bytes(129, 256)),
                                        (1024, 256, _l2x_bytes(1024, 256)),
                                        (512, 128, 0), (513, 128, _l2x_bytes(513, 128)),
                                        (2048, 256, _l2x_bytes(2048, 256)), (4096, 200, 0)])
def test_bptt_workspace_bytes(lib, B, C, expect):
    out = ctypes.c_size_t(123)
    assert lib.cfc_bptt_workspace_bytes(B, 8, C, 16, ctypes.byref(out)) == OK
    assert out.value == expect
    assert lib.cfc_bptt_workspace_bytes(B, 8, C, 16, None) == NULL_PTR
    assert lib.cfc_bptt_workspace_bytes(B, 0, C, 16, ctypes.byref(out)) == INVALID_DIM


def test_bptt_workspace_checked_before_launch(lib):
    f = ctypes.c_void_p(0x10000)
    need = 24 * 128 * 128
    args = (f, f, f, f, 1536, 4, 128, 8, f, f)
    assert lib.cfc_backward_recurrence_ws(*args, None, need, None) == NULL_PTR
    assert lib.cfc_backward_recurrence_ws(*args, ctypes.c_void_p(0x10008), need, None) == MISALIGNED
    assert lib.cfc_backward_recurrence_ws(*args, f, need - 16, None) == WS_TOO_SMALL


def _fwd_xch_bytes(B, C):
    """The tensor-core forward's exchange buffer: two step parities x clusters x C / 32 CTAs x
    one slot (the CTA's slab of h as two fp16 terms, rows x 32 channels x 2 bytes each), for the
    larger of the two row tiles (128 or 144 rows per cluster) rounded up over B."""
    rows = max(-(-B // nr) * nr for nr in (128, 144))
    return 2 * (C // 32) * 2 * rows * 32 * 2


@pytest.mark.parametrize("B,C,expect", [(32, 128, 0), (383, 256, 0), (384, 256, _fwd_xch_bytes(384, 256)),
                                        (767, 128, 0), (768, 128, _fwd_xch_bytes(768, 128)),
                                        (2048, 256, _fwd_xch_bytes(2048, 256)), (4096, 200, 0)])
def test_forward_workspace_bytes(lib, B, C, expect):
    out = ctypes.c_size_t(123)
    assert lib.cfc_forward_workspace_bytes(B, 8, C, 16, ctypes.byref(out)) == OK
    assert out.value == expect
    assert lib.cfc_forward_workspace_bytes(B, 8, C, 16, None) == NULL_PTR
    assert lib.cfc_forward_workspace_bytes(B, 0, C, 16, ctypes.byref(out)) == INVALID_DIM
    # cfc_forward_backward's workspace holds the forward's after the backward's own
    bwd = ctypes.c_size_t(0)
    assert lib.cfc_workspace_bytes(B, 8, C, 16, 0, ctypes.byref(bwd)) == OK
    assert bwd.value >= expect + K_ROWS_D_PRE(B, 8, C)


def K_ROWS_D_PRE(B, K, C):
    return K * B * 4 * C * 4


def test_forward_workspace_checked_before_launch(lib):
    f = ctypes.c_void_p(0x10000)
    need = _fwd_xch_bytes(2048, 256)
    args = [f] * 5 + [2048, 4, 256, 16, f, f]
    assert lib.cfc_forward(*args, None, need, None) == NULL_PTR
    assert lib.cfc_forward(*args, ctypes.c_void_p(0x10008), need, None) == MISALIGNED
    assert lib.cfc_forward(*args, f, need - 16, None) == WS_TOO_SMALL
    rargs = [f] * 3 + [2048, 4, 256, 16, f, f]
    assert lib.cfc_forward_recurrence(*rargs, None, need, None) == NULL_PTR
    assert lib.cfc_forward_recurrence(*rargs, f, need - 16, None) == WS_TOO_SMALL


def test_header_compiles_as_plain_c(tmp_path):
    """The boundary is a C ABI: include/cfc.h compiles as C99 with no C++ or CUDA headers."""
    import shutil

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "cfc.h"\nint main(void) { return cfc_error_string(0) == 0; }\n')
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                    str(tmp_path / "use_header.o")], check=True, capture_output=True)


def test_weight_grad_rejects_an_unsafe_in_place_d_pre(lib):
    """cfc_weight_grad may rewrite an fp32 d_pre in place at the workspace head only when C is
    even (each row's operand bytes are then its fp32 bytes); other overlaps are refused before
    anything is launched."""
    B, K, n_x = 3, 4, 5
    f = ctypes.c_void_p(0x100000)
    for C, mode, want in ((41, 0, INVALID_ARG), (41, 1, INVALID_ARG)):
        rc_ws, n = ws_bytes(lib, B, K, C, n_x, mode)
        assert rc_ws == OK
        d_pre = ctypes.c_void_p(0x100000)  # the head of ws
        rc = lib.cfc_weight_grad(d_pre, f, f, f, f, B, K, C, n_x, f, f, f, f, n, mode, None)
        assert rc == want, (C, mode, rc)
        inside = ctypes.c_void_p(0x100000 + 256)  # inside the head, not at it
        rc = lib.cfc_weight_grad(inside, f, f, f, f, B, K, 40, n_x, f, f, f, f, 1 << 30, mode,
                                 None)
        assert rc == INVALID_ARG


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_workspace_bytes_per_mode(lib, mode):
    rc, n = ws_bytes(lib, 32, 64, 128, 48, mode)
    assert rc == OK and n >= 32 * 64 * 4 * 128 * 4


def test_bf16_state_argument_checks(lib):
    """The bf16-state entry points: workspace size (X of every step in fp32: [K][B][C] padded
    to 256 bytes, then [K][B][3][C]), odd C and missing pointers refused before any launch."""
    out = ctypes.c_size_t(0)
    assert lib.cfc_forward_bf16_workspace_bytes(4, 8, 32, 16, ctypes.byref(out)) == OK
    assert out.value == -(-(8 * 4 * 32 * 4) // 256) * 256 + 8 * 4 * 3 * 32 * 4
    assert lib.cfc_forward_bf16_workspace_bytes(4, 8, 33, 16, ctypes.byref(out)) == INVALID_DIM
    assert lib.cfc_forward_bf16_workspace_bytes(4, 8, 32, 16, None) == NULL_PTR
    f = ctypes.c_void_p(0x10000)
    big = ctypes.c_size_t(1 << 30)
    assert lib.cfc_forward_bf16(*([f] * 5), 4, 8, 33, 16, f, f, f, big, None) == INVALID_DIM
    assert lib.cfc_forward_bf16(*([f] * 5), 4, 8, 32, 16, None, f, f, big, None) == NULL_PTR
    assert lib.cfc_forward_bf16(*([f] * 5), 4, 8, 32, 16, f, f, f, ctypes.c_size_t(16),
                                None) == WS_TOO_SMALL
    assert lib.cfc_backward_bf16(*([f] * 7), 4, 8, 33, 16, *([f] * 5), big, None) == INVALID_DIM
    assert lib.cfc_backward_bf16(*([f] * 5), None, f, 4, 8, 32, 16, *([f] * 5), big,
                                 None) == NULL_PTR


def test_decay_argument_checks(lib):
    """The tau-decay entry points: C beyond 128 and missing pointers refused before any launch;
    the workspace grows with the batch."""
    out = ctypes.c_size_t(0)
    assert lib.cfc_decay_workspace_bytes(4, 8, 129, 16, ctypes.byref(out)) == INVALID_DIM
    assert lib.cfc_decay_workspace_bytes(4, 8, 128, 16, None) == NULL_PTR
    assert lib.cfc_decay_workspace_bytes(4, 8, 128, 16, ctypes.byref(out)) == OK
    small = out.value
    assert lib.cfc_decay_workspace_bytes(40, 8, 128, 16, ctypes.byref(out)) == OK
    assert out.value > small
    f = ctypes.c_void_p(0x10000)
    assert lib.cfc_decay_forward(*([f] * 6), 4, 8, 129, 16, f, f, None) == INVALID_DIM
    assert lib.cfc_decay_forward(*([f] * 6), 4, 8, 32, 16, None, f, None) == NULL_PTR
    big = ctypes.c_size_t(1 << 30)
    assert lib.cfc_decay_backward(*([f] * 8), 4, 8, 32, 16, *([f] * 5), f, ctypes.c_size_t(16),
                                  None) == WS_TOO_SMALL
    assert lib.cfc_decay_backward(*([f] * 8), 4, 8, 32, 16, None, *([f] * 4), f, big,
                                  None) == NULL_PTR


def test_copy_argument_errors(lib):
    """cfc_copy refuses missing and unaligned buffers before it touches a device, and a copy of
    no bytes enqueues nothing."""
    p16, q16 = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)  # never dereferenced
    assert lib.cfc_copy(None, q16, 16, None) == NULL_PTR
    assert lib.cfc_copy(p16, None, 16, None) == NULL_PTR
    assert lib.cfc_copy(ctypes.c_void_p((1 << 20) + 8), q16, 16, None) == MISALIGNED
    assert lib.cfc_copy(p16, ctypes.c_void_p((2 << 20) + 4), 16, None) == MISALIGNED
    assert lib.cfc_copy(p16, q16, 24, None) == MISALIGNED
    assert lib.cfc_copy(p16, q16, 0, None) == OK
