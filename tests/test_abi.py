"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/sdpa09.h declares, and rejects bad arguments before making
any CUDA call."""
import ctypes
import os
import re

import pytest

import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa09.h")

FAKE = 0x10000  # 16-byte aligned, never dereferenced by argument checks


def _header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return sdpa.load_library()


def test_header_symbols_match_binding():
    assert _header_functions() == sorted(sdpa.HEADER_SYMBOLS)


def test_library_exports_every_header_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_library_targets_sm103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_abi_version(lib):
    # 2: attn_swin_args gained its token layout field; 3: attn_fwd_varlen;
    # 4: attn_sam_args gained the table lengths (unequal grids, resampling);
    # 5: attn_bwd; 6: attn_fwd_train (row log-sum-exp for the backward)
    assert lib.attn_abi_version() == 6


def _call(lib, q=FAKE, k=FAKE + 4096, v=FAKE + 8192, out=FAKE + 1 << 20, B=1, H=1, Nq=64, Nk=64,
          d=32, scale=0.125, dtype=0, kind=0, args=None):
    return lib.attn_fwd(q, k, v, out, B, H, Nq, Nk, d, scale, dtype, kind, args, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), sdpa.ATTN_ERR_ARG),
    (dict(out=None), sdpa.ATTN_ERR_ARG),
    (dict(q=FAKE + 8), sdpa.ATTN_ERR_ARG),       # misaligned
    (dict(B=0), sdpa.ATTN_ERR_ARG),
    (dict(Nq=0), sdpa.ATTN_ERR_ARG),
    (dict(Nk=-3), sdpa.ATTN_ERR_ARG),
    (dict(d=36), sdpa.ATTN_ERR_ARG),             # not a multiple of 8
    (dict(d=0), sdpa.ATTN_ERR_ARG),
    (dict(d=256), sdpa.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=7), sdpa.ATTN_ERR_ARG),
    (dict(kind=9), sdpa.ATTN_ERR_ARG),
    (dict(scale=float("nan")), sdpa.ATTN_ERR_ARG),
    (dict(out=FAKE), sdpa.ATTN_ERR_ARG),         # aliases q
    (dict(B=1 << 16, H=1 << 8, Nq=1 << 8), sdpa.ATTN_ERR_UNSUPPORTED),  # 2^32 query rows
    (dict(Nk=(1 << 20) + 1), sdpa.ATTN_ERR_UNSUPPORTED),                # over 2^20 keys
])
def test_bad_arguments_rejected_before_cuda(lib, kw, code):
    assert _call(lib, **kw) == code
    assert lib.attn_last_error().decode()


def test_swin_argument_checks(lib):
    a = sdpa._SwinArgs(FAKE, 7, 56, 56, 3)
    # Nq != win*win
    assert _call(lib, Nq=50, Nk=50, kind=1, args=ctypes.byref(a)) == sdpa.ATTN_ERR_ARG
    # missing struct / table
    assert _call(lib, Nq=49, Nk=49, kind=1, args=None) == sdpa.ATTN_ERR_ARG
    bad = sdpa._SwinArgs(None, 7, 56, 56, 3)
    assert _call(lib, Nq=49, Nk=49, kind=1, args=ctypes.byref(bad)) == sdpa.ATTN_ERR_ARG
    # shift out of range, grid not a multiple of win, B not whole images
    for s in (sdpa._SwinArgs(FAKE, 7, 56, 56, 7), sdpa._SwinArgs(FAKE, 7, 50, 56, 3)):
        assert _call(lib, B=64, Nq=49, Nk=49, kind=1, args=ctypes.byref(s)) == sdpa.ATTN_ERR_ARG
    assert _call(lib, B=63, Nq=49, Nk=49, kind=1, args=ctypes.byref(a)) == sdpa.ATTN_ERR_ARG
    # windows above 128 tokens
    big = sdpa._SwinArgs(FAKE, 12, 24, 24, 0)
    assert _call(lib, B=4, Nq=144, Nk=144, kind=1, args=ctypes.byref(big)) == sdpa.ATTN_ERR_UNSUPPORTED
    # unknown token layout
    lay = sdpa._SwinArgs(FAKE, 7, 56, 56, 3, 2)
    assert _call(lib, B=64, Nq=49, Nk=49, kind=1, args=ctypes.byref(lay)) == sdpa.ATTN_ERR_ARG
    assert b"layout" in lib.attn_last_error()


def test_image_layout_binding_checks():
    import torch
    b = sdpa.SwinBias(torch.zeros(169, 3), 7, 56, 56, 3, layout="image")
    q = torch.zeros(2, 56, 56, 3, 32, dtype=torch.float16)
    assert sdpa._shape_image(q, q, q, b) == (2 * 64, 3, 49, 49, 32)
    with pytest.raises(sdpa.AttnError):
        sdpa._shape_image(q[:, :49], q[:, :49], q[:, :49], b)  # grid mismatch
    with pytest.raises(ValueError):
        sdpa.SwinBias(torch.zeros(169, 3), 7, 56, 56, 3, layout="rows")


def test_sam_argument_checks(lib):
    ok = sdpa._SamArgs(FAKE, FAKE, 8, 8, 8, 8)
    assert _call(lib, Nq=65, Nk=65, kind=2, args=ctypes.byref(ok)) == sdpa.ATTN_ERR_ARG
    diff = sdpa._SamArgs(FAKE, FAKE, 8, 8, 4, 4)
    # unequal grids are valid; the key count must match the key grid
    assert _call(lib, Nq=64, Nk=64, kind=2, args=ctypes.byref(diff)) == sdpa.ATTN_ERR_ARG
    long_table = sdpa._SamArgs(FAKE, FAKE, 8, 8, 8, 8, 129, 0)
    assert _call(lib, Nq=64, Nk=64, kind=2, args=ctypes.byref(long_table)) == sdpa.ATTN_ERR_UNSUPPORTED
    assert b"longer than 128" in lib.attn_last_error()
    none = sdpa._SamArgs(None, FAKE, 8, 8, 8, 8)
    assert _call(lib, Nq=64, Nk=64, kind=2, args=ctypes.byref(none)) == sdpa.ATTN_ERR_ARG
    huge = sdpa._SamArgs(FAKE, FAKE, 100, 100, 100, 100)
    assert _call(lib, Nq=10000, Nk=10000, kind=2, args=ctypes.byref(huge)) == sdpa.ATTN_ERR_UNSUPPORTED


def test_debug_bias_rejects_null_output(lib):
    assert lib.attn_debug_bias(FAKE, FAKE, FAKE, None, 1, 1, 64, 64, 32, 0.1, 0, 0, None, None) \
        == sdpa.ATTN_ERR_ARG


def test_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16)
    with pytest.raises(sdpa.AttnError):
        sdpa.attn_fwd(q, q[:, :1], q)
    with pytest.raises(sdpa.AttnError):
        sdpa.attn_fwd(q.float(), q.float(), q.float())


def test_selftest_limit_checked_before_cuda(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == sdpa.ATTN_ERR_ARG
    assert lib.attn_selftest_wait_timeout(2000001, None) == sdpa.ATTN_ERR_ARG
    assert b"limit_us" in lib.attn_last_error()


def _varlen(lib, cu_q, cu_k, n_seq=None, H=2, d=32, q=FAKE, out=FAKE + (1 << 20)):
    cq = (ctypes.c_int * len(cu_q))(*cu_q)
    ck = (ctypes.c_int * len(cu_k))(*cu_k)
    n = len(cu_q) - 1 if n_seq is None else n_seq
    return lib.attn_fwd_varlen(q, FAKE + 4096, FAKE + 8192, out, cq, ck, n, H, d, 0.125, 0, None)


def test_varlen_argument_checks(lib):
    ok_q, ok_k = [0, 5, 9], [0, 3, 9]
    assert _varlen(lib, ok_q, ok_k, q=None) == sdpa.ATTN_ERR_ARG
    assert _varlen(lib, ok_q, ok_k, n_seq=0) == sdpa.ATTN_ERR_ARG
    assert _varlen(lib, ok_q, ok_k, H=0) == sdpa.ATTN_ERR_ARG
    assert _varlen(lib, [1, 5, 9], ok_k) == sdpa.ATTN_ERR_ARG            # does not start at 0
    assert _varlen(lib, [0, 5, 4], ok_k) == sdpa.ATTN_ERR_ARG            # decreasing
    assert b"nondecreasing" in lib.attn_last_error()
    assert _varlen(lib, [0, 5, 9], [0, 0, 9]) == sdpa.ATTN_ERR_ARG       # queries without keys
    assert b"no keys" in lib.attn_last_error()
    assert _varlen(lib, ok_q, ok_k, d=36) == sdpa.ATTN_ERR_ARG           # checked as for attn_fwd
    big = list(range(0, 130))
    assert _varlen(lib, big, big) == sdpa.ATTN_ERR_UNSUPPORTED           # 129 sequences
    # no sequence has a query: nothing to launch
    assert _varlen(lib, [0, 0, 0], [0, 4, 4]) == sdpa.ATTN_OK


def test_varlen_binding_checks():
    import torch
    q = torch.zeros(2 * 9, 32, dtype=torch.float16)
    with pytest.raises(sdpa.AttnError):
        sdpa.attn_fwd_varlen(q, q, q, [0, 5, 9], [0, 4], H=2)             # different n_seq
    with pytest.raises(sdpa.AttnError):
        sdpa.attn_fwd_varlen(q, q, q, [0, 5, 10], [0, 4, 9], H=2)        # q too short for the offsets


def _bwd(lib, B=64, H=3, Nq=49, Nk=49, d=32, kind=0, args=None, d_table=None, q=FAKE, lse=None):
    return lib.attn_bwd(q, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, lse, FAKE + 20480, FAKE + 24576,
                        FAKE + 28672, B, H, Nq, Nk, d, 0.125, 0, kind, args, d_table, None, 0, None)


def test_bwd_argument_checks(lib):
    assert _bwd(lib, q=None) == sdpa.ATTN_ERR_ARG
    assert _bwd(lib, q=FAKE + 8) == sdpa.ATTN_ERR_ARG                       # misaligned
    assert _bwd(lib, d=36) == sdpa.ATTN_ERR_ARG
    # long sequences (or d > 64) take the two-pass path: the forward's lse and a workspace are required
    assert _bwd(lib, Nq=129) == sdpa.ATTN_ERR_ARG
    assert b"lse" in lib.attn_last_error()
    assert _bwd(lib, Nq=129, lse=FAKE + 32768) == sdpa.ATTN_ERR_ARG
    assert b"workspace" in lib.attn_last_error()
    assert lib.attn_bwd_workspace_size(64, 3, 129, 49, 32, 0, None) >= 64 * 3 * 129 * 4
    assert lib.attn_bwd_workspace_size(64, 3, 49, 49, 32, 0, None) == 0     # windows need none
    assert _bwd(lib, d=88) == sdpa.ATTN_ERR_UNSUPPORTED                     # d > 80
    sam = sdpa._SamArgs(FAKE, FAKE, 7, 7, 7, 7)
    assert _bwd(lib, kind=2, args=ctypes.byref(sam)) == sdpa.ATTN_ERR_ARG          # no d_bias
    assert _bwd(lib, kind=2, args=ctypes.byref(sam), d_table=FAKE) == sdpa.ATTN_ERR_UNSUPPORTED  # 7 x 7 grid
    assert b"14 x 14, 48 x 48 or 64 x 64" in lib.attn_last_error()
    long_tab = sdpa._SamArgs(FAKE, FAKE, 14, 14, 14, 14, 129, 27)               # a table over 128 rows
    assert _bwd(lib, Nq=196, Nk=196, d=80, kind=2, args=ctypes.byref(long_tab), d_table=FAKE) == sdpa.ATTN_ERR_UNSUPPORTED
    assert b"128 rows" in lib.attn_last_error()
    # tables of another length than 2 * side - 1: the workspace holds their resampled copies
    plain = sdpa._SamArgs(FAKE, FAKE, 48, 48, 48, 48)
    resized = sdpa._SamArgs(FAKE, FAKE, 48, 48, 48, 48, 127, 127)
    assert (lib.attn_bwd_workspace_size(1, 1, 2304, 2304, 80, 2, ctypes.byref(resized))
            > lib.attn_bwd_workspace_size(1, 1, 2304, 2304, 80, 2, ctypes.byref(plain)) > 0)
    swin = sdpa._SwinArgs(FAKE, 7, 56, 56, 3)
    assert _bwd(lib, kind=1, args=ctypes.byref(swin)) == sdpa.ATTN_ERR_ARG    # no d_table
    assert b"d_bias" in lib.attn_last_error()
    lay = sdpa._SwinArgs(FAKE, 7, 56, 56, 3, 2)                             # unknown token layout
    assert _bwd(lib, kind=1, args=ctypes.byref(lay), d_table=FAKE) == sdpa.ATTN_ERR_ARG
    assert b"layout" in lib.attn_last_error()
    assert _bwd(lib, B=63, kind=1, args=ctypes.byref(swin), d_table=FAKE) == sdpa.ATTN_ERR_ARG


def test_swin_bias_mma_variant_rejects_unrepresentable_scale(lib):
    # 10x10 windows (100 tokens, 128-row slots) add the bias through 16-bit
    # MMA operands holding table / scale and -100 / scale: scale = 0 (and,
    # for fp16, a scale that overflows -100 / scale) is refused before any
    # CUDA call instead of producing NaN or Inf
    a = sdpa._SwinArgs(FAKE, 10, 20, 20, 5)
    for dtype, scale in ((0, 0.0), (1, 0.0), (1, 1e-3), (1, -1e-3)):
        assert _call(lib, B=4, Nq=100, Nk=100, kind=1, args=ctypes.byref(a), dtype=dtype,
                     scale=scale) == sdpa.ATTN_ERR_UNSUPPORTED, (dtype, scale)
        assert b"scale" in lib.attn_last_error()


def test_varlen_offsets_marshalling():
    """The token offsets reach the C ABI as int32 arrays whatever host type
    holds them (list, tuple, numpy of any integer width, CPU tensor)."""
    import numpy as np
    import torch
    from scaled_dot_product_09_gb300 import _cu_array
    want = [0, 3, 9, 70]
    for cu in (want, tuple(want), np.array(want, dtype=np.int64), np.array(want, dtype=np.int32),
               torch.tensor(want), torch.tensor(want, dtype=torch.int32)):
        arr, vals = _cu_array(cu)
        assert list(arr) == want and list(vals) == want and vals[-1] == 70, type(cu)
    for big in ([0, 1 << 40], np.array([0, 1 << 40]), torch.tensor([0, 1 << 40])):
        with pytest.raises(OverflowError):
            _cu_array(big)
