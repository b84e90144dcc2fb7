"""The C-ABI library builds, loads, exports every symbol include/attn.h declares, and rejects
bad arguments synchronously (CPU only: no call here launches a kernel; a few reach a CUDA
device query, which fails without a GPU)."""
import ctypes
import os
import re

import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("attn_fwd", "attn_fwd_lse", "attn_fwd_path", "attn_status_str",
                     "attn_read_device_status"):
        assert required in names


def test_every_declared_symbol_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(_lib.SIGNATURES), "Python binding and header disagree"


def test_status_strings(lib):
    for code in range(0, 7):
        s = _lib.status_str(code)
        assert s and s != "unknown status"
    assert _lib.status_str(99) == "unknown status"


# Fake, never-dereferenced device addresses: validation must reject before any CUDA call.
A = 0x10000


def call(lib, q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=8, d=64, scale=0.125, causal=0,
         kl=None, path=0):
    return lib.attn_fwd_path(q, k, v, o, lse, B, H, N, d, scale, causal, kl, path, None)


@pytest.mark.parametrize("kw,expected", [
    (dict(q=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(k=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(v=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(H=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(N=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=48), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(path=7), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(d=128, path=_lib.PATH_SHORT), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(N=300, d=32, path=_lib.PATH_SHORT), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(q=A + 8), _lib.ATTN_ERR_MISALIGNED),
    (dict(o=A + 2), _lib.ATTN_ERR_MISALIGNED),
    (dict(lse=A + 2), _lib.ATTN_ERR_MISALIGNED),
    (dict(kl=A + 1), _lib.ATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=1 << 20, H=1 << 10, N=1 << 30, d=128), _lib.ATTN_ERR_INVALID_ARG),
])
def test_argument_validation(lib, kw, expected):
    assert call(lib, **kw) == expected


def test_fwd_and_fwd_lse_validate_too(lib):
    assert lib.attn_fwd(None, A, A, A, 1, 1, 8, 64, 0.1, 0, None, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_lse(A, A, A, A, None, 1, 1, 8, 40, 0.1, 0, None, None) == \
        _lib.ATTN_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.lib()


def test_splitkv_workspace_bytes(lib):
    # n_splits * B*H*N * (d + 1) * 4
    assert lib.attn_splitkv_workspace_bytes(2, 3, 100, 64, 4) == 4 * 2 * 3 * 100 * 65 * 4
    assert lib.attn_splitkv_workspace_bytes(1, 1, 1, 128, 1) == 129 * 4
    for bad in [(0, 1, 8, 64, 1), (1, 1, 8, 48, 1), (1, 1, 8, 64, 0), (1, 1, 8, 64, 17)]:
        assert lib.attn_splitkv_workspace_bytes(*bad) == 0


def test_splitkv_validation(lib):
    def sk(n_splits=2, ws=A, ws_bytes=1 << 30, **kw):
        args = dict(q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=256, d=64, scale=0.125, causal=0,
                    kl=None)
        args.update(kw)
        return lib.attn_fwd_splitkv(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                    args["B"], args["H"], args["N"], args["d"], args["scale"],
                                    args["causal"], args["kl"], n_splits, ws, ws_bytes, None)
    need = lib.attn_splitkv_workspace_bytes(1, 1, 256, 64, 2)
    assert sk(ws=None) == _lib.ATTN_ERR_INVALID_ARG
    assert sk(ws_bytes=need - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert sk(n_splits=17) == _lib.ATTN_ERR_INVALID_ARG
    assert sk(ws=A + 4, ws_bytes=need) == _lib.ATTN_ERR_MISALIGNED
    assert sk(d=48) == _lib.ATTN_ERR_UNSUPPORTED
    assert sk(q=None) == _lib.ATTN_ERR_INVALID_ARG


def test_naive_workspace_bytes(lib):
    # B*H*N*Np*6 with Np = N rounded up to a multiple of 128 (fp32 S, fp16 P)
    assert lib.attn_naive_workspace_bytes(2, 3, 100) == 2 * 3 * 100 * 128 * 6
    assert lib.attn_naive_workspace_bytes(4, 32, 4096) == 4 * 32 * 4096 * 4096 * 6
    assert lib.attn_naive_workspace_bytes(1, 1, 129) == 129 * 256 * 6
    for bad in [(0, 1, 8), (1, 0, 8), (1, 1, 0), (1, 1, -5)]:
        assert lib.attn_naive_workspace_bytes(*bad) == 0


def test_naive_validation(lib):
    """Argument errors of the naive forward come back before any launch."""
    def nv(ws=A, ws_bytes=1 << 30, **kw):
        args = dict(q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=256, d=64, scale=0.125, causal=0,
                    kl=None)
        args.update(kw)
        return lib.attn_fwd_naive(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                  args["B"], args["H"], args["N"], args["d"], args["scale"],
                                  args["causal"], args["kl"], ws, ws_bytes, None)
    need = lib.attn_naive_workspace_bytes(1, 1, 256)
    assert nv(ws=None) == _lib.ATTN_ERR_INVALID_ARG
    assert nv(ws_bytes=need - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert nv(ws=A + 8, ws_bytes=need) == _lib.ATTN_ERR_MISALIGNED
    assert nv(d=48) == _lib.ATTN_ERR_UNSUPPORTED
    assert nv(q=None) == _lib.ATTN_ERR_INVALID_ARG
    assert nv(causal=2) == _lib.ATTN_ERR_INVALID_ARG
    assert nv(scale=float("nan")) == _lib.ATTN_ERR_INVALID_ARG
    assert nv(o=A + 2) == _lib.ATTN_ERR_MISALIGNED


def test_noalloc_scratch_limit(lib):
    """The no-allocation split-KV entry point states its fixed scratch size and rejects a
    problem that needs more, before any launch."""
    cap = lib.attn_noalloc_scratch_bytes()
    assert cap == 64 << 20
    B, H, N, d, S = 1, 8, 32768, 128, 4
    assert lib.attn_splitkv_workspace_bytes(B, H, N, d, S) > cap
    st = lib.attn_fwd_splitkv_noalloc(A, A, A, A, None, B, H, N, d, 0.088, 1, None, S, None)
    assert st == _lib.ATTN_ERR_SCRATCH_LIMIT
    assert lib.attn_fwd_splitkv_noalloc(A, A, A, A, None, 1, 1, 256, 64, 0.125, 0, None, 17,
                                        None) == _lib.ATTN_ERR_INVALID_ARG
    # the automatic count cannot fit when even one range overflows the array
    assert lib.attn_splitkv_workspace_bytes(B, H, N, d, 1) > cap
    st = lib.attn_fwd_splitkv_noalloc(A, A, A, A, None, B, H, N, d, 0.088, 1, None, 0, None)
    assert st == _lib.ATTN_ERR_SCRATCH_LIMIT


def test_noalloc_auto_count_lowered_to_fit(lib):
    """With n_splits <= 0 the no-allocation entry point lowers the automatic count until the
    partials fit its array: here the automatic count (2 ranges on the 152-SM count assumed
    without a GPU) needs more than the array and one range fits, so the call gets past the
    scratch check (and, with no GPU, fails at the device lookup). Skipped where a GPU is
    present: the call would launch on the fake pointers."""
    if torch.cuda.is_available():
        pytest.skip("would launch on fake device pointers")
    cap = lib.attn_noalloc_scratch_bytes()
    B, H, N, d = 1, 4, 16384, 128
    auto = lib.attn_splitkv_auto_splits(B, H, N, d, 1)
    assert auto >= 2 and lib.attn_splitkv_workspace_bytes(B, H, N, d, auto) > cap
    assert lib.attn_splitkv_workspace_bytes(B, H, N, d, 1) <= cap
    st = lib.attn_fwd_splitkv_noalloc(A, A, A, A, None, B, H, N, d, 0.088, 1, None, 0, None)
    assert st == _lib.ATTN_ERR_CUDA


def call_ex(lib, q=A, k=A, v=A, o=A, lse=None, B=1, H=4, Hkv=2, Nq=8, Nk=32, d=64, dtype=0,
            scale=0.125, causal=0, kl=None, path=0):
    return lib.attn_fwd_ex(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, dtype, scale, causal, kl, path,
                           None)


@pytest.mark.parametrize("kw,expected", [
    (dict(Hkv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=3), _lib.ATTN_ERR_INVALID_ARG),        # H not a multiple of H_kv
    (dict(Hkv=8), _lib.ATTN_ERR_INVALID_ARG),        # more key/value heads than query heads
    (dict(Nk=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(Nq=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(k=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(path=_lib.PATH_SHORT, d=32), _lib.ATTN_ERR_UNSUPPORTED),            # cross shape
    (dict(path=_lib.PATH_SHORT, d=32, Nk=8), _lib.ATTN_ERR_UNSUPPORTED),      # grouped heads
    (dict(v=A + 8), _lib.ATTN_ERR_MISALIGNED),
    (dict(dtype=3), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=_lib.DTYPE_F32, d=64), _lib.ATTN_ERR_UNSUPPORTED),   # fp32: d = 32 only
    (dict(dtype=_lib.DTYPE_F32, d=32, path=_lib.PATH_SHORT), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=-1), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=_lib.DTYPE_BF16, path=_lib.PATH_WARP_MMA), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=_lib.DTYPE_BF16, Hkv=4, Nk=8, d=32, path=_lib.PATH_SHORT), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(H=4, Hkv=1, Nq=5, path=_lib.PATH_DECODE), _lib.ATTN_ERR_UNSUPPORTED),   # 20 packed rows
    (dict(H=4, Hkv=4, Nq=17, path=_lib.PATH_DECODE), _lib.ATTN_ERR_UNSUPPORTED),  # 17 rows
    (dict(dtype=_lib.DTYPE_F32, d=32, Nq=1, path=_lib.PATH_DECODE), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(path=5), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(B=1 << 17, H=1 << 10, Hkv=1 << 10, Nq=8, Nk=1 << 30, d=128), _lib.ATTN_ERR_INVALID_ARG),
])
def test_fwd_ex_validation(lib, kw, expected):
    assert call_ex(lib, **kw) == expected


def test_splitkv_ex_validation(lib):
    need = lib.attn_splitkv_workspace_bytes(1, 4, 8, 64, 2)
    args = (A, A, A, A, None, 1, 4, 2, 8, 32, 64, 0, 0.125, 0, None)
    assert lib.attn_fwd_splitkv_ex(*args, 2, None, need, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_splitkv_ex(*args, 2, A, need - 1, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_splitkv_ex(*args, 17, A, 1 << 30, None) == _lib.ATTN_ERR_INVALID_ARG
    bad = (A, A, A, A, None, 1, 4, 3, 8, 32, 64, 0, 0.125, 0, None)
    assert lib.attn_fwd_splitkv_ex(*bad, 2, A, 1 << 30, None) == _lib.ATTN_ERR_INVALID_ARG
    bad_dtype = (A, A, A, A, None, 1, 4, 2, 8, 32, 64, 5, 0.125, 0, None)
    assert lib.attn_fwd_splitkv_ex(*bad_dtype, 2, A, 1 << 30, None) == _lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_splitkv_auto_splits_ex(1, 4, 2, 8, 0, 64, 0) == -1
    assert lib.attn_splitkv_auto_splits_ex(1, 4, 2, 8, 32, 48, 0) == -1
    assert lib.attn_splitkv_auto_splits_ex(1, 4, 2, 8, 32, 64, 2) == -1
    assert lib.attn_splitkv_auto_splits_ex(1, 4, 3, 8, 32, 64, 0) == -1  # H not a multiple of H_kv


@pytest.mark.parametrize("args,expected", [
    # H, H_kv, N_q, N_k, d, dtype, causal -> kernel
    ((32, 8, 1, 8192, 128, _lib.DTYPE_F16, 1), _lib.PATH_DECODE),    # 4 packed rows
    ((32, 8, 4, 8192, 128, _lib.DTYPE_BF16, 1), _lib.PATH_DECODE),   # 16 packed rows
    ((32, 8, 5, 8192, 128, _lib.DTYPE_F16, 1), _lib.PATH_TCGEN05),   # 20 packed rows
    ((32, 8, 1, 256, 64, _lib.DTYPE_F16, 0), _lib.PATH_DECODE),      # the fewest keys it takes
    ((32, 8, 1, 255, 64, _lib.DTYPE_F16, 0), _lib.PATH_TCGEN05),
    ((4, 4, 16, 4096, 32, _lib.DTYPE_F16, 0), _lib.PATH_DECODE),     # unpacked, 16 rows
    ((4, 4, 17, 4096, 32, _lib.DTYPE_F16, 0), _lib.PATH_TCGEN05),
    ((32, 8, 1, 8192, 32, _lib.DTYPE_F32, 1), _lib.PATH_WARP_MMA),   # fp32: fp32 accuracy
    ((12, 12, 256, 256, 32, _lib.DTYPE_F16, 0), _lib.PATH_SHORT),    # self-attention, short
    ((32, 32, 4096, 4096, 128, _lib.DTYPE_F16, 1), _lib.PATH_TCGEN05),
    ((32, 32, 4096, 4096, 128, _lib.DTYPE_BF16, 1), _lib.PATH_TCGEN05),
    ((4, 3, 1, 512, 64, _lib.DTYPE_F16, 0), -1),                     # H not a multiple of H_kv
    ((4, 4, 1, 512, 48, _lib.DTYPE_F16, 0), -1),
    ((4, 4, 1, 512, 64, _lib.DTYPE_F32, 0), -1),                     # fp32 needs d = 32
    ((4, 4, 1, 512, 64, _lib.DTYPE_F16, 2), -1),
])
def test_auto_path_ex(lib, args, expected):
    """The automatic kernel choice of attn_fwd_ex, a host computation (no device needed)."""
    assert lib.attn_auto_path_ex(*args) == expected
