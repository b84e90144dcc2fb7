"""Argument checks of the Python binding that run before any CUDA call (CPU only).

api._shapes reads (B, H, N, d, H_kv, N_k) from q [B, H, N, d] and k [B, H_kv, N_k, d] and
refuses shapes the C ABI cannot take. api._dtype_code maps the torch dtype to the C ABI's
element type.
"""
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, api


def _t(*shape, dtype=torch.float16):
    return torch.empty(shape, dtype=dtype, device="meta")


def test_shapes_self_cross_and_grouped():
    assert api._shapes(_t(2, 8, 100, 64), _t(2, 8, 100, 64)) == (2, 8, 100, 64, 8, 100)
    assert api._shapes(_t(2, 8, 1, 128), _t(2, 2, 4096, 128)) == (2, 8, 1, 128, 2, 4096)
    assert api._shapes(_t(1, 32, 1024, 128), _t(1, 8, 16384, 128)) == (1, 32, 1024, 128, 8, 16384)


@pytest.mark.parametrize("q,k", [
    ((2, 8, 100), (2, 8, 100, 64)),          # q not 4-D
    ((2, 8, 100, 64), (2, 8, 100)),          # k not 4-D
    ((2, 8, 100, 64), (3, 8, 100, 64)),      # batch mismatch
    ((2, 8, 100, 64), (2, 8, 100, 32)),      # head dimension mismatch
    ((2, 8, 100, 64), (2, 3, 100, 64)),      # H not a multiple of H_kv
])
def test_shapes_refused(q, k):
    with pytest.raises(ValueError):
        api._shapes(_t(*q), _t(*k))


def test_dtype_codes():
    assert api._dtype_code(_t(1, 1, 1, 32)) == _lib.DTYPE_F16
    assert api._dtype_code(_t(1, 1, 1, 32, dtype=torch.bfloat16)) == _lib.DTYPE_BF16
    assert api._dtype_code(_t(1, 1, 1, 32, dtype=torch.float32)) == _lib.DTYPE_F32
    for dt in (torch.float64, torch.int32, torch.float8_e4m3fn):
        with pytest.raises(TypeError):
            api._dtype_code(_t(1, 1, 1, 32, dtype=dt))


def test_path_names_match_the_c_enum():
    # attn_path_t: AUTO 0, WARP_MMA 1, TCGEN05 2, SHORT 3, DECODE 4
    assert _lib.PATHS == {"auto": 0, "warp_mma": 1, "tcgen05": 2, "short": 3, "decode": 4}
