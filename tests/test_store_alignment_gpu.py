"""The epilogues write O with 32-byte stores when the output (or the split-KV workspace) is
32-byte aligned and with 16-byte stores otherwise; the ABI only requires 16 bytes. Every test
here runs the same call twice, once into an output 16 bytes past a 32-byte boundary, and
expects bit-identical O and lse (one CTA computes each row in a fixed order). The aligned
results are checked against the oracle by the other GPU tests."""
import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import ensure_built, to_dev

pytestmark = pytest.mark.gpu

_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _outputs(shape, dtype, misaligned):
    """O [shape] and lse [shape[:-1]] views; O starts 16 bytes past a 32-byte boundary when
    `misaligned` (torch allocations are 256-byte aligned)."""
    tdt = _DT[dtype]
    shift = 16 // torch.tensor([], dtype=tdt).element_size() if misaligned else 0
    n = int(np.prod(shape))
    buf = torch.full((n + 64,), float("nan"), dtype=tdt, device="cuda")
    o = buf[shift:shift + n].view(*shape)
    assert o.data_ptr() % 32 == (16 if misaligned else 0)
    lse = torch.full(shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def _fwd_twice(q, k, v, *, dtype, path, causal, key_lengths=None):
    ensure_built()
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    kld = to_dev(key_lengths)
    res = []
    for mis in (False, True):
        o, lse = _outputs(q.shape, dtype, mis)
        api.fwd(qd, kd, vd, causal=causal, key_lengths=kld, return_lse=True, out=o, lse_out=lse,
                path=path)
        assert api.read_device_status() == _lib.ATTN_OK
        torch.cuda.synchronize()
        res.append((o.float().cpu().numpy(), lse.cpu().numpy()))
    return res


def _assert_identical(res):
    (o0, l0), (o1, l1) = res
    assert not np.isnan(o0).any() and not np.isnan(l0).any()
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_tiled_fp16_misaligned_output(d):
    q, k, v, _ = synth.draw(2, 3, 389, d, seed=7100 + d)
    _assert_identical(_fwd_twice(q, k, v, dtype="f16", path="tcgen05", causal=True))


def test_tiled_bf16_misaligned_output():
    q, k, v, _ = synth.draw_ex(1, 4, 4, 300, 300, 128, seed=7200, dtype="bf16")
    _assert_identical(_fwd_twice(q, k, v, dtype="bf16", path="tcgen05", causal=False))


def test_tiled_tf32_misaligned_output():
    q, k, v, _ = synth.draw(2, 2, 260, 32, seed=7300)
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    _assert_identical(_fwd_twice(q, k, v, dtype="f32", path="tcgen05", causal=False))


def test_short_kernel_misaligned_output():
    q, k, v, _ = synth.draw(5, 3, 200, 32, seed=7400)
    kl = np.array([200, 17, 0, 128, 199], dtype=np.int32)
    _assert_identical(_fwd_twice(q, k, v, dtype="f16", path="short", causal=False, key_lengths=kl))


def test_splitkv_misaligned_workspace_and_output():
    ensure_built()
    q, k, v, _ = synth.draw(1, 2, 700, 128, seed=7500)
    B, H, N, d = q.shape
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    n_splits = 3
    need = api.splitkv_workspace_bytes(B, H, N, d, n_splits)
    res = []
    for mis in (False, True):
        raw = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
        ws = raw[16:16 + need] if mis else raw[:need]
        assert ws.data_ptr() % 32 == (16 if mis else 0)
        o, lse = _outputs(q.shape, "f16", mis)
        api.fwd_splitkv(qd, kd, vd, causal=True, return_lse=True, out=o, lse_out=lse,
                        n_splits=n_splits, workspace=ws)
        assert api.read_device_status() == _lib.ATTN_OK
        torch.cuda.synchronize()
        res.append((o.float().cpu().numpy(), lse.cpu().numpy()))
    _assert_identical(res)
