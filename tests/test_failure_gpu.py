"""Failure detection on the GPU without a fault: a bounded on-chip wait is made to run out
(the softmax warps withhold one arrival that nothing else provides), the kernel records
ATTN_ERR_TIMEOUT in the device status word and returns, and the context stays usable."""
import ctypes

import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import compare, ensure_built, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    ensure_built()
    lib = _lib.lib()
    q, k, v, _ = synth.draw(1, 2, 512, 64, seed=21)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    o = torch.empty_like(qd)
    assert api.read_device_status() == _lib.ATTN_OK
    opts = _lib.DebugOpts(wait_limit_ns=50_000_000, inject_missing_arrive=1)
    st = lib.attn_fwd_debug(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), None,
                            1, 2, 512, 64, 0.125, 0, None, _lib.PATH_TCGEN05, ctypes.byref(opts),
                            torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ATTN_OK
    assert api.read_device_status() == _lib.ATTN_ERR_TIMEOUT
    assert api.read_device_status() == _lib.ATTN_OK  # read-and-clear
    # the same process and context still compute correctly afterwards
    o_ref, lse_ref = oracle_full(q, k, v, causal=True)
    o2, lse2 = run_gpu(q, k, v, causal=True, path="tcgen05")
    compare(o2, lse2, o_ref, lse_ref, what="after timeout")


def test_default_limit_is_not_hit_by_normal_work():
    q, k, v, _ = synth.draw(2, 4, 2048, 128, seed=22)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    api.fwd(qd, kd, vd, causal=True)
    assert api.read_device_status() == _lib.ATTN_OK


def test_timeout_under_the_dynamic_schedule():
    """The same withheld arrival on a launch of 512 units (the dynamic schedule on GB300's
    152 SMs): every CTA's first unit runs out, aborted CTAs take no more units, the CTAs not yet
    started still run and run out in turn, and the context stays usable."""
    ensure_built()
    lib = _lib.lib()
    q, k, v, _ = synth.draw(4, 16, 4096, 64, seed=23)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    o = torch.empty_like(qd)
    assert api.read_device_status() == _lib.ATTN_OK
    opts = _lib.DebugOpts(wait_limit_ns=20_000_000, inject_missing_arrive=1)
    st = lib.attn_fwd_debug(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), None,
                            4, 16, 4096, 64, 0.125, 1, None, _lib.PATH_TCGEN05, ctypes.byref(opts),
                            torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ATTN_OK
    assert api.read_device_status() == _lib.ATTN_ERR_TIMEOUT
    assert api.read_device_status() == _lib.ATTN_OK
    qs, ks, vs, _ = synth.draw(1, 2, 512, 64, seed=24)
    o_ref, lse_ref = oracle_full(qs, ks, vs, causal=True)
    o2, lse2 = run_gpu(qs, ks, vs, causal=True, path="tcgen05")
    compare(o2, lse2, o_ref, lse_ref, what="after timeout (dynamic schedule)")
    # a launch of the same dynamic size still completes normally
    out = torch.empty_like(qd)
    api.fwd(qd, kd, vd, causal=True, out=out, path="tcgen05")
    torch.cuda.synchronize()
    assert api.read_device_status() == _lib.ATTN_OK
    assert not torch.isnan(out).any()
