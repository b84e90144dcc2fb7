"""The tiled kernel's dynamic unit schedule (one CTA per unit; running CTAs take over the units
of CTAs that have not started, by cluster launch control) under concurrency and graph replay.

Which CTA runs a unit changes from launch to launch, but a unit's arithmetic does not, so
every result must be bit-identical to a plain launch of the same problem:
- two dynamically scheduled launches running at once on two streams (cancellation acts within
  one grid, so neither may take the other's units);
- a launch captured in a CUDA graph and replayed several times;
- a problem below the dynamic threshold (static table) beside one above it.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu

# 4 x 16 heads x 8 Q-tile pairs = 512 units (dynamic on 152 SMs); 2 x 16 x 8 = 256 (static)
BIG = (4, 16, 4096, 64)
SMALL = (2, 16, 4096, 64)


def _inputs(shape, seed):
    q, k, v, _ = synth.draw(*shape, seed=seed)
    return tuple(torch.from_numpy(x).cuda() for x in (q, k, v))


def _plain(q, k, v, causal):
    o, lse = api.fwd(q, k, v, causal=causal, return_lse=True, path="tcgen05")
    torch.cuda.synchronize()
    assert api.read_device_status() == _lib.ATTN_OK
    return o.clone(), lse.clone()


def test_two_streams_at_once():
    a = _inputs(BIG, 8101)
    b = _inputs(BIG, 8102)
    ref_a = _plain(*a, causal=True)
    ref_b = _plain(*b, causal=False)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa, la = torch.empty_like(a[0]), torch.empty(BIG[:3], dtype=torch.float32, device="cuda")
    ob, lb = torch.empty_like(b[0]), torch.empty(BIG[:3], dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(sa):
            api.fwd(*a, causal=True, return_lse=True, out=oa, lse_out=la, path="tcgen05")
        with torch.cuda.stream(sb):
            api.fwd(*b, causal=False, return_lse=True, out=ob, lse_out=lb, path="tcgen05")
        torch.cuda.synchronize()
        assert api.read_device_status() == _lib.ATTN_OK
        assert torch.equal(oa, ref_a[0]) and torch.equal(la, ref_a[1])
        assert torch.equal(ob, ref_b[0]) and torch.equal(lb, ref_b[1])


def test_graph_replay():
    q, k, v = _inputs(BIG, 8103)
    ref = _plain(q, k, v, causal=True)
    o = torch.empty_like(q)
    lse = torch.empty(BIG[:3], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up outside the capture
        api.fwd(q, k, v, causal=True, return_lse=True, out=o, lse_out=lse, path="tcgen05")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.fwd(q, k, v, causal=True, return_lse=True, out=o, lse_out=lse, path="tcgen05")
    for _ in range(4):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert api.read_device_status() == _lib.ATTN_OK
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])


def test_static_and_dynamic_side_by_side():
    small = _inputs(SMALL, 8104)
    big = _inputs(BIG, 8105)
    ref_s = _plain(*small, causal=True)
    ref_b = _plain(*big, causal=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    os_, ob = torch.empty_like(small[0]), torch.empty_like(big[0])
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        api.fwd(*small, causal=True, out=os_, path="tcgen05")
    with torch.cuda.stream(s2):
        api.fwd(*big, causal=True, out=ob, path="tcgen05")
    torch.cuda.synchronize()
    assert api.read_device_status() == _lib.ATTN_OK
    assert torch.equal(os_, ref_s[0]) and torch.equal(ob, ref_b[0])
    assert not torch.isnan(ob).any()
