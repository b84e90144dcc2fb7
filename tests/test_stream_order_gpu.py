"""Launch order on one stream with no host synchronisation in between.

The tiled and short-sequence kernels use programmatic dependent launch: they set up while
the previous kernel on the stream is still running and let the next kernel start early, but
they read or write global memory only after the previous kernel has completed. These tests
chain forwards on one stream with no synchronisation between them:
- a read of the previous launch's output (read after write);
- an overwrite of a buffer that the previous launch reads (write after read);
- an overwrite of a buffer that an earlier launch wrote (write after write).
Each chain is compared bit for bit with the same calls made one at a time with a
synchronize after each. The kernels are deterministic, so any difference means a launch
touched memory out of order.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import api, synth

pytestmark = pytest.mark.gpu

PAIRS_SHORT = [("tcgen05", "tcgen05"), ("short", "short"), ("tcgen05", "short"),
               ("short", "tcgen05"), ("short", "warp_mma"), ("warp_mma", "short")]


def _fwd(q, k, v, out, path, causal, kl):
    api.fwd(q, k, v, causal=causal, key_lengths=kl, out=out, path=path)


def _chain(q, q2, k, v, pa, pb, causal, kl, sync):
    """x1 = A(q); y = B(x1); x1 = A(q2); z = B(x1). Returns y, x1, z."""
    x1, y, z = (torch.empty_like(q) for _ in range(3))
    steps = [(q, x1, pa), (x1, y, pb), (q2, x1, pa), (x1, z, pb)]
    for src, dst, path in steps:
        _fwd(src, k, v, dst, path, causal, kl)
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return y, x1, z


def _check(q, q2, k, v, pa, pb, causal, kl, reps=4):
    y0, x0, z0 = _chain(q, q2, k, v, pa, pb, causal, kl, sync=True)
    assert not torch.isnan(z0).any()
    for _ in range(reps):
        y, x, z = _chain(q, q2, k, v, pa, pb, causal, kl, sync=False)
        assert torch.equal(y, y0), f"{pa}->{pb}: read after write"
        assert torch.equal(x, x0), f"{pa}->{pb}: write after write / read"
        assert torch.equal(z, z0), f"{pa}->{pb}: second read after write"


@pytest.mark.parametrize("pa,pb", PAIRS_SHORT, ids=[f"{a}-{b}" for a, b in PAIRS_SHORT])
def test_chained_launches_reranking_shape(pa, pb):
    """Reranking shape (B=50 H=12 N=256 d=32, key padding): every kernel takes it."""
    q, k, v, kl = synth.draw(50, 12, 256, 32, seed=31, key_len_range=(64, 256))
    q2, _, _, _ = synth.draw(50, 12, 256, 32, seed=32)
    qd, q2d, kd, vd = (torch.from_numpy(x).cuda() for x in (q, q2, k, v))
    _check(qd, q2d, kd, vd, pa, pb, False, torch.from_numpy(kl).cuda())


def test_chained_launches_tiled_causal():
    """Tiled kernel after itself on a causal d = 128 problem (persistent CTAs, one per SM)."""
    q, k, v, _ = synth.draw(2, 16, 2048, 128, seed=33)
    q2, _, _, _ = synth.draw(2, 16, 2048, 128, seed=34)
    qd, q2d, kd, vd = (torch.from_numpy(x).cuda() for x in (q, q2, k, v))
    _check(qd, q2d, kd, vd, "tcgen05", "tcgen05", True, None)


def test_chained_splitkv_and_merge():
    """Split-KV (split kernel, then merge kernel) feeding the tiled kernel and back."""
    q, k, v, _ = synth.draw(1, 4, 4096, 128, seed=35)
    q2, _, _, _ = synth.draw(1, 4, 4096, 128, seed=36)
    qd, q2d, kd, vd = (torch.from_numpy(x).cuda() for x in (q, q2, k, v))

    def chain(sync):
        x1, y = torch.empty_like(qd), torch.empty_like(qd)
        api.fwd_splitkv(qd, kd, vd, causal=True, out=x1, n_splits=4)
        if sync:
            torch.cuda.synchronize()
        api.fwd(x1, kd, vd, causal=True, out=y, path="tcgen05")
        if sync:
            torch.cuda.synchronize()
        api.fwd_splitkv(q2d, kd, vd, causal=True, out=x1, n_splits=4)
        torch.cuda.synchronize()
        return y, x1

    y0, x0 = chain(True)
    for _ in range(4):
        y, x = chain(False)
        assert torch.equal(y, y0) and torch.equal(x, x0)
    assert np.isfinite(y0.float().cpu().numpy()).all()
