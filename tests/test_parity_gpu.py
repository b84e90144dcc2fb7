"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Small shapes run the whole output through the oracle; they span several tiles of every
kernel and end in ragged tails. The five measured workloads run at full size: the tiny,
reranking, prefill and stress ones are compared on every row (the reranking workload ignores
its padded query rows), the long one (whose full oracle would take minutes) on tile-edge and
random rows in every one of its heads. Analytic cases (uniform keys, one-hot selection, causal
row 0, empty rows) are checked against their closed forms on the GPU too.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_attn_gb300 import synth
from parity import compare, oracle_full, run_gpu, sample_rows, workload_oracle

pytestmark = pytest.mark.gpu

# Kernels to check on every shape they support.
KERNELS = ["warp_mma", "tcgen05", "short"]


def kernels_for(d, N=None):
    out = []
    for k in KERNELS:
        if k == "short" and (d > 64 or (N is not None and N > 256)):
            continue
        out.append(k)
    return out


SMALL = [
    # B, H, N, d, causal, key_lengths
    (3, 4, 256, 32, True, [256, 100, 3]),
    (2, 3, 200, 64, True, [150, 200]),
    (1, 2, 16, 64, False, None),
    (1, 1, 1, 64, False, None),
    (1, 2, 48, 32, False, None),
    (2, 3, 127, 64, True, None),
    (1, 2, 129, 128, False, None),
    (2, 2, 200, 128, True, None),
    (3, 1, 333, 64, False, [333, 1, 170]),
    (2, 2, 384, 128, True, [0, 300]),
    (2, 1, 517, 32, True, [517, 77]),
    (1, 3, 640, 64, True, [600]),
    (1, 1, 1000, 128, False, [999]),
    (5, 7, 65, 32, False, [65, 64, 1, 0, 30]),
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{'c' if s[4] else ''}{'k' if s[5] else ''}" for s in SMALL])
def test_small_shapes(shape):
    B, H, N, d, causal, kl = shape
    q, k, v, _ = synth.draw(B, H, N, d, seed=1000 + N + d)
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    for kern in kernels_for(d, N):
        o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, path=kern)
        compare(o, lse, o_ref, lse_ref, what=f"{kern} {shape}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [0.05, 1.0, 2.5])
def test_scales(scale, d):
    """Wide score ranges (scale 1.0 and 2.5) make the rows of one warp disagree about when to
    move the softmax reference; small ones never move it after the first tile."""
    q, k, v, _ = synth.draw(2, 2, 300, d, seed=77)
    o_ref, lse_ref = oracle_full(q, k, v, causal=True, sm_scale=scale)
    for kern in kernels_for(d, 300):
        o, lse = run_gpu(q, k, v, causal=True, sm_scale=scale, path=kern)
        compare(o, lse, o_ref, lse_ref, what=f"{kern} scale={scale}")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("sign", [1.0, -1.0], ids=["pos", "neg"])
@pytest.mark.parametrize("N,period", [(640, 128), (256, 64)], ids=["N640", "N256"])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_growing_scores_move_reference(d, N, period, sign, causal):
    """Scores that grow by about 2^12 per block of `period` keys (the tiled kernels' 128-key
    tiles, the short kernel's 64-column blocks): every later block's exponentials against the
    row's reference would leave fp16, so the reference moves on every block. Rows alternate the
    sign of q, so in every warp half the rows grow and half shrink (the warp moves for some rows
    only); a negative scale mirrors it."""
    B, H = 1, 2
    rng = np.random.Generator(np.random.PCG64(4242 + d + N))
    step = 12.0 / (math.sqrt(d) * 1.4426950408889634)  # per-block growth of k: +12 in log2 units
    t = (np.arange(N) // period).astype(np.float64)
    k = (step * t)[None, None, :, None] * (1.0 + 0.05 * rng.standard_normal((B, H, N, d)))
    s = np.where(np.arange(N) % 2 == 0, 1.0, -1.0)[None, None, :, None]
    q = s * (1.0 + 0.05 * rng.standard_normal((B, H, N, d)))
    v = rng.standard_normal((B, H, N, d))
    q, k, v = (x.astype(np.float16) for x in (q, k, v))
    scale = sign / math.sqrt(d)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, sm_scale=scale)
    for kern in kernels_for(d, N):
        o, lse = run_gpu(q, k, v, causal=causal, sm_scale=scale, path=kern)
        compare(o, lse, o_ref, lse_ref, what=f"{kern} d={d} sign={sign} causal={causal}")


def _workload_case(name):
    w = synth.WORKLOADS[name]
    q, k, v, kl = synth.draw_workload(w)
    return w, q, k, v, kl


def _workload_kernels(w):
    """The automatic choice, then every other kernel that takes the shape (the automatic one
    is not launched twice)."""
    from exact_scaled_dot_attn_gb300 import api
    auto = api.auto_path(w.N, w.d)
    return ["auto"] + [k for k in kernels_for(w.d, w.N) if k != auto]


@pytest.mark.parametrize("name", ["tiny", "rerank", "prefill", "stress"])
def test_workload_full_rows(name):
    """Every row of the workload against the oracle (the stress workload checks lse too, as
    every comparison here does); the padded query rows of the reranking workload are the
    only rows left out."""
    w, q, k, v, kl, o_ref, lse_ref = workload_oracle(name)
    row_mask = None
    if w.ignore_padded_queries:
        i = np.arange(w.N)[None, None, :]
        row_mask = np.broadcast_to(i < kl[:, None, None], (w.B, w.H, w.N))
    for kern in _workload_kernels(w):
        o, lse = run_gpu(q, k, v, causal=w.causal, key_lengths=kl, path=kern)
        compare(o, lse, o_ref, lse_ref, row_mask=row_mask, what=f"{name} {kern}")
        if w.causal:
            # causal row 0 of every head: O_0 = V_0 up to the fp16 rounding of the output
            assert np.max(np.abs(o[:, :, 0] - v[:, :, 0].astype(np.float64))) <= 1e-3


def test_long_workload_rows_in_every_head():
    """The long workload (N = 32768, causal) at full size: tile-edge rows, the ragged end and
    24 random rows in every one of its 32 heads, which the oracle computes one by one."""
    w, q, k, v, kl = _workload_case("long")
    rows = sample_rows(w.B, w.H, w.N, seed=w.seed, per_head=24, heads=range(w.B * w.H))
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal,
                                 key_lengths=kl, rows=rows)
    for kern in _workload_kernels(w):
        o, lse = run_gpu(q, k, v, causal=w.causal, key_lengths=kl, path=kern)
        o_s = o.reshape(-1, w.d)[rows]
        lse_s = lse.reshape(-1)[rows]
        assert not np.isnan(o).any(), f"long {kern}: unwritten rows"
        compare(o_s, lse_s, o_ref, lse_ref, what=f"long {kern}")
        assert np.max(np.abs(o[:, :, 0] - v[:, :, 0].astype(np.float64))) <= 1e-3


@pytest.mark.parametrize("d", [32, 64, 128])
def test_uniform_keys_mean_of_v(d):
    """All keys equal: O is the mean of V over the allowed set (prefix means under causal)."""
    B, H, N = 1, 2, 300
    q, _, v, _ = synth.draw(B, H, N, d, seed=5)
    k = np.broadcast_to(synth.draw(B, H, 1, d, seed=6)[1], (B, H, N, d)).copy()
    kl = np.array([257], np.int32)
    for causal in (False, True):
        v64 = v.astype(np.float64)
        n_allowed = np.minimum(np.arange(N) + 1, kl[0]) if causal else np.full(N, kl[0])
        csum = np.cumsum(v64, axis=2)
        mean = csum[:, :, n_allowed - 1] / n_allowed[None, None, :, None]
        for kern in kernels_for(d, N):
            o, _ = run_gpu(q, k, v, causal=causal, key_lengths=kl, path=kern)
            assert np.max(np.abs(o - mean)) <= 1e-2, (kern, causal)


@pytest.mark.parametrize("d", [64, 128])
def test_one_hot_selection(d):
    """K_j = e_j, Q_i = 20 e_pi(i), scale 1: O_i = V_pi(i) (off-target weight < 1e-6)."""
    N = d
    rng = np.random.Generator(np.random.PCG64(9))
    k = np.eye(N, d, dtype=np.float16)[None, None]
    v = synth.draw(1, 1, N, d, seed=10)[2]
    for causal in (False, True):
        pi = np.array([rng.integers(0, i + 1) for i in range(N)]) if causal else rng.permutation(N)
        q = np.zeros((1, 1, N, d), np.float16)
        q[0, 0, np.arange(N), pi] = 20.0
        for kern in kernels_for(d, N):
            o, lse = run_gpu(q, k, v, causal=causal, sm_scale=1.0, path=kern)
            assert np.max(np.abs(o[0, 0] - v[0, 0, pi].astype(np.float64))) <= 2e-3, (kern, causal)
            assert np.max(np.abs(lse[0, 0] - 20.0)) <= 1e-3


@pytest.mark.parametrize("d", [32, 64, 128])
def test_empty_rows_zero_output(d):
    """key_lengths = 0 empties every row of that batch: O = 0 and lse = -inf."""
    q, k, v, _ = synth.draw(2, 2, 130, d, seed=12)
    kl = np.array([0, 130], np.int32)
    for kern in kernels_for(d, 130):
        o, lse = run_gpu(q, k, v, causal=False, key_lengths=kl, path=kern)
        assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)
        assert np.all(np.isfinite(lse[1]))


def test_deterministic():
    q, k, v, _ = synth.draw(2, 4, 700, 128, seed=13)
    for kern in kernels_for(128, 700):
        o1, l1 = run_gpu(q, k, v, causal=True, path=kern)
        o2, l2 = run_gpu(q, k, v, causal=True, path=kern)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), kern
    q, k, v, kl = synth.draw(50, 12, 256, 32, seed=16, key_len_range=(64, 256))
    for kern in kernels_for(32, 256):
        o1, l1 = run_gpu(q, k, v, causal=False, key_lengths=kl, path=kern)
        o2, l2 = run_gpu(q, k, v, causal=False, key_lengths=kl, path=kern)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), kern


def test_host_tensors_end_to_end():
    """CPU tensors go through the same C entry point with the copies done by the binding."""
    from exact_scaled_dot_attn_gb300 import api
    q, k, v, kl = synth.draw(2, 2, 160, 32, seed=14, key_len_range=(10, 160))
    o_ref, lse_ref = oracle_full(q, k, v, causal=False, key_lengths=kl)
    tq, tk, tv = (torch.from_numpy(x).pin_memory() for x in (q, k, v))
    o, lse = api.fwd(tq, tk, tv, key_lengths=torch.from_numpy(kl), return_lse=True)
    assert o.device.type == "cpu"
    compare(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, what="host")


@pytest.mark.parametrize("shape", [(4, 8, 2048, 128, 8, True), (1, 16, 8192, 128, 4, False)],
                         ids=["batch-pieces", "head-group-pieces"])
def test_host_tensors_in_pieces(shape):
    """Host problems of 64 MB and more go in pieces on two streams (along the batch, or along
    the key/value heads of one batch); the result is the one device call's, bit for bit."""
    from exact_scaled_dot_attn_gb300 import api
    B, H, N, d, Hkv, causal = shape
    q, k, v, kl = synth.draw_ex(B, H, Hkv, N, N, d, seed=15, key_len_range=(N // 2, N))
    assert api._host_pieces(torch.from_numpy(q), torch.from_numpy(k)) is not None
    tq, tk, tv = (torch.from_numpy(x).pin_memory() for x in (q, k, v))
    o_h, l_h = api.fwd(tq, tk, tv, causal=causal, key_lengths=torch.from_numpy(kl), return_lse=True)
    o_d, l_d = api.fwd(tq.cuda(), tk.cuda(), tv.cuda(), causal=causal,
                       key_lengths=torch.from_numpy(kl).cuda(), return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_non_default_stream():
    from exact_scaled_dot_attn_gb300 import api
    q, k, v, _ = synth.draw(1, 2, 257, 64, seed=15)
    o_ref, lse_ref = oracle_full(q, k, v, causal=True)
    s = torch.cuda.Stream()
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = api.fwd(qd, kd, vd, causal=True, return_lse=True)
    s.synchronize()
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, what="stream")
