"""GPU parity of the decoding kernel (ATTN_PATH_DECODE; the automatic choice for at most 16
query rows per head, after query-group packing, over at least ATTN_DECODE_MIN_KEYS keys).

A head is handled by a thread-block cluster of 1 to 8 CTAs, each streaming a contiguous share of
the head's 32-key tiles, and the CTAs merge their (m, l, O) through distributed shared memory.
Every case is compared element by element with the fp64 oracle at the stated tolerances:
packed query groups of 2 to 16 rows (one query, and causal draft blocks whose rows keep their
own query's diagonal), unpacked multi-head decoding with 1 to 16 query rows, key padding with
zero and one valid key, fewer keys than one tile, more query rows than keys (rows that see no
key: O = 0, lse = -inf), a single head split over eight CTAs with a ragged last tile, every head
dimension, bf16 inputs, and the decoding workload at full size on every row. Results are
bit-identical from launch to launch (a fixed merge order).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import (TOL_REL_L2_BF16, bf16_atol, compare, ensure_built, oracle_full, run_gpu,
                    to_dev)

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, H_kv, N_q, N_k, d, causal, key_lengths
    (2, 8, 2, 1, 1000, 128, True, [1000, 37]),      # 4 packed rows, key padding
    (3, 12, 4, 5, 300, 64, False, [300, 1, 0]),     # 15 packed rows; one key; no key
    (2, 4, 1, 1, 64, 32, True, None),               # 4 packed rows over two tiles
    (1, 8, 2, 4, 500, 64, True, None),              # causal block of 4 queries x 4 heads
    (2, 16, 2, 2, 4096, 128, True, [4096, 999]),    # 16 packed rows, row r = query r % 2
    (1, 4, 4, 3, 777, 64, True, None),              # unpacked: 3 query rows per head
    (1, 2, 2, 5, 3, 32, True, None),                # 5 queries over 3 keys: 2 empty rows
    (1, 1, 1, 1, 5000, 128, False, None),           # one head over 8 CTAs, ragged last tile
    (4, 8, 8, 1, 2500, 64, True, [2500, 1, 1250, 33]),  # multi-head decoding
    (1, 16, 1, 1, 3000, 64, True, None),            # multi-query: 16 packed rows
    (2, 16, 2, 1, 2048, 128, False, None),          # 8 packed rows
    (2, 4, 4, 16, 900, 32, False, [17, 900]),       # 16 unpacked rows
    (1, 2, 2, 1, 20, 64, False, None),              # fewer keys than one tile
]


def _ids(c):
    return (f"B{c[0]}H{c[1]}kv{c[2]}Nq{c[3]}Nk{c[4]}d{c[5]}{'c' if c[6] else ''}"
            f"{'k' if c[7] else ''}")


def _draw(case, seed, dtype="f16"):
    B, H, Hkv, Nq, Nk, d, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, d, seed=seed, dtype=dtype)
    return q, k, v, (None if kl is None else np.array(kl, np.int32))


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_decode_matches_oracle(case):
    B, H, Hkv, Nq, Nk, d, causal, _ = case
    q, k, v, kl = _draw(case, seed=9000 + Nq + Nk + d + Hkv)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, path="decode")
    compare(o, lse, o_ref, lse_ref, what=f"decode {_ids(case)}")


def test_empty_rows_and_single_key():
    """N_q > N_k under the causal mask: queries 0 and 1 of 5 over 3 keys see no key (O = 0,
    lse = -inf); query 2 sees key 0 only, so its output is V_0 and its lse the one score."""
    q, k, v, _ = synth.draw_ex(1, 2, 2, 5, 3, 32, seed=9101)
    o, lse = run_gpu(q, k, v, causal=True, path="decode")
    assert np.all(o[:, :, :2] == 0.0) and np.all(lse[:, :, :2] == -np.inf)
    assert np.max(np.abs(o[:, :, 2] - v[:, :, 0].astype(np.float64))) <= 1e-3
    s = (q[:, :, 2].astype(np.float64) * k[:, :, 0].astype(np.float64)).sum(-1) / np.sqrt(32)
    assert np.max(np.abs(lse[:, :, 2] - s)) <= 1e-3


@pytest.mark.parametrize("case", [(2, 8, 2, 4, 500, 64, True, [500, 77]),
                                  (3, 8, 4, 1, 700, 128, True, None),
                                  (2, 4, 4, 2, 1500, 32, False, [1500, 2])],
                         ids=_ids)
def test_decode_bf16(case):
    B, H, Hkv, Nq, Nk, d, causal, _ = case
    q, k, v, kl = _draw(case, seed=9200 + Nq + Nk + d, dtype="bf16")
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=causal, key_lengths=kl,
                                 dtype="bf16")
    o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, path="decode", dtype="bf16")
    compare(o, lse, o_ref, lse_ref, atol=bf16_atol(o_ref, v), rel_l2=TOL_REL_L2_BF16,
            what=f"decode bf16 {_ids(case)}")


def test_auto_path_takes_the_decoding_kernel():
    assert api.auto_path_ex(32, 8, 1, 8192, 128, "f16", True) == "decode"
    assert api.auto_path_ex(32, 8, 4, 8192, 128, "bf16", True) == "decode"
    assert api.auto_path_ex(32, 8, 8, 8192, 128, "f16", True) == "tcgen05"   # 32 packed rows
    assert api.auto_path_ex(32, 8, 1, 255, 128, "f16", True) == "tcgen05"    # too few keys
    assert api.auto_path_ex(4, 4, 16, 8192, 64, "f16", False) == "decode"
    assert api.auto_path_ex(4, 4, 17, 8192, 64, "f16", False) == "tcgen05"
    # the automatic path gives the explicit decoding kernel's bits
    case = (2, 8, 2, 1, 1000, 128, True, [1000, 37])
    q, k, v, kl = _draw(case, seed=9300)
    o1, l1 = run_gpu(q, k, v, causal=True, key_lengths=kl, path="decode")
    o2, l2 = run_gpu(q, k, v, causal=True, key_lengths=kl)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_decode_deterministic():
    case = (1, 1, 1, 1, 5000, 128, False, None)
    q, k, v, kl = _draw(case, seed=9400)
    runs = [run_gpu(q, k, v, causal=False, path="decode") for _ in range(3)]
    for o, lse in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(lse, runs[0][1])


def test_decode_workload_all_rows():
    """The decoding workload at full size (B = 8, 32 query heads over 8, one query over 8192
    keys, d = 128), every row against the oracle, through the automatic path."""
    w = synth.WORKLOADS["decode_gqa"]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal, key_lengths=kl)
    ensure_built()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, return_lse=True)
    assert api.read_device_status() == _lib.ATTN_OK
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, what=w.name)


def test_decode_streams_and_graph():
    """Two launches on two streams at once, and a launch replayed from a CUDA graph, give the
    plain launch's bits."""
    case = (8, 32, 8, 1, 4096, 128, True, None)
    q, k, v, _ = _draw(case, seed=9500)
    ensure_built()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    ref = api.fwd(qd, kd, vd, causal=True, path="decode").clone()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, o2 = torch.empty_like(qd), torch.empty_like(qd)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        api.fwd(qd, kd, vd, causal=True, out=o1, path="decode")
    with torch.cuda.stream(s2):
        api.fwd(qd, kd, vd, causal=True, out=o2, path="decode")
    torch.cuda.synchronize()
    assert torch.equal(o1, ref) and torch.equal(o2, ref)
    o3 = torch.empty_like(qd)
    with torch.cuda.stream(s1):  # warm-up outside the capture
        api.fwd(qd, kd, vd, causal=True, out=o3, path="decode")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        api.fwd(qd, kd, vd, causal=True, out=o3, path="decode")
    for _ in range(3):
        o3.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o3, ref)
