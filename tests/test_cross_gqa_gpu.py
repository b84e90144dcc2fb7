"""GPU parity of cross-attention and grouped-query attention (attn_fwd_ex, attn_fwd_splitkv_ex):
queries [B, H, N_q, d] over keys and values [B, H_kv, N_k, d], query head h reading key/value
head h // (H // H_kv), and under the causal mask query i seeing keys j <= i + N_k - N_q.

Every case runs through the C ABI on the tcgen05 and warp-level kernels, on the decoding kernel
where it fits (at most 16 query rows per head after packing), and on split-KV, and is
compared element by element with the fp64 oracle: query blocks shorter and longer than the key
sequence (the latter with leading rows that see no key), one query row, ragged lengths, key
padding, every head dimension and group size 1 (multi-query) to H (multi-head). The two
grouped-query workloads run at full size on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import compare, ensure_built, oracle_full, run_gpu, sample_rows, to_dev
from test_splitkv_gpu import run_splitkv

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, H_kv, N_q, N_k, d, causal, key_lengths
    (2, 8, 2, 300, 300, 64, True, None),
    (2, 6, 1, 257, 257, 128, False, [257, 100]),
    (1, 4, 4, 128, 1000, 128, True, None),
    (2, 4, 2, 1000, 128, 64, True, None),
    (1, 8, 2, 1, 4096, 128, True, None),
    (3, 4, 1, 77, 333, 32, False, [333, 20, 0]),
    (2, 2, 1, 513, 257, 32, True, [257, 130]),
    (1, 3, 3, 200, 64, 128, False, None),
    (2, 4, 4, 384, 640, 64, True, [640, 300]),
    # decode-sized query blocks: the G query heads of a group run as G * N_q packed rows
    (2, 8, 2, 1, 1000, 128, True, [1000, 37]),
    (3, 12, 4, 5, 300, 64, False, [300, 1, 0]),
    (1, 32, 8, 16, 2048, 128, False, None),
    (2, 4, 1, 1, 64, 32, True, None),
    (2, 8, 2, 16, 64, 32, False, [64, 20]),   # packed: 64 rows over 64 keys, a self-attention shape
    # causal blocks of several queries (speculative decoding): packed rows, row r = query r % N_q
    (1, 8, 2, 4, 500, 64, True, None),
    (2, 8, 2, 7, 300, 128, True, [300, 150]),
    (1, 16, 2, 16, 1000, 64, True, None),
    (2, 12, 4, 33, 129, 32, True, [129, 5]),
    (1, 4, 2, 127, 700, 128, True, None),
    (1, 4, 2, 40, 30, 64, True, None),         # N_q > N_k: the first 10 queries of a head see no key
    (1, 4, 2, 128, 300, 64, True, None),       # 128 query rows: not packed
]


def _ids(c):
    return (f"B{c[0]}H{c[1]}kv{c[2]}Nq{c[3]}Nk{c[4]}d{c[5]}{'c' if c[6] else ''}"
            f"{'k' if c[7] else ''}")


def _draw(case, seed):
    B, H, Hkv, Nq, Nk, d, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, d, seed=seed)
    return q, k, v, (None if kl is None else np.array(kl, np.int32))


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_cross_gqa_matches_oracle(case):
    B, H, Hkv, Nq, Nk, d, causal, _ = case
    q, k, v, kl = _draw(case, seed=3000 + Nq + Nk + d + Hkv)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    packed_rows = (H // Hkv) * Nq if (Hkv < H and Nq < 128) else Nq
    kernels = ("tcgen05", "warp_mma") + (("decode",) if packed_rows <= _lib.DECODE_MAX_ROWS else ())
    for kern in kernels:
        o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, path=kern)
        compare(o, lse, o_ref, lse_ref, what=f"{kern} {_ids(case)}")
    for S in (2, 0):
        o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=S)
        compare(o, lse, o_ref, lse_ref, what=f"splitkv S={S} {_ids(case)}")


def test_gqa_equals_repeated_kv_heads():
    """The library's grouped-query result against its own multi-head result with each K/V head
    repeated for its group: the same attention, so the same bits on the same kernel."""
    B, H, Hkv, N, d = 2, 8, 2, 700, 128
    q, k, v, _ = synth.draw_ex(B, H, Hkv, N, N, d, seed=41)
    g = H // Hkv
    o1, l1 = run_gpu(q, k, v, causal=True, path="tcgen05")
    o2, l2 = run_gpu(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), causal=True,
                     path="tcgen05")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_cross_causal_leading_rows_empty():
    """N_q > N_k under the causal mask: the first N_q - N_k queries see no key (O = 0,
    lse = -inf); query N_q - N_k sees key 0 only, so its output is V_0."""
    B, H, Nq, Nk, d = 1, 2, 400, 150, 64
    q, k, v, _ = synth.draw_ex(B, H, H, Nq, Nk, d, seed=42)
    for kern in ("tcgen05", "warp_mma"):
        o, lse = run_gpu(q, k, v, causal=True, path=kern)
        e = Nq - Nk
        assert np.all(o[:, :, :e] == 0.0) and np.all(lse[:, :, :e] == -np.inf), kern
        assert np.max(np.abs(o[:, :, e] - v[:, :, 0].astype(np.float64))) <= 1e-3, kern


def test_short_path_refuses_cross_shapes():
    ensure_built()
    q, k, v, _ = synth.draw_ex(1, 2, 1, 64, 64, 32, seed=43)
    with pytest.raises(_lib.AttnError) as exc:
        api.fwd(to_dev(q), to_dev(k), to_dev(v), path="short")
    assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["gqa_prefill", "chunk_prefill"])
def test_gqa_workload_all_rows(name):
    """The grouped-query workloads at full size, every row against the oracle."""
    w = synth.WORKLOADS[name]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal, key_lengths=kl)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, return_lse=True)
    assert api.read_device_status() == _lib.ATTN_OK
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    compare(o, lse, o_ref, lse_ref, what=name)
