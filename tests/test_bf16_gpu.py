"""GPU parity of bf16 inputs (attn_fwd_ex / attn_fwd_splitkv_ex with ATTN_DTYPE_BF16) on the
tcgen05 kernel, against the fp64 oracle decoding the same bfloat16 bit patterns.

Tolerances follow from bf16's unit roundoff u = 2^-8 (tests/parity.py): per element
|dO| <= u (|O_ref| + max|V|) + 1e-3, relative L2 <= 2u, lse within 1e-3. Cases: self-attention,
cross-attention and grouped-query heads, every head dimension, causal and key padding,
split-KV, the bf16 prefill workload at full size on sampled rows, and inputs beyond fp16's range.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import (TOL_REL_L2_BF16, bf16_atol, compare, oracle_full, run_gpu, sample_rows,
                    to_dev)
from test_splitkv_gpu import run_splitkv

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, H_kv, N_q, N_k, d, causal, key_lengths
    (1, 2, 2, 256, 256, 128, True, None),
    (2, 3, 3, 333, 333, 64, False, [333, 17]),
    (3, 2, 2, 129, 129, 32, True, [129, 1, 0]),
    (2, 8, 2, 300, 700, 128, True, None),
    (1, 4, 1, 640, 200, 64, True, [200]),
    (2, 4, 2, 65, 65, 32, False, None),
    (2, 8, 2, 4, 500, 64, True, [500, 77]),    # causal draft block, query groups packed
    (3, 8, 4, 1, 700, 128, True, None),        # one query per sequence, packed
]


def _ids(c):
    return (f"B{c[0]}H{c[1]}kv{c[2]}Nq{c[3]}Nk{c[4]}d{c[5]}{'c' if c[6] else ''}"
            f"{'k' if c[7] else ''}")


def _oracle_bf16(q, k, v, *, causal, key_lengths=None, sm_scale=None, rows=None):
    d = q.shape[-1]
    return oracle.attn(q, k, v, sm_scale=(d ** -0.5 if sm_scale is None else sm_scale),
                       causal=causal, key_lengths=key_lengths, rows=rows, dtype="bf16")


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_bf16_matches_oracle(case):
    B, H, Hkv, Nq, Nk, d, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, d, seed=5000 + Nq + Nk + d, dtype="bf16")
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = _oracle_bf16(q, k, v, causal=causal, key_lengths=kl)
    atol = bf16_atol(o_ref, v)
    o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, dtype="bf16")
    compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=TOL_REL_L2_BF16, what=f"bf16 {_ids(case)}")
    o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=3, dtype="bf16")
    compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=TOL_REL_L2_BF16,
            what=f"bf16 splitkv {_ids(case)}")


def test_bf16_beyond_fp16_range():
    """Q scaled by 2^17 and K by 2^-17: Q overflows fp16 (max 65504) but is exact in bf16's
    range; the scores, and so the result, are those of the unscaled problem."""
    B, H, N, d = 1, 2, 300, 64
    rng = np.random.Generator(np.random.PCG64(77))
    q32 = rng.standard_normal((B, H, N, d), dtype=np.float32)
    k32 = rng.standard_normal((B, H, N, d), dtype=np.float32)
    v32 = rng.standard_normal((B, H, N, d), dtype=np.float32)
    q = synth.to_bf16_bits(q32 * np.float32(2.0 ** 17))
    k = synth.to_bf16_bits(k32 * np.float32(2.0 ** -17))
    v = synth.to_bf16_bits(v32)
    o_ref, lse_ref = _oracle_bf16(q, k, v, causal=True)
    o, lse = run_gpu(q, k, v, causal=True, dtype="bf16")
    compare(o, lse, o_ref, lse_ref, atol=bf16_atol(o_ref, v), rel_l2=TOL_REL_L2_BF16,
            what="bf16 large range")
    # the same problem unscaled gives the same oracle result (scaling by powers of two is exact)
    o2, lse2 = _oracle_bf16(synth.to_bf16_bits(q32), synth.to_bf16_bits(k32), v, causal=True)
    assert np.array_equal(o_ref, o2) and np.array_equal(lse_ref, lse2)


def test_bf16_other_paths_refused():
    q, k, v, _ = synth.draw_ex(1, 2, 2, 64, 64, 32, seed=78, dtype="bf16")
    for path in ("warp_mma", "short"):
        with pytest.raises(_lib.AttnError) as exc:
            api.fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), path=path)
        assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED


def test_bf16_prefill_workload_all_rows():
    """The bf16 prefill workload at full size, every row against the oracle's bf16 decode."""
    w = synth.WORKLOADS["prefill_bf16"]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = _oracle_bf16(q, k, v, causal=w.causal, key_lengths=kl, sm_scale=w.sm_scale)
    o, lse = api.fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), causal=w.causal,
                     sm_scale=w.sm_scale, return_lse=True)
    assert api.read_device_status() == _lib.ATTN_OK
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    compare(o, lse, o_ref, lse_ref, atol=bf16_atol(o_ref, v), rel_l2=TOL_REL_L2_BF16,
            what="prefill_bf16")
