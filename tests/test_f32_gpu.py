"""GPU parity of fp32 inputs at d = 32 (attn_fwd_ex / attn_fwd_splitkv_ex with ATTN_DTYPE_F32):
both products on the tensor cores as TF32, fp32 accumulation, fp32 output, against the fp64
oracle on the same float32 inputs.

Bounds (derived in tests/parity.py, `tf32_bounds`): inputs exact in TF32 (fp16 values held as
fp32) leave only P's truncation, |dO| <= 2^-10 max|V|; full-precision fp32 inputs add the score
perturbation of reading Q and K with 10 fraction bits. Cases: self-attention with key padding
and causal masks, cross-attention, grouped heads, split-KV, the fp32 reranking workload at full
size (every valid query row), and the refusal of other head dimensions and kernels.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import compare, run_gpu, tf32_bounds, to_dev
from test_splitkv_gpu import run_splitkv

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, H_kv, N_q, N_k, causal, key_lengths
    (3, 4, 4, 256, 256, False, [256, 64, 0]),
    (2, 2, 2, 300, 300, True, None),
    (2, 8, 2, 200, 517, True, [517, 100]),
    (1, 4, 1, 640, 130, False, None),
    (2, 8, 2, 5, 400, True, [400, 33]),        # causal draft block, query groups packed
]


def _ids(c):
    return f"B{c[0]}H{c[1]}kv{c[2]}Nq{c[3]}Nk{c[4]}{'c' if c[5] else ''}{'k' if c[6] else ''}"


def _oracle(q, k, v, *, causal, key_lengths=None, rows=None):
    return oracle.attn(q, k, v, sm_scale=32 ** -0.5, causal=causal, key_lengths=key_lengths,
                       rows=rows, dtype="f32")


def _check(o, lse, o_ref, lse_ref, q, k, v, exact, what, row_mask=None):
    atol, lse_tol = tf32_bounds(q, k, v, 32 ** -0.5, exact_inputs=exact)
    m = None if row_mask is None else np.asarray(row_mask).reshape(-1)
    a = atol.reshape(-1, atol.shape[-1])
    r = o_ref.reshape(-1, o_ref.shape[-1])
    if m is not None:
        a, r = a[m], r[m]
    rel = float(np.linalg.norm(a) / max(np.linalg.norm(r), 1e-30))
    compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=rel, lse_tol=lse_tol, what=what,
            row_mask=row_mask)


@pytest.mark.parametrize("exact", [True, False], ids=["tf32-exact", "full-fp32"])
@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_f32_matches_oracle(case, exact):
    B, H, Hkv, Nq, Nk, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, 32, seed=6000 + Nq + Nk, dtype="f32")
    if exact:  # values with 10 fraction bits: exact in TF32
        q, k, v = (x.astype(np.float16).astype(np.float32) for x in (q, k, v))
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = _oracle(q, k, v, causal=causal, key_lengths=kl)
    o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, dtype="f32")
    _check(o, lse, o_ref, lse_ref, q, k, v, exact, f"f32 {_ids(case)}")
    o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=2, dtype="f32")
    _check(o, lse, o_ref, lse_ref, q, k, v, exact, f"f32 splitkv {_ids(case)}")


def test_f32_rerank_workload_all_rows():
    """The reranking shape with fp32 inputs at full size; padded query rows are not compared
    (the workload ignores them), every other row is."""
    w = synth.WORKLOADS["rerank_f32"]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = _oracle(q, k, v, causal=w.causal, key_lengths=kl)
    o, lse = run_gpu(q, k, v, causal=w.causal, key_lengths=kl, dtype="f32")
    rows = np.arange(w.N)[None, None, :] < kl[:, None, None]
    mask = np.broadcast_to(rows, (w.B, w.H, w.N))
    _check(o, lse, o_ref, lse_ref, q, k, v, False, "rerank_f32", row_mask=mask)


def test_f32_refuses_other_head_dims_and_kernels():
    q, k, v, _ = synth.draw_ex(1, 2, 2, 64, 64, 64, seed=79, dtype="f32")
    with pytest.raises(_lib.AttnError) as exc:
        api.fwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"))
    assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED
    q, k, v, _ = synth.draw_ex(1, 2, 2, 64, 64, 32, seed=80, dtype="f32")
    for path in ("warp_mma", "short"):
        with pytest.raises(_lib.AttnError) as exc:
            api.fwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"), path=path)
        assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED
