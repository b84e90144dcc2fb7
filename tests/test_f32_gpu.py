"""GPU parity of fp32 inputs at d = 32 (attn_fwd_ex / attn_fwd_splitkv_ex with ATTN_DTYPE_F32),
against the fp64 oracle on the same float32 inputs, on both of its paths:

- the automatic path (and ATTN_PATH_WARP_MMA): every operand of both products split into a TF32
  part and a TF32 remainder, each product formed from three TF32 products, fp32 accumulation,
  fp32 P and O. Bounds derived in tests/parity.py (`f32_split_bounds`): per element the worst
  case of the split products, fp32 sums and the exponential; over the tensor a relative L2
  error below 3e-5, thirty times under TF32's unit roundoff.
- ATTN_PATH_TCGEN05 and split-KV: TF32 products (`tf32_bounds`): inputs exact in TF32 (fp16
  values held as fp32) leave only P's truncation, |dO| <= 2^-10 max|V|; full-precision fp32
  inputs add the score perturbation of reading Q and K with 10 fraction bits.

Cases: self-attention with key padding and causal masks, cross-attention, grouped heads, a
causal draft block, the fp32 reranking workload at full size (every valid query row), and the
refusal of other head dimensions and of the short-sequence kernel.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import F32_REL_L2, compare, f32_split_bounds, run_gpu, tf32_bounds, to_dev
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
    """TF32 bounds (the tcgen05 kernel and split-KV)."""
    atol, lse_tol = tf32_bounds(q, k, v, 32 ** -0.5, exact_inputs=exact)
    m = None if row_mask is None else np.asarray(row_mask).reshape(-1)
    a = atol.reshape(-1, atol.shape[-1])
    r = o_ref.reshape(-1, o_ref.shape[-1])
    if m is not None:
        a, r = a[m], r[m]
    rel = float(np.linalg.norm(a) / max(np.linalg.norm(r), 1e-30))
    compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=rel, lse_tol=lse_tol, what=what,
            row_mask=row_mask)


def _check_f32(o, lse, o_ref, lse_ref, q, k, v, what, row_mask=None):
    """fp32 bounds (the split-TF32 path)."""
    atol, lse_tol = f32_split_bounds(q, k, v, 32 ** -0.5)
    return compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=F32_REL_L2, lse_tol=lse_tol,
                   what=what, row_mask=row_mask)


@pytest.mark.parametrize("exact", [True, False], ids=["tf32-exact", "full-fp32"])
@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_f32_matches_oracle(case, exact):
    B, H, Hkv, Nq, Nk, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, 32, seed=6000 + Nq + Nk, dtype="f32")
    if exact:  # values with 10 fraction bits: exact in TF32
        q, k, v = (x.astype(np.float16).astype(np.float32) for x in (q, k, v))
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = _oracle(q, k, v, causal=causal, key_lengths=kl)
    for path in ("auto", "warp_mma"):
        o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, dtype="f32", path=path)
        _check_f32(o, lse, o_ref, lse_ref, q, k, v, f"f32 {path} {_ids(case)}")
    o, lse = run_gpu(q, k, v, causal=causal, key_lengths=kl, dtype="f32", path="tcgen05")
    _check(o, lse, o_ref, lse_ref, q, k, v, exact, f"f32 tcgen05 {_ids(case)}")
    o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=2, dtype="f32")
    _check(o, lse, o_ref, lse_ref, q, k, v, exact, f"f32 splitkv {_ids(case)}")


def test_f32_wide_scores():
    """Scores spread over a wide range (sm_scale 1, Q and K scaled by 3, |s| up to hundreds): the
    split products stay within the per-element fp32 bounds, where TF32 products would move the
    softmax weights by percents; the relative L2 error is checked against the norm of those
    bounds."""
    q, k, v, _ = synth.draw_ex(2, 2, 2, 200, 200, 32, seed=6100, dtype="f32")
    q, k = q * 3.0, k * 3.0
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=1.0, causal=True, dtype="f32")
    o, lse = run_gpu(q, k, v, causal=True, sm_scale=1.0, dtype="f32")
    atol, lse_tol = f32_split_bounds(q, k, v, 1.0)
    rel = float(np.linalg.norm(atol) / np.linalg.norm(o_ref))
    compare(o, lse, o_ref, lse_ref, atol=atol, rel_l2=rel, lse_tol=lse_tol, what="f32 wide")


def test_f32_rerank_workload_all_rows():
    """The reranking shape with fp32 inputs at full size; padded query rows are not compared
    (the workload ignores them), every other row is: the automatic (fp32-accurate) path against
    the fp32 bounds, the TF32 kernel against the TF32 bounds."""
    w = synth.WORKLOADS["rerank_f32"]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = _oracle(q, k, v, causal=w.causal, key_lengths=kl)
    rows = np.arange(w.N)[None, None, :] < kl[:, None, None]
    mask = np.broadcast_to(rows, (w.B, w.H, w.N))
    o, lse = run_gpu(q, k, v, causal=w.causal, key_lengths=kl, dtype="f32")
    err = _check_f32(o, lse, o_ref, lse_ref, q, k, v, "rerank_f32", row_mask=mask)
    assert err["rel_l2"] <= F32_REL_L2
    o, lse = run_gpu(q, k, v, causal=w.causal, key_lengths=kl, dtype="f32", path="tcgen05")
    _check(o, lse, o_ref, lse_ref, q, k, v, False, "rerank_f32 tcgen05", row_mask=mask)


def test_f32_refuses_other_head_dims_and_kernels():
    q, k, v, _ = synth.draw_ex(1, 2, 2, 64, 64, 64, seed=79, dtype="f32")
    for path in ("auto", "warp_mma", "tcgen05"):
        with pytest.raises(_lib.AttnError) as exc:
            api.fwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"), path=path)
        assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED
    q, k, v, _ = synth.draw_ex(1, 2, 2, 64, 64, 32, seed=80, dtype="f32")
    with pytest.raises(_lib.AttnError) as exc:
        api.fwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"), path="short")
    assert exc.value.status == _lib.ATTN_ERR_UNSUPPORTED
