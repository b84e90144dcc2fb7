"""GPU parity of the naive three-pass forward (attn_fwd_naive: S and P written to and read back
from device memory), element by element against the fp64 oracle.

Small shapes span several 128-row and 128-key tiles and end in ragged tails (the padded
columns of S and P), with the causal mask, key padding and rows that have no allowed key. The
measured workloads it serves (tiny, reranking, prefill, stress) run at full size on every row
(the reranking workload ignores its padded query rows), with lse. The workspace is filled with
NaN before each call, so a score or probability the passes fail to write would show.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import compare, ensure_built, oracle_full, to_dev, workload_oracle

pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, N, d, causal, key_lengths
    (1, 1, 1, 64, False, None),
    (1, 2, 65, 32, False, None),
    (2, 3, 127, 64, True, None),
    (2, 2, 200, 128, True, [150, 0]),
    (3, 1, 333, 64, False, [333, 1, 170]),
    (1, 2, 517, 32, True, [400]),
    (1, 1, 1000, 128, False, [999]),
]


def run_naive(q, k, v, *, causal, key_lengths=None, sm_scale=None):
    ensure_built()
    B, H, N, d = q.shape
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    kld = to_dev(key_lengths)
    ws = torch.full((api.naive_workspace_bytes(B, H, N) // 4,), float("nan"), dtype=torch.float32,
                    device="cuda")
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    api.fwd_naive(qd, kd, vd, causal=causal, sm_scale=sm_scale, key_lengths=kld,
                  return_lse=True, out=o, lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("shape", SMALL, ids=[f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{'c' if s[4] else ''}{'k' if s[5] else ''}" for s in SMALL])
def test_naive_small_shapes(shape):
    B, H, N, d, causal, kl = shape
    q, k, v, _ = synth.draw(B, H, N, d, seed=3000 + N + d)
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    o, lse = run_naive(q, k, v, causal=causal, key_lengths=kl)
    compare(o, lse, o_ref, lse_ref, what=f"naive {shape}")


def test_naive_wide_scale():
    """sm_scale = 2.5 makes rows peaked (scores spread over a wide range)."""
    q, k, v, _ = synth.draw(2, 2, 300, 64, seed=3077)
    o_ref, lse_ref = oracle_full(q, k, v, causal=True, sm_scale=2.5)
    o, lse = run_naive(q, k, v, causal=True, sm_scale=2.5)
    compare(o, lse, o_ref, lse_ref, what="naive scale 2.5")


@pytest.mark.parametrize("name", ["tiny", "rerank", "prefill", "stress"])
def test_naive_workload_full_rows(name):
    w, q, k, v, kl, o_ref, lse_ref = workload_oracle(name)
    row_mask = None
    if w.ignore_padded_queries:
        i = np.arange(w.N)[None, None, :]
        row_mask = np.broadcast_to(i < kl[:, None, None], (w.B, w.H, w.N))
    o, lse = run_naive(q, k, v, causal=w.causal, key_lengths=kl, sm_scale=w.sm_scale)
    compare(o, lse, o_ref, lse_ref, row_mask=row_mask, what=f"naive {name}")


def test_naive_refuses_other_types_and_small_workspace():
    ensure_built()
    q, k, v, _ = synth.draw(1, 2, 64, 64, seed=3090)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    with pytest.raises(TypeError):
        api.fwd_naive(qd.float(), kd.float(), vd.float())
    small = torch.empty(api.naive_workspace_bytes(1, 2, 64) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.AttnError) as exc:
        api.fwd_naive(qd, kd, vd, workspace=small)
    assert exc.value.status == _lib.ATTN_ERR_INVALID_ARG
