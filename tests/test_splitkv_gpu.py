"""GPU parity of split-KV (attn_fwd_splitkv): the keys of every query tile pair are divided
into ranges that run as separate units and are merged through their logsumexps. The result
is the same attention, so it is compared with the fp64 oracle like every other path, with
several split counts (more ranges than key tiles, empty batches, ragged lengths) and one long
single-head sequence with the automatic split count."""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, synth
from parity import compare, ensure_built, oracle_full, sample_rows, to_dev

pytestmark = pytest.mark.gpu


def run_splitkv(q, k, v, *, causal, key_lengths=None, sm_scale=None, n_splits=0, dtype="f16"):
    """attn_fwd_splitkv on device copies; O and lse sit inside guarded, NaN-prefilled buffers."""
    ensure_built()
    B, H, N, d = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    kld = to_dev(key_lengths)
    pad_o, pad_l = 4096, 1024
    n_o, n_l = q.size, B * H * N
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}.get(dtype, torch.float16)
    o_buf = torch.full((n_o + 2 * pad_o,), float("nan"), dtype=tdt, device="cuda")
    l_buf = torch.full((n_l + 2 * pad_l,), float("nan"), dtype=torch.float32, device="cuda")
    o_buf[:pad_o] = 1234.0
    o_buf[pad_o + n_o:] = 1234.0
    l_buf[:pad_l] = 4321.0
    l_buf[pad_l + n_l:] = 4321.0
    o = o_buf[pad_o:pad_o + n_o].view(B, H, N, d)
    lse = l_buf[pad_l:pad_l + n_l].view(B, H, N)
    api.fwd_splitkv(qd, kd, vd, causal=causal, sm_scale=sm_scale, key_lengths=kld,
                    return_lse=True, out=o, lse_out=lse, n_splits=n_splits)
    assert api.read_device_status() == _lib.ATTN_OK
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad_o] == 1234.0) and torch.all(o_buf[pad_o + n_o:] == 1234.0)
    assert torch.all(l_buf[:pad_l] == 4321.0) and torch.all(l_buf[pad_l + n_l:] == 4321.0)
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


CASES = [
    # B, H, N, d, causal, key_lengths, n_splits
    (1, 2, 300, 64, True, None, 2),
    (2, 1, 517, 128, True, [517, 77], 3),
    (1, 1, 1000, 32, False, [999], 5),
    (3, 2, 256, 64, False, [256, 1, 0], 2),
    (1, 1, 130, 128, False, None, 16),
    (2, 2, 640, 64, True, None, 4),
    (1, 3, 1024, 128, False, None, 7),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{'c' if c[4] else ''}S{c[6]}" for c in CASES])
def test_splitkv_matches_oracle(case):
    B, H, N, d, causal, kl, S = case
    q, k, v, _ = synth.draw(B, H, N, d, seed=2000 + N + d + S)
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=S)
    compare(o, lse, o_ref, lse_ref, what=f"splitkv {case}")


def test_splitkv_long_single_head_auto():
    """One long causal sequence per head (few query tile pairs): the automatic split count."""
    B, H, N, d = 1, 2, 8192, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=31)
    rows = sample_rows(B, H, N, seed=31, per_head=32)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=True, rows=rows)
    o, lse = run_splitkv(q, k, v, causal=True, n_splits=0)
    assert not np.isnan(o).any()
    compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, what="splitkv auto")
    # causal row 0: O_0 = V_0
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0].astype(np.float64))) <= 1e-3


def test_splitkv_uniform_keys_mean_of_v():
    """All keys equal: every range sees equal scores, and the merge must give the mean of V."""
    B, H, N, d = 1, 2, 700, 64
    q, _, v, _ = synth.draw(B, H, N, d, seed=32)
    k = np.broadcast_to(synth.draw(B, H, 1, d, seed=33)[1], (B, H, N, d)).copy()
    o, _ = run_splitkv(q, k, v, causal=False, n_splits=3)
    mean = v.astype(np.float64).mean(axis=2, keepdims=True)
    assert np.max(np.abs(o - mean)) <= 1e-2


def test_splitkv_agrees_with_unsplit_path():
    B, H, N, d = 2, 4, 1536, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=34)
    o1, l1 = run_splitkv(q, k, v, causal=True, n_splits=4)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o2, l2 = api.fwd(qd, kd, vd, causal=True, return_lse=True, path="tcgen05")
    torch.cuda.synchronize()
    assert np.max(np.abs(o1 - o2.double().cpu().numpy())) <= 4e-3
    assert np.max(np.abs(l1 - l2.double().cpu().numpy())) <= 1e-4


def test_splitkv_one_head_workload_all_rows():
    """The workload split-KV is measured on (one long causal head), full size, every row."""
    w = synth.WORKLOADS["one_head"]
    q, k, v, kl = synth.draw_workload(w)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal)
    o, lse = run_splitkv(q, k, v, causal=w.causal, n_splits=0)
    compare(o, lse, o_ref, lse_ref, what="one_head splitkv")


BALANCED = [
    # B, H, H_kv, N_q, N_k, d, causal, ragged key lengths
    (32, 32, 8, 1, 8192, 128, True, False),
    (32, 32, 8, 1, 8192, 128, True, True),
]


@pytest.mark.parametrize("case", BALANCED, ids=["decode", "decode-ragged"])
def test_splitkv_balanced_runs_decode(case):
    """A decoding batch large enough that the automatic split lays the key tiles of all
    (head, pair) units end to end and cuts them into one equal run per SM (two ranges per pair
    where an equal split would take one): every row against the oracle. Ragged key lengths
    leave ranges past a batch's keys empty."""
    B, H, Hkv, Nq, Nk, d, causal, ragged = case
    assert _lib.lib().attn_splitkv_auto_splits_ex(B, H, Hkv, Nq, Nk, d, int(causal)) >= 2
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, d, seed=2100 + int(ragged))
    kl = None
    if ragged:
        rng = np.random.Generator(np.random.PCG64(2102))
        kl = rng.integers(1, Nk + 1, size=B).astype(np.int32)
        kl[0], kl[1] = 1, Nk
    o_ref, lse_ref = oracle_full(q, k, v, causal=causal, key_lengths=kl)
    o, lse = run_splitkv(q, k, v, causal=causal, key_lengths=kl, n_splits=0)
    compare(o, lse, o_ref, lse_ref, what=f"balanced decode ragged={ragged}")


def test_splitkv_balanced_runs_single_pair_causal():
    """Causal self-attention with one Q tile pair per head (every pair sees the same key tiles)
    at a size where the automatic split may use balanced runs; sampled rows."""
    B, H, N, Nk, d = 8, 16, 200, 8192, 128
    q, k, v, _ = synth.draw_ex(B, H, H, N, Nk, d, seed=2110)
    rows = sample_rows(B, H, N, seed=2111, per_head=16)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=True, rows=rows)
    o, lse = run_splitkv(q, k, v, causal=True, n_splits=0)
    assert not np.isnan(o).any()
    compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, what="balanced causal pair")
