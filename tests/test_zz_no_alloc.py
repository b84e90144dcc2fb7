"""The split-KV forward that allocates nothing (attn_fwd_splitkv_noalloc), through the C ABI.

Some callers cannot allocate device memory where they call the attention: their device memory
already belongs to their own pool or caching allocator, the runtime that hosts them gives them
no allocator, or their request loop cannot afford the synchronisation of cudaMalloc/cudaFree.
This entry point serves them from a fixed scratch array inside the library, so its results must
be those of the allocating entry points. Calls in a row on different problems (a later call
must not be affected by what an earlier one left in the shared array) are each compared with
the fp64 oracle and with attn_fwd_lse on the same inputs, within the parity tolerances of the
other GPU tests. One case takes the automatic split count, lowered by the entry point until its
partials fit the array. After a warm-up call, a further call leaves the device's free memory
unchanged.

The file name makes pytest collect it last, so a run that stops at the first failure has run
every other test before it; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_attn_gb300 import _lib, build, synth

pytestmark = pytest.mark.gpu

TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 2e-3
TOL_LSE = 1e-3


def _call(fn, q, k, v, o, lse, causal, kl, n_splits=None):
    B, H, N, d = q.shape
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(d ** -0.5), int(causal), kl.data_ptr() if kl is not None else None]
    if n_splits is not None:
        args.append(n_splits)
    args.append(torch.cuda.current_stream().cuda_stream)
    return fn(*args)


def _check(a, b, la, lb, what):
    """a, la: the no-allocation result (or the rows of it being checked); b, lb: what it must
    match on the same rows."""
    assert not np.isnan(a).any(), what
    assert np.max(np.abs(a - b)) <= TOL_MAX_ABS, what
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL_REL_L2, what
    assert np.array_equal(np.isfinite(la), np.isfinite(lb)), what
    fin = np.isfinite(lb)
    assert np.all(la[~fin] == -np.inf), what
    if fin.any():
        assert np.max(np.abs(la[fin] - lb[fin])) <= TOL_LSE, what


CASES = [
    # B, H, N, d, causal, key_lengths, n_splits (0: automatic, lowered to fit the array)
    (1, 2, 2000, 128, True, None, 3),
    (2, 3, 700, 64, False, [700, 123], 2),
    (1, 4, 16384, 128, True, None, 0),
]


def test_noalloc_matches_oracle_and_allocating_entry_point():
    build.build()
    L = _lib.lib()
    cap = L.attn_noalloc_scratch_bytes()
    for B, H, N, d, causal, kl, S in CASES:
        if S > 0:
            assert L.attn_splitkv_workspace_bytes(B, H, N, d, S) <= cap
        else:
            # the automatic count alone would overflow the array; one range fits
            auto = L.attn_splitkv_auto_splits(B, H, N, d, int(causal))
            assert L.attn_splitkv_workspace_bytes(B, H, N, d, auto) > cap
            assert L.attn_splitkv_workspace_bytes(B, H, N, d, 1) <= cap
        q, k, v, _ = synth.draw(B, H, N, d, seed=500 + N)
        kl_np = np.array(kl, np.int32) if kl is not None else None
        qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
        kld = torch.from_numpy(kl_np).cuda() if kl is not None else None
        o1 = torch.full_like(qd, float("nan"))
        o2 = torch.full_like(qd, float("nan"))
        l1 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        l2 = torch.full_like(l1, float("nan"))
        assert _call(L.attn_fwd_splitkv_noalloc, qd, kd, vd, o1, l1, causal, kld, S) == _lib.ATTN_OK
        assert _call(L.attn_fwd_lse, qd, kd, vd, o2, l2, causal, kld) == _lib.ATTN_OK
        assert L.attn_read_device_status(torch.cuda.current_stream().cuda_stream) == _lib.ATTN_OK
        torch.cuda.synchronize()
        a, b = o1.double().cpu().numpy(), o2.double().cpu().numpy()
        la, lb = l1.double().cpu().numpy(), l2.double().cpu().numpy()
        what = f"B={B} H={H} N={N} d={d} causal={causal} S={S}"
        _check(a, b, la, lb, what + " vs attn_fwd_lse")
        # against the oracle: every row of the small cases, sampled rows of the long one
        if B * H * N <= 8192:
            o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=causal,
                                         key_lengths=kl_np)
            _check(a, o_ref, la, lse_ref, what + " vs oracle")
        else:
            rng = np.random.Generator(np.random.PCG64(N))
            rows = np.unique(np.concatenate([
                np.array([0, 1, 127, 128, 255, 256, N - 1]),
                rng.integers(0, B * H * N, size=200)])).astype(np.int64)
            o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=causal,
                                         key_lengths=kl_np, rows=rows)
            _check(a.reshape(-1, d)[rows], o_ref, la.reshape(-1)[rows], lse_ref,
                   what + " vs oracle (sampled rows)")


def test_noalloc_call_allocates_nothing():
    """After a warm-up call (which may make the driver load the library's device code and
    reserve the array), another call leaves the device's free memory as it was."""
    build.build()
    L = _lib.lib()
    B, H, N, d = 2, 4, 1500, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=501)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    assert _call(L.attn_fwd_splitkv_noalloc, qd, kd, vd, o, lse, True, None, 2) == _lib.ATTN_OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _call(L.attn_fwd_splitkv_noalloc, qd, kd, vd, o, lse, True, None, 2) == _lib.ATTN_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert L.attn_read_device_status(torch.cuda.current_stream().cuda_stream) == _lib.ATTN_OK
