"""The split-KV forward that allocates nothing (attn_fwd_splitkv_noalloc), through the C ABI.

Some callers cannot allocate device memory where they call the attention: their device memory
already belongs to their own pool or caching allocator, the runtime that hosts them gives them
no allocator, or their request loop cannot afford the synchronisation of cudaMalloc/cudaFree.
This entry point serves them from a fixed scratch array inside the library, so its results must
be those of the allocating entry points. Two calls in a row on different problems (the second
must not be affected by what the first left in the shared array) are each compared with
attn_fwd_lse on the same inputs, within the parity tolerances of the other GPU tests.

The file name makes pytest collect it last, so a run that stops at the first failure has run
every other test before it; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

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


def test_noalloc_matches_allocating_entry_point_twice():
    build.build()
    L = _lib.lib()
    cases = [
        # B, H, N, d, causal, key_lengths, n_splits
        (1, 2, 2000, 128, True, None, 3),
        (2, 3, 700, 64, False, [700, 123], 2),
    ]
    for B, H, N, d, causal, kl, S in cases:
        assert L.attn_splitkv_workspace_bytes(B, H, N, d, S) <= L.attn_noalloc_scratch_bytes()
        q, k, v, _ = synth.draw(B, H, N, d, seed=500 + N)
        qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
        kld = torch.from_numpy(np.array(kl, np.int32)).cuda() if kl is not None else None
        o1 = torch.full_like(qd, float("nan"))
        o2 = torch.full_like(qd, float("nan"))
        l1 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        l2 = torch.full_like(l1, float("nan"))
        assert _call(L.attn_fwd_splitkv_noalloc, qd, kd, vd, o1, l1, causal, kld, S) == _lib.ATTN_OK
        assert _call(L.attn_fwd_lse, qd, kd, vd, o2, l2, causal, kld) == _lib.ATTN_OK
        assert L.attn_read_device_status(torch.cuda.current_stream().cuda_stream) == _lib.ATTN_OK
        torch.cuda.synchronize()
        a, b = o1.double().cpu().numpy(), o2.double().cpu().numpy()
        assert not np.isnan(a).any()
        assert np.max(np.abs(a - b)) <= TOL_MAX_ABS
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL_REL_L2
        la, lb = l1.double().cpu().numpy(), l2.double().cpu().numpy()
        assert np.array_equal(np.isfinite(la), np.isfinite(lb))
        fin = np.isfinite(lb)
        assert np.max(np.abs(la[fin] - lb[fin])) <= TOL_LSE
