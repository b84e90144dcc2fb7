"""The decoding kernel's decomposition of a head, restated in numpy (fp64) and checked against
the oracle on the CPU.

The kernel packs the G query heads of a group into G * N_q rows when H_kv < H and N_q < 128
(under the causal mask row r is query r % N_q), gives every row the key limit
min(clamp(key_lengths[b], 0, N_k), query + N_k - (query rows) + 1), and covers keys up to the
largest limit with 64-key tiles. CTA c of a C-CTA cluster takes tiles
[n_tiles * c / C, n_tiles * (c + 1) / C). Warp w of a CTA takes keys 16w .. 16w + 15 of each of
those tiles with its own running maximum m, sum l and output O (scores in log2 units, keys past a
row's limit excluded). The four warps are then merged, and the C CTAs after them, each step by
the two-block merge: M = max m_i, l = sum l_i 2^(m_i - M), O = sum O_i 2^(m_i - M). A row with no
allowed key gets O = 0 and lse = -inf.

If the decomposition or the merges lost or double-counted a key, shifted a limit or mishandled
an empty block, the result would leave the oracle's, which is computed directly.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_attn_gb300 import synth

KT, WARPS, KW = 64, 4, 16


def _pack(H, Hkv, Nq, causal):
    if Hkv < H and Nq < 128:
        return Hkv, (H // Hkv) * Nq, (Nq if (causal and Nq > 1) else 0), (causal and Nq > 1)
    return H, Nq, 0, causal


def _merge(parts, N, D):
    m = np.stack([p[0] for p in parts])
    M = m.max(axis=0)
    w = np.where(np.isfinite(m), np.exp2(m - np.where(np.isfinite(M), M, 0.0)), 0.0)
    l = (np.stack([p[1] for p in parts]) * w).sum(axis=0)
    o = (np.stack([p[2] for p in parts]) * w[:, :, None]).sum(axis=0)
    return M, l, o


def decode_plan(q, k, v, causal, key_lengths, C):
    B, H0, Nq0, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    H, N, qrows, causal = _pack(H0, Hkv, Nq0, causal)
    qp = q.reshape(B, H, N, D).astype(np.float64) * (D ** -0.5) / np.log(2.0)
    o = np.zeros((B, H, N, D))
    lse = np.zeros((B, H, N))
    for b in range(B):
        klen = Nk if key_lengths is None else min(max(int(key_lengths[b]), 0), Nk)
        for h in range(H):
            K = k[b, h // (H // Hkv)].astype(np.float64)
            V = v[b, h // (H // Hkv)].astype(np.float64)
            lim = np.full(N, klen)
            if causal:
                nq = qrows if qrows else N
                qi = np.arange(N) % qrows if qrows else np.arange(N)
                lim = np.minimum(lim, np.maximum(qi + Nk - nq + 1, 0))
            n_keys = int(lim.max())
            n_tiles = (n_keys + KT - 1) // KT
            ctas = []
            for c in range(C):
                warps = []
                for w in range(WARPS):
                    m, l, acc = np.full(N, -np.inf), np.zeros(N), np.zeros((N, D))
                    for t in range(n_tiles * c // C, n_tiles * (c + 1) // C):
                        keys = t * KT + w * KW + np.arange(KW)
                        inside = keys < n_keys
                        Kt = np.where(inside[:, None], K[np.minimum(keys, Nk - 1)], 0.0)
                        Vt = np.where(inside[:, None], V[np.minimum(keys, Nk - 1)], 0.0)
                        s = np.where(keys[None, :] < lim[:, None], qp[b, h] @ Kt.T, -np.inf)
                        mn = np.maximum(m, s.max(axis=1))
                        mu = np.where(np.isfinite(mn), mn, 0.0)
                        p = np.exp2(s - mu[:, None])
                        alpha = np.exp2(m - mu)
                        l = l * alpha + p.sum(axis=1)
                        acc = acc * alpha[:, None] + p @ Vt
                        m = mn
                    warps.append((m, l, acc))
                ctas.append(_merge(warps, N, D))
            M, L, O = _merge(ctas, N, D)
            empty = ~np.isfinite(M)
            o[b, h] = np.where(empty[:, None], 0.0, O / np.where(empty, 1.0, L)[:, None])
            lse[b, h] = np.where(empty, -np.inf, (np.where(empty, 0.0, M) + np.log2(np.where(empty, 1.0, L))) * np.log(2.0))
    return o.reshape(q.shape), lse.reshape(q.shape[:3])


CASES = [
    # B, H, H_kv, N_q, N_k, d, causal, key_lengths
    (2, 8, 2, 1, 1000, 64, True, [1000, 37]),
    (3, 12, 4, 5, 300, 32, False, [300, 1, 0]),
    (1, 8, 2, 4, 500, 32, True, None),
    (1, 4, 4, 3, 777, 32, True, None),
    (1, 2, 2, 5, 3, 32, True, None),
    (1, 1, 1, 1, 5000, 64, False, None),
    (1, 2, 2, 1, 20, 32, False, None),
]


@pytest.mark.parametrize("C", [1, 2, 4, 8])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}kv{c[2]}Nq{c[3]}Nk{c[4]}")
def test_decomposition_reproduces_the_oracle(case, C):
    B, H, Hkv, Nq, Nk, d, causal, kl = case
    q, k, v, _ = synth.draw_ex(B, H, Hkv, Nq, Nk, d, seed=9600 + Nk)
    kl = None if kl is None else np.array(kl, np.int32)
    o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=d ** -0.5, causal=causal, key_lengths=kl)
    o, lse = decode_plan(q, k, v, causal, kl, C)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(o[~fin] == 0.0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)
