"""Pins for the fp64 oracle: checks against facts that do not come from the oracle.

Each pin takes an oracle handle (``oracle.Oracle``) and raises AssertionError on
a mismatch. They are run against the real oracle (test_oracle_pins.py) and
against deliberately broken copies of it (test_oracle_mutants.py), which shows
that a plausible mistake anywhere in the oracle fails at least one pin.

What pins what:
  worked examples printed on the pages (tests/golden/)   -> dot product, softmax values
  numpy's own binary16 -> float64 conversion             -> the fp16 decoder
  numpy's float32 bit view (bfloat16 = upper half)        -> the bf16 decoder
  values exact in both formats (fp16 vs bf16 result)      -> bf16 routing
  fp16 values as fp32; scipy on full fp32 inputs          -> fp32 inputs
  scipy.special.softmax / logsumexp on tiny inputs       -> scores, masks, softmax, PV, lse
  P1's two-block online-softmax merge                     -> normalisation and lse
  closed forms (uniform keys, one-hot selection, causal
  row 0, N = 1, d = 1 / N = 2 logistic weight)           -> masks, index order, scale
  invariances (joint permutation, score shift)            -> operand roles, lse offset
  reductions to the self-attention case (repeated K/V
  heads, padded Q or K/V, shifted query rows)              -> head groups, Nq != Nk, causal
                                                              diagonal of cross-attention
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _h(x):
    return np.asarray(x, dtype=np.float16)


def _rand(shape, seed, sigma=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal(shape) * sigma).astype(np.float16)


def _allowed(N, causal, L):
    """Boolean [N, N] allowed-set matrix: key j allowed for query i."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    a = np.broadcast_to(j < L, (N, N))
    if causal:
        a = a & (j <= i)
    return a


def pin_half_decoder(orc):
    """Every binary16 bit pattern decodes as numpy's float16 -> float64 conversion does."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_dot_product_golden(orc):
    """Page example q.k = 32: with one key the score is the logsumexp and O = V."""
    g = _read_golden("dot_product.txt")
    q = _h(g["q"]).reshape(1, 1, 1, 3)
    k = _h(g["k"]).reshape(1, 1, 1, 3)
    v = _h([0.5, -1.0, 2.0]).reshape(1, 1, 1, 3)
    o, lse = orc.attn(q, k, v, sm_scale=1.0)
    assert lse[0, 0, 0] == g["dot"][0]
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0].astype(np.float64))


def pin_softmax_golden(orc):
    """Page example softmax([2, 1, 0]) = [0.665, 0.245, 0.090] to three decimals."""
    g = _read_golden("softmax_2_1_0.txt")
    x = g["x"]
    n = len(x)
    q = np.zeros((1, 1, n, n), np.float16)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, n, n), np.float16)
    k[0, 0, :, 0] = x  # score of key j = x_j
    v = np.eye(n, dtype=np.float16).reshape(1, 1, n, n)  # O row = P row
    o, lse = orc.attn(q, k, v, sm_scale=1.0)
    dec = int(g["decimals"][0])
    for i in range(n):
        assert np.array_equal(np.round(o[0, 0, i], dec), np.array(g["p"])), o[0, 0, i]
        assert abs(o[0, 0, i].sum() - 1.0) < 1e-12


def pin_rows_sum_to_one(orc):
    """Rows of P sum to 1: with V = 1 every non-empty row of O is exactly 1 (to rounding)."""
    B, H, N, d = 2, 3, 19, 8
    q = _rand((B, H, N, d), 11, 2.0)
    k = _rand((B, H, N, d), 12, 2.0)
    v = np.ones((B, H, N, d), np.float16)
    for causal in (False, True):
        kl = np.array([19, 7], np.int32)
        o, _ = orc.attn(q, k, v, sm_scale=0.3, causal=causal, key_lengths=kl)
        assert np.max(np.abs(o - 1.0)) < 1e-12


def _scipy_reference(q, k, v, sm_scale, causal, key_lengths):
    from scipy.special import logsumexp, softmax

    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        L = N if key_lengths is None else int(np.clip(key_lengths[b], 0, N))
        allow = _allowed(N, causal, L)
        for h in range(H):
            s = sm_scale * (q64[b, h] @ k64[b, h].T)
            s = np.where(allow, s, -np.inf)
            for i in range(N):
                if not allow[i].any():
                    continue
                p = softmax(s[i])
                o[b, h, i] = p @ v64[b, h]
                lse[b, h, i] = logsumexp(s[i])
    return o, lse


def pin_scipy_tiny(orc):
    """Against scipy.special.softmax / logsumexp over explicitly masked score rows."""
    B, H, N, d = 3, 2, 11, 5
    q = _rand((B, H, N, d), 21)
    k = _rand((B, H, N, d), 22)
    v = _rand((B, H, N, d), 23)
    for causal in (False, True):
        for kl in (None, np.array([0, 6, 40], np.int32), np.array([11, 1, -3], np.int32)):
            o, lse = orc.attn(q, k, v, sm_scale=0.37, causal=causal, key_lengths=kl)
            ro, rl = _scipy_reference(q, k, v, 0.37, causal, kl)
            assert np.max(np.abs(o - ro)) < 1e-12
            fin = np.isfinite(rl)
            assert np.array_equal(np.isfinite(lse), fin)
            assert np.all(lse[~fin] == -np.inf)
            assert np.max(np.abs(lse[fin] - rl[fin])) < 1e-12


def pin_merge_identity(orc):
    """Self-Attention Kernel & Inference Engine from Scratch, "Online Softmax Formulation":
    merging the results of two key blocks with m = max(m1, m2),
    l = e^(m1-m) l1 + e^(m2-m) l2 and O = (e^(m1-m) l1 O1 + e^(m2-m) l2 O2) / l gives
    the two-pass result over the union, for every split point."""
    N, d = 13, 6
    q = _rand((1, 1, N, d), 31, 1.5)
    k = _rand((1, 1, N, d), 32, 1.5)
    v = _rand((1, 1, N, d), 33)
    scale = 0.8
    o_all, lse_all = orc.attn(q, k, v, sm_scale=scale)
    for t in range(1, N):
        # block 1 = keys [0, t): key padding at t. block 2 = keys [t, N): the tail rows of K, V.
        o1, lse1 = orc.attn(q, k, v, sm_scale=scale, key_lengths=np.array([t], np.int32))
        q2 = q
        k2 = np.zeros_like(k)
        v2 = np.zeros_like(v)
        k2[0, 0, : N - t] = k[0, 0, t:]
        v2[0, 0, : N - t] = v[0, 0, t:]
        o2, lse2 = orc.attn(q2, k2, v2, sm_scale=scale, key_lengths=np.array([N - t], np.int32))
        for i in range(N):
            # with m_b the block max and l_b its normaliser, lse_b = m_b + ln l_b; take m_b from
            # an independent max over the block's scores so m and l enter separately.
            s = scale * (q[0, 0, i].astype(np.float64) @ k[0, 0].astype(np.float64).T)
            m1, m2 = s[:t].max(), s[t:].max()
            l1 = math.exp(lse1[0, 0, i] - m1)
            l2 = math.exp(lse2[0, 0, i] - m2)
            m = max(m1, m2)
            l = math.exp(m1 - m) * l1 + math.exp(m2 - m) * l2
            o = (math.exp(m1 - m) * l1 / l) * o1[0, 0, i] + (math.exp(m2 - m) * l2 / l) * o2[0, 0, i]
            assert np.max(np.abs(o - o_all[0, 0, i])) < 1e-12
            assert abs((m + math.log(l)) - lse_all[0, 0, i]) < 1e-12


def pin_uniform_keys(orc):
    """All key rows equal: every allowed score ties, so O_i is the mean of V over the allowed
    set and lse_i = scale * q_i.k + ln|A_i| (prefix means under causal, first L_b rows under
    padding)."""
    B, H, N, d = 2, 2, 17, 4
    q = _rand((B, H, N, d), 41)
    k = np.broadcast_to(_rand((B, H, 1, d), 42), (B, H, N, d)).copy()
    v = _rand((B, H, N, d), 43)
    kl = np.array([17, 9], np.int32)
    scale = 0.5
    for causal in (False, True):
        o, lse = orc.attn(q, k, v, sm_scale=scale, causal=causal, key_lengths=kl)
        for b in range(B):
            for h in range(H):
                for i in range(N):
                    n_allowed = min(kl[b], i + 1) if causal else kl[b]
                    mean = v[b, h, :n_allowed].astype(np.float64).mean(axis=0)
                    assert np.max(np.abs(o[b, h, i] - mean)) < 1e-12
                    s = scale * float(q[b, h, i].astype(np.float64) @ k[b, h, 0].astype(np.float64))
                    assert abs(lse[b, h, i] - (s + math.log(n_allowed))) < 1e-12


def pin_one_hot_selection(orc):
    """K_j = e_j and Q_i = 20 e_pi(i) with scale 1: the target score is 20, all others 0, so
    O_i = V_pi(i) up to (N-1) e^-20 of the other rows. Under causal pi(i) <= i."""
    N = d = 32
    rng = np.random.Generator(np.random.PCG64(51))
    k = np.eye(N, d, dtype=np.float16).reshape(1, 1, N, d)
    v = _rand((1, 1, N, d), 52)
    for causal in (False, True):
        if causal:
            pi = np.array([rng.integers(0, i + 1) for i in range(N)])
        else:
            pi = rng.permutation(N)
        q = np.zeros((1, 1, N, d), np.float16)
        q[0, 0, np.arange(N), pi] = 20.0
        o, _ = orc.attn(q, k, v, sm_scale=1.0, causal=causal)
        tol = (N - 1) * math.exp(-20) * 8.0
        assert np.max(np.abs(o[0, 0] - v[0, 0, pi].astype(np.float64))) < tol


def pin_causal_row0(orc):
    """Causal: query 0 sees key 0 only, so O_0 = V_0 and lse_0 = scale * q_0.k_0."""
    B, H, N, d = 2, 3, 9, 8
    q, k, v = _rand((B, H, N, d), 61), _rand((B, H, N, d), 62), _rand((B, H, N, d), 63)
    o, lse = orc.attn(q, k, v, sm_scale=0.25, causal=True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].astype(np.float64))
    s0 = 0.25 * np.einsum("bhc,bhc->bh", q[:, :, 0].astype(np.float64), k[:, :, 0].astype(np.float64))
    assert np.max(np.abs(lse[:, :, 0] - s0)) < 1e-12


def pin_single_key(orc):
    """N = 1: the softmax over one key is 1, O = V, lse = the score."""
    q, k, v = _rand((2, 2, 1, 8), 71), _rand((2, 2, 1, 8), 72), _rand((2, 2, 1, 8), 73)
    o, lse = orc.attn(q, k, v, sm_scale=0.7)
    assert np.array_equal(o, v.astype(np.float64))
    s = 0.7 * np.einsum("bhnc,bhnc->bhn", q.astype(np.float64), k.astype(np.float64))
    assert np.max(np.abs(lse - s)) < 1e-12


def pin_two_keys_logistic(orc):
    """d = 1, N = 2: the weight on key 0 is the logistic function of s_0 - s_1."""
    q = _h([1.5, -2.0]).reshape(1, 1, 2, 1)
    k = _h([0.75, 2.5]).reshape(1, 1, 2, 1)
    v = _h([3.0, -1.0]).reshape(1, 1, 2, 1)
    scale = 0.9
    o, lse = orc.attn(q, k, v, sm_scale=scale)
    for i in range(2):
        s0, s1 = scale * float(q[0, 0, i, 0]) * float(k[0, 0, 0, 0]), scale * float(q[0, 0, i, 0]) * float(k[0, 0, 1, 0])
        w0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        assert abs(o[0, 0, i, 0] - (w0 * 3.0 + (1 - w0) * -1.0)) < 1e-12
        assert abs(lse[0, 0, i] - math.log(math.exp(s0) + math.exp(s1))) < 1e-12


def pin_permutation_invariance(orc):
    """Without a causal mask, permuting the K and V rows jointly leaves O and lse unchanged;
    permuting V alone changes O (the operands are not interchangeable)."""
    B, H, N, d = 1, 2, 15, 6
    q, k, v = _rand((B, H, N, d), 81), _rand((B, H, N, d), 82), _rand((B, H, N, d), 83)
    perm = np.random.Generator(np.random.PCG64(84)).permutation(N)
    o, lse = orc.attn(q, k, v, sm_scale=0.6)
    o2, lse2 = orc.attn(q, k[:, :, perm], v[:, :, perm], sm_scale=0.6)
    assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(lse - lse2)) < 1e-12
    o3, _ = orc.attn(q, k, v[:, :, perm], sm_scale=0.6)
    assert np.max(np.abs(o - o3)) > 1e-3


def pin_shift_invariance(orc):
    """"Tensor Parallelism with CUDA - Standard Attention", section "Step 2: Softmax": adding a
    constant to a score row leaves P unchanged. An extra coordinate with q = c/scale and k = 1
    adds c to every score of the row: O is unchanged and lse grows by c exactly."""
    B, H, N, d = 1, 2, 12, 7
    q, k, v = _rand((B, H, N, d), 91), _rand((B, H, N, d), 92), _rand((B, H, N, d), 93)
    scale = 0.5
    c = 3.0
    q2 = np.concatenate([q, np.full((B, H, N, 1), c / scale, np.float16)], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, N, 1), np.float16)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1), np.float16)], axis=-1)
    for causal in (False, True):
        o, lse = orc.attn(q, k, v, sm_scale=scale, causal=causal)
        o2, lse2 = orc.attn(q2, k2, v2, sm_scale=scale, causal=causal)
        assert np.max(np.abs(o2[..., :d] - o)) < 1e-12
        assert np.max(np.abs(lse2 - (lse + c))) < 1e-12


def pin_row_sampling(orc):
    """Computing a sorted subset of rows gives exactly those rows of the full output."""
    B, H, N, d = 2, 2, 21, 8
    q, k, v = _rand((B, H, N, d), 101), _rand((B, H, N, d), 102), _rand((B, H, N, d), 103)
    kl = np.array([21, 5], np.int32)
    o, lse = orc.attn(q, k, v, sm_scale=0.4, causal=True, key_lengths=kl)
    rows = np.array([0, 3, 20, 21, 40, 41, 62, 83])
    o_r, lse_r = orc.attn(q, k, v, sm_scale=0.4, causal=True, key_lengths=kl, rows=rows)
    assert np.array_equal(o_r, o.reshape(-1, d)[rows])
    assert np.array_equal(lse_r, lse.reshape(-1)[rows])


def pin_gqa_is_repeated_kv(orc):
    """Grouped-query attention ("natural extensions" of the cuda-reranker README): query head h
    reads key/value head h // (H // Hkv), so the result equals multi-head attention with each
    K, V head repeated for its group of consecutive query heads."""
    B, H, N, d = 2, 6, 13, 8
    q = _rand((B, H, N, d), 111)
    for Hkv in (1, 2, 3):
        k, v = _rand((B, Hkv, N, d), 112 + Hkv), _rand((B, Hkv, N, d), 122 + Hkv)
        kr, vr = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
        for causal in (False, True):
            kl = np.array([13, 6], np.int32)
            o, lse = orc.attn(q, k, v, sm_scale=0.45, causal=causal, key_lengths=kl)
            ro, rl = orc.attn(q, kr, vr, sm_scale=0.45, causal=causal, key_lengths=kl)
            assert np.array_equal(o, ro) and np.array_equal(lse, rl)
    # a mapping by h % Hkv instead would differ: check the groups are not interleaved
    k, v = _rand((B, 2, N, d), 131), _rand((B, 2, N, d), 132)
    o, _ = orc.attn(q, k, v, sm_scale=0.45)
    oi, _ = orc.attn(q, np.tile(k, (1, 3, 1, 1)), np.tile(v, (1, 3, 1, 1)), sm_scale=0.45)
    assert np.max(np.abs(o - oi)) > 1e-3


def pin_cross_is_padded_self(orc):
    """Cross-attention (Nq != Nk) without a causal mask: every query row sees the same keys as in
    self-attention, so the rows equal those of a self-attention problem whose Q is padded with
    extra rows (Nq < Nk) or whose K, V are padded with rows excluded by key padding (Nq > Nk)."""
    B, H, d = 2, 2, 8
    for Nq, Nk in ((5, 19), (19, 5), (1, 33)):
        q = _rand((B, H, Nq, d), 140 + Nq)
        k, v = _rand((B, H, Nk, d), 150 + Nk), _rand((B, H, Nk, d), 160 + Nk)
        N = max(Nq, Nk)
        qp = np.concatenate([q, _rand((B, H, N - Nq, d), 170)], axis=2)
        kp = np.concatenate([k, _rand((B, H, N - Nk, d), 171)], axis=2)
        vp = np.concatenate([v, _rand((B, H, N - Nk, d), 172)], axis=2)
        for kl in (None, np.array([Nk, max(1, Nk // 2)], np.int32)):
            o, lse = orc.attn(q, k, v, sm_scale=0.55, key_lengths=kl)
            klp = np.full(B, Nk, np.int32) if kl is None else kl
            ro, rl = orc.attn(qp, kp, vp, sm_scale=0.55, key_lengths=klp)
            assert np.array_equal(o, ro[:, :, :Nq]) and np.array_equal(lse, rl[:, :, :Nq])


def pin_cross_causal_alignment(orc):
    """Causal cross-attention with the diagonal at the last rows: query i sees keys
    j <= i + Nk - Nq. For Nq < Nk the rows are the last Nq rows of self-attention over Nk keys
    (the real queries placed at positions Nk - Nq ..). For Nq > Nk the first Nq - Nk rows see no
    key (O = 0, lse = -inf) and the rest are self-attention of the last Nk queries."""
    B, H, d = 2, 2, 8
    for Nq, Nk in ((6, 21), (21, 6), (1, 17), (9, 9)):
        q = _rand((B, H, Nq, d), 180 + Nq)
        k, v = _rand((B, H, Nk, d), 190 + Nk), _rand((B, H, Nk, d), 200 + Nk)
        kl = np.array([Nk, max(1, Nk - 4)], np.int32)
        o, lse = orc.attn(q, k, v, sm_scale=0.6, causal=True, key_lengths=kl)
        if Nq <= Nk:
            qp = np.concatenate([_rand((B, H, Nk - Nq, d), 210), q], axis=2)
            ro, rl = orc.attn(qp, k, v, sm_scale=0.6, causal=True, key_lengths=kl)
            assert np.array_equal(o, ro[:, :, Nk - Nq:]) and np.array_equal(lse, rl[:, :, Nk - Nq:])
        else:
            e = Nq - Nk
            assert np.all(o[:, :, :e] == 0.0) and np.all(lse[:, :, :e] == -np.inf)
            ro, rl = orc.attn(q[:, :, e:], k, v, sm_scale=0.6, causal=True, key_lengths=kl)
            assert np.array_equal(o[:, :, e:], ro) and np.array_equal(lse[:, :, e:], rl)


def pin_cross_gqa_uniform_keys(orc):
    """All key rows equal, cross-attention with groups: O_i is the mean of V over the first
    n_i = min(L_b, i + Nk - Nq + 1) keys of the group's key/value head (the first L_b
    keys without the causal mask), and lse_i = scale * q_i.k + ln n_i; n_i = 0 gives O = 0,
    lse = -inf."""
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 11, 7, 4
    q = _rand((B, H, Nq, d), 221)
    k = np.broadcast_to(_rand((B, Hkv, 1, d), 222), (B, Hkv, Nk, d)).copy()
    v = _rand((B, Hkv, Nk, d), 223)
    kl = np.array([7, 3], np.int32)
    scale = 0.5
    for causal in (False, True):
        o, lse = orc.attn(q, k, v, sm_scale=scale, causal=causal, key_lengths=kl)
        for b in range(B):
            for h in range(H):
                g = h // (H // Hkv)
                for i in range(Nq):
                    n = min(kl[b], i + Nk - Nq + 1) if causal else kl[b]
                    n = max(n, 0)
                    if n == 0:
                        assert np.all(o[b, h, i] == 0.0) and lse[b, h, i] == -np.inf
                        continue
                    mean = v[b, g, :n].astype(np.float64).mean(axis=0)
                    assert np.max(np.abs(o[b, h, i] - mean)) < 1e-12
                    s = scale * float(q[b, h, i].astype(np.float64) @ k[b, g, 0].astype(np.float64))
                    assert abs(lse[b, h, i] - (s + math.log(n))) < 1e-12


def pin_bf16_decoder(orc):
    """bfloat16 is the upper half of an IEEE binary32: every bit pattern b decodes as numpy's
    float32 with bits b << 16 (converted to float64)."""
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_bf16_agrees_with_f16_on_common_values(orc):
    """Inputs whose values are exact in both formats (multiples of 1/16 up to 4 in magnitude,
    and powers of two from 2^-10 to 2^3) decode to the same doubles, so the bf16 and fp16
    results are the same bits; a wrong decode table or format routing breaks this."""
    rng = np.random.Generator(np.random.PCG64(231))
    vals = np.concatenate([np.arange(-64, 65) / 16.0, 2.0 ** np.arange(-10, 4),
                           -(2.0 ** np.arange(-10, 4))])
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 9, 13, 8
    q64, k64, v64 = (rng.choice(vals, size=sh) for sh in
                     ((B, H, Nq, d), (B, Hkv, Nk, d), (B, Hkv, Nk, d)))

    def as_bf16(x):
        return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    for causal in (False, True):
        kl = np.array([13, 5], np.int32)
        o16, l16 = orc.attn(q64.astype(np.float16), k64.astype(np.float16), v64.astype(np.float16),
                            sm_scale=0.3, causal=causal, key_lengths=kl)
        ob, lb = orc.attn(as_bf16(q64), as_bf16(k64), as_bf16(v64), sm_scale=0.3, causal=causal,
                          key_lengths=kl, dtype="bf16")
        assert np.array_equal(o16, ob) and np.array_equal(l16, lb)
    # values outside fp16's range are finite in bf16: 2^20 * 2^-20 products give score 1 per term
    big = np.full((1, 1, 2, 1), 2.0 ** 20)
    small = np.full((1, 1, 2, 1), 2.0 ** -20)
    o, lse = orc.attn(as_bf16(big), as_bf16(small), as_bf16(np.array([1.0, 3.0]).reshape(1, 1, 2, 1)),
                      sm_scale=1.0, dtype="bf16")
    assert np.allclose(o, 2.0, atol=1e-12, rtol=0) and np.allclose(lse, 1.0 + math.log(2.0))


def pin_f32_inputs(orc):
    """fp32 inputs: fp16 values (exact in fp32) give the fp16 result's bits; full-precision fp32
    values match scipy's softmax / logsumexp over the float64 conversion of the same inputs."""
    B, H, N, d = 2, 2, 11, 6
    q, k, v = _rand((B, H, N, d), 241), _rand((B, H, N, d), 242), _rand((B, H, N, d), 243)
    kl = np.array([11, 4], np.int32)
    for causal in (False, True):
        o16, l16 = orc.attn(q, k, v, sm_scale=0.4, causal=causal, key_lengths=kl)
        o32, l32 = orc.attn(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                            sm_scale=0.4, causal=causal, key_lengths=kl, dtype="f32")
        assert np.array_equal(o16, o32) and np.array_equal(l16, l32)
    rng = np.random.Generator(np.random.PCG64(244))
    qf, kf, vf = (rng.standard_normal((B, H, N, d)).astype(np.float32) for _ in range(3))
    for causal in (False, True):
        o, lse = orc.attn(qf, kf, vf, sm_scale=0.4, causal=causal, key_lengths=kl, dtype="f32")
        ro, rl = _scipy_reference(qf, kf, vf, 0.4, causal, kl)
        assert np.max(np.abs(o - ro)) < 1e-12
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.max(np.abs(lse[fin] - rl[fin])) < 1e-12


ALL_PINS = [
    pin_half_decoder,
    pin_dot_product_golden,
    pin_softmax_golden,
    pin_rows_sum_to_one,
    pin_scipy_tiny,
    pin_merge_identity,
    pin_uniform_keys,
    pin_one_hot_selection,
    pin_causal_row0,
    pin_single_key,
    pin_two_keys_logistic,
    pin_permutation_invariance,
    pin_shift_invariance,
    pin_row_sampling,
    pin_gqa_is_repeated_kv,
    pin_cross_is_padded_self,
    pin_cross_causal_alignment,
    pin_cross_gqa_uniform_keys,
    pin_bf16_decoder,
    pin_bf16_agrees_with_f16_on_common_values,
    pin_f32_inputs,
]
