"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and compare
with the fp64 oracle element by element.

Tolerances (fp16 inputs and output, fp16 probabilities, fp32 accumulation):
  max |O_gpu - O_ref|           <= 1e-2
  ||O_gpu - O_ref||_2 / ||O_ref||_2 <= 2e-3
  max |lse_gpu - lse_ref|       <= 1e-3   (finite rows; empty rows must be -inf on both sides)
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_scaled_dot_attn_gb300 import _lib, api, build

TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 2e-3
TOL_LSE = 1e-3

# bf16 (8 significant bits, unit roundoff u = 2^-8): O is rounded to bf16 (error <= u |O|) and so
# is P before the PV product (error <= u sum_j P_j |v_j| <= u max|v|); the normaliser l sums the
# unrounded fp32 probabilities and the scores are exact products of bf16 values accumulated in
# fp32, so lse keeps the fp16 bound. Per element: |dO| <= u (|O_ref| + max|V|) + 1e-3 (fp32 and
# exp2 noise); over the tensor: relative L2 error <= 2u.
BF16_U = 2.0 ** -8
TOL_REL_L2_BF16 = 2 * BF16_U


def bf16_atol(o_ref, v_bits):
    """Per-element bound on |O_gpu - O_ref| for bf16 (see above); v_bits: uint16 bf16 V."""
    vmax = float(np.max(np.abs(bf16_to_float(v_bits)))) if v_bits.size else 0.0
    return BF16_U * (np.abs(o_ref) + vmax) + 1e-3


# fp32 inputs on the tensor cores (TF32): each operand of both products, P included, is read
# with 10 fraction bits, assumed truncated (relative error < u_t = 2^-10). Scores then move by at
# most D_i = 2.001 u_t sm_scale max_j sum_c |q_ic||k_jc| (both operands), so the softmax weights
# move by a factor within exp(+-2 D_i) and sum_j |dP_ij| <= exp(2 D_i) - 1; truncating P and V
# adds <= 2 u_t sum_j P_ij |v_jc|. Per element |dO_ic| <= (exp(2 D_i) - 1 + 2 u_t) max_j |v_jc|
# + 1e-5 (fp32 accumulation, exp2); |dlse_i| <= D_i + 1e-4. For inputs exact in TF32 (at most
# 10 fraction bits) D_i = 0 and the V term vanishes: |dO_ic| <= u_t max_j |v_jc| + 1e-5. The
# relative L2 bound is the norm of the per-element bounds over the norm of O_ref.
TF32_U = 2.0 ** -10


def tf32_bounds(q, k, v, sm_scale, *, exact_inputs):
    """(atol [B,H,N,d], lse_tol [B,H,N]) for fp32 inputs on the TF32 path (see above)."""
    q64, k64, v64 = (np.abs(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    B, H, N, d = q64.shape
    g = H // k64.shape[1]
    kr = np.repeat(k64, g, axis=1)
    vmax = np.repeat(v64.max(axis=2, keepdims=True), g, axis=1)  # [B,H,1,d]
    if exact_inputs:
        delta = np.zeros((B, H, N))
        per = TF32_U
    else:
        delta = 2.001 * TF32_U * abs(sm_scale) * np.einsum("bhid,bhjd->bhij", q64, kr).max(axis=3)
        per = 2 * TF32_U
    atol = (np.expm1(2 * delta)[..., None] + per) * vmax + 1e-5
    return atol, delta + 1e-4


# fp32 inputs at fp32 accuracy (split-TF32 products, the automatic path for fp32): each operand x
# of both products, P included, is split into hi = x rounded to 10 fraction bits
# (|x - hi| <= 2^-11 |x|) and lo = x - hi, of which the tensor core reads 10 fraction bits
# (error <= 2^-10 |lo| <= 2^-21 |x|, truncation assumed); a product is hi*hi + hi*lo + lo*hi,
# within (2^-21 + 2^-21 + 2^-22) |a b| = SPLIT_U = 5 * 2^-22 of |a b|. Sums are fp32; the tensor
# core may truncate, so the unit roundoff is taken as ACC_U = 2^-23 and a sum of n terms errs by
# at most n ACC_U of the sum of their magnitudes (the linear worst case). Per row i, with S_i = max_j sum_c |q_ic||k_jc|:
#   scores      |ds_ij| <= D_i = |sm_scale| (SPLIT_U + 3 d ACC_U) S_i   (3 d products per score)
#   exponential relative error <= E_i = 2^-21 + 2^-22 |sm_scale| log2(e) S_i (ex2.approx and the
#               fp32 rounding of its scaled argument)
#   weights     P_ij / l_i move by a factor within exp(+-(2 D_i + 2 E_i))
#   P V         sum_j P_ij v_jc within (SPLIT_U + 3 N_k ACC_U) l_i max_j |v_jc|
# so |dO_ic| <= (expm1(2 D_i + 2 E_i) + SPLIT_U + 3 N_k ACC_U) max_j |v_jc| + 1e-7 and
# |dlse_i| <= D_i + 2 E_i + N_k ACC_U + 1e-6. These are worst cases. Independent rounding
# errors add in quadrature: for scores of a few units (|sm_scale q.k| <~ 10, the normal-scale
# test inputs and workloads), score errors are ~1e-6 and so are the relative errors of P and O.
# On such inputs the relative L2 error over a tensor is checked against F32_REL_L2 = 3e-5:
# thirty times above that estimate and thirty times below TF32's unit roundoff 2^-10, so a
# result with TF32 products fails it. (With scores in the hundreds, fp32 itself moves the
# weights by ~1e-4; those cases are checked against the norm of the per-element bounds.)
SPLIT_U = 5 * 2.0 ** -22
ACC_U = 2.0 ** -23
F32_REL_L2 = 3e-5


def f32_split_bounds(q, k, v, sm_scale):
    """(atol [B,H,N,d], lse_tol [B,H,N]) for fp32 inputs on the split-TF32 path (see above)."""
    q64, k64, v64 = (np.abs(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    B, H, N, d = q64.shape
    n_keys = k64.shape[2]
    g = H // k64.shape[1]
    kr = np.repeat(k64, g, axis=1)
    vmax = np.repeat(v64.max(axis=2, keepdims=True), g, axis=1)  # [B,H,1,d]
    s_abs = np.einsum("bhid,bhjd->bhij", q64, kr).max(axis=3) if n_keys else np.zeros((B, H, N))
    delta = abs(sm_scale) * (SPLIT_U + 3 * d * ACC_U) * s_abs
    eps_e = 2.0 ** -21 + 2.0 ** -22 * abs(sm_scale) * 1.4426950408889634 * s_abs
    atol = (np.expm1(2 * delta + 2 * eps_e)[..., None] + SPLIT_U + 3 * n_keys * ACC_U) * vmax + 1e-7
    return atol, delta + 2 * eps_e + n_keys * ACC_U + 1e-6


def bf16_to_float(bits):
    """uint16 bfloat16 bit patterns -> float64 (bfloat16 is the upper half of a binary32)."""
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        _built = True


def to_dev(x, dtype="f16"):
    """numpy -> CUDA tensor; dtype "bf16" reads uint16 bit patterns as torch.bfloat16, "f32"
    takes float32 arrays."""
    if x is None:
        return None
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(q, k, v, *, causal, key_lengths=None, sm_scale=None, path="auto", guard=True,
            dtype="f16"):
    """Runs the C-ABI forward on device copies of the numpy inputs.

    O and lse are allocated inside larger buffers whose margins hold a sentinel, and the
    interior is pre-filled with NaN, so writes out of bounds and rows left unwritten both
    show up. Returns numpy (o, lse) as float64.
    """
    ensure_built()
    B, H, N, d = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    kld = to_dev(key_lengths)
    pad_o = 4096  # 16-bit elements of guard on each side (8 KiB: keeps 16-byte alignment)
    pad_l = 1024
    n_o = q.size
    n_l = B * H * N
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}.get(dtype, torch.float16)
    o_buf = torch.full((n_o + 2 * pad_o,), float("nan"), dtype=tdt, device="cuda")
    l_buf = torch.full((n_l + 2 * pad_l,), float("nan"), dtype=torch.float32, device="cuda")
    o_buf[:pad_o] = 1234.0
    o_buf[pad_o + n_o:] = 1234.0
    l_buf[:pad_l] = 4321.0
    l_buf[pad_l + n_l:] = 4321.0
    o = o_buf[pad_o:pad_o + n_o].view(B, H, N, d)
    lse = l_buf[pad_l:pad_l + n_l].view(B, H, N)
    api.fwd(qd, kd, vd, causal=causal, sm_scale=sm_scale, key_lengths=kld, return_lse=True,
            out=o, lse_out=lse, path=path)
    st = api.read_device_status()
    assert st == _lib.ATTN_OK, f"device status {st}"
    torch.cuda.synchronize()
    if guard:
        assert torch.all(o_buf[:pad_o] == 1234.0) and torch.all(o_buf[pad_o + n_o:] == 1234.0), \
            "O guard region overwritten"
        assert torch.all(l_buf[:pad_l] == 4321.0) and torch.all(l_buf[pad_l + n_l:] == 4321.0), \
            "lse guard region overwritten"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, *, row_mask=None, check_lse=True, what="",
            atol=TOL_MAX_ABS, rel_l2=TOL_REL_L2, lse_tol=TOL_LSE):
    """Element-wise comparison; row_mask (bool, per row) selects the rows that count. atol is a
    scalar or an array of o_ref's shape (per-element bound)."""
    o_gpu = o_gpu.reshape(-1, o_gpu.shape[-1])
    o_ref = o_ref.reshape(-1, o_ref.shape[-1])
    atol = np.asarray(atol, dtype=np.float64).reshape(o_ref.shape) if np.ndim(atol) \
        else np.full(o_ref.shape, float(atol))
    lse_gpu = lse_gpu.reshape(-1)
    lse_ref = lse_ref.reshape(-1)
    lse_tol = np.asarray(lse_tol, dtype=np.float64).reshape(-1) if np.ndim(lse_tol) \
        else np.full(lse_ref.shape, float(lse_tol))
    if row_mask is not None:
        row_mask = np.asarray(row_mask).reshape(-1)
        o_gpu, o_ref, atol = o_gpu[row_mask], o_ref[row_mask], atol[row_mask]
        lse_gpu, lse_ref, lse_tol = lse_gpu[row_mask], lse_ref[row_mask], lse_tol[row_mask]
    assert not np.isnan(o_gpu).any(), f"{what}: NaN in O (unwritten or invalid rows)"
    err = np.abs(o_gpu - o_ref)
    max_abs = float(err.max()) if err.size else 0.0
    ref_norm = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o_gpu - o_ref) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(o_gpu))
    if err.size:
        worst = int(np.argmax(err - atol))
        assert np.all(err <= atol), \
            f"{what}: |dO| = {err.flat[worst]:.3e} above its bound {atol.flat[worst]:.3e}"
    assert rel <= rel_l2, f"{what}: rel L2 = {rel:.3e}"
    lse_err = 0.0
    if check_lse:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: lse finiteness differs"
        assert np.all(lse_gpu[~fin] == -np.inf), f"{what}: empty rows must have lse = -inf"
        if fin.any():
            d_lse = np.abs(lse_gpu[fin] - lse_ref[fin])
            lse_err = float(d_lse.max())
            assert np.all(d_lse <= lse_tol[fin]), f"{what}: max |dlse| = {lse_err:.3e}"
    return dict(max_abs=max_abs, rel_l2=rel, lse_max_abs=lse_err)


def oracle_full(q, k, v, *, causal, key_lengths=None, sm_scale=None):
    d = q.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    return oracle.attn(q, k, v, sm_scale=sm_scale, causal=causal, key_lengths=key_lengths)


_WORKLOAD_CACHE: dict = {}


def workload_oracle(name):
    """(w, q, k, v, key_lengths, o_ref, lse_ref) of a named workload with the oracle's output
    for every row. Computed once per test session and kept for the last four workloads asked
    for (about 0.7 GB for the prefill and stress workloads together): the large ones take
    seconds of host time each and several test files compare different kernels with them."""
    from exact_scaled_dot_attn_gb300 import synth
    if name not in _WORKLOAD_CACHE:
        w = synth.WORKLOADS[name]
        q, k, v, kl = synth.draw_workload(w)
        o_ref, lse_ref = oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal,
                                     key_lengths=kl, dtype=w.dtype)
        while len(_WORKLOAD_CACHE) >= 4:
            _WORKLOAD_CACHE.pop(next(iter(_WORKLOAD_CACHE)))
        _WORKLOAD_CACHE[name] = (w, q, k, v, kl, o_ref, lse_ref)
    return _WORKLOAD_CACHE[name]


def sample_rows(B, H, N, seed, per_head=48, heads=None):
    """Deterministic sample of flat row ids: tile edges, ragged tail and random rows in each of
    the given flat (batch*head) heads, or by default in a few heads (first, last and random
    ones)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    BH = B * H
    if heads is None:
        heads = sorted({0, BH - 1, *rng.integers(0, BH, size=2).tolist()})
    rows = []
    fixed = [0, 1, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    for h in heads:
        picks = {i for i in fixed if 0 <= i < N}
        picks |= set(rng.integers(0, N, size=per_head).tolist())
        rows += [h * N + i for i in sorted(picks)]
    return np.array(sorted(rows), dtype=np.int64)
