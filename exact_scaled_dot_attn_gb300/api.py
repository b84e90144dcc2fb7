"""Python entry point over the C ABI: ``fwd(q, k, v, ...)``.

PyTorch supplies device memory and the current CUDA stream; every step of the
attention runs in the CUDA library. Host (CPU) tensors are accepted too: they
are copied to the current device, the same C entry point runs on them, and the
results are copied back (this is the end-to-end call a host-side user makes).
"""
from __future__ import annotations

import math

import torch

from . import _lib


def _check_device_tensor(name, t, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
        sm_scale: float | None = None, key_lengths: torch.Tensor | None = None,
        return_lse: bool = False, out: torch.Tensor | None = None,
        lse_out: torch.Tensor | None = None, path: str = "auto"):
    """O = softmax(sm_scale * Q K^T + mask) V for fp16, bf16 or fp32 tensors (q, k, v and out of
    one dtype; bf16 and fp32 run on the tcgen05 kernel, fp32 with d = 32 and TF32 products):
    q [B, H, N, d] and k, v of the same shape
    (self-attention) or [B, H_kv, N_k, d] (cross-attention and grouped-query attention: H a
    multiple of H_kv, query head h reads key/value head h // (H // H_kv)).

    causal: key j allowed for query i only when j <= i + N_k - N (j <= i for self-attention).
    key_lengths: int32 [B]; keys j >= key_lengths[b] are excluded.
    sm_scale: defaults to 1/sqrt(d).
    return_lse: also return the fp32 [B, H, N] logsumexp.
    path: "auto", "warp_mma", "tcgen05", "short" or "decode" (kernel choice; see
    include/attn.h; "short" takes N <= 256 with d in {32, 64}; "decode" at most 16 query rows
    per head, counting the query heads of a group together when H_kv < H).
    Device tensors run asynchronously on the current stream. CPU tensors are
    copied to the current CUDA device and back, and the call returns after the
    copy back has finished.
    """
    if q.device.type == "cpu":
        return _fwd_host(q, k, v, causal=causal, sm_scale=sm_scale, key_lengths=key_lengths,
                         return_lse=return_lse, out=out, lse_out=lse_out, path=path)
    B, H, N, d, Hkv, Nk = _shapes(q, k)
    dev = q.device
    dt = _dtype_code(q)
    _check_device_tensor("q", q, (B, H, N, d), q.dtype, dev)
    for name, t in (("k", k), ("v", v)):
        _check_device_tensor(name, t, (B, Hkv, Nk, d), q.dtype, dev)
    if dev.type != "cuda":
        raise ValueError("tensors must be CUDA tensors (or CPU tensors for the host path)")
    if out is None:
        out = torch.empty_like(q)
    _check_device_tensor("out", out, (B, H, N, d), q.dtype, dev)
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, H, N), device=dev,
                                                               dtype=torch.float32)
        _check_device_tensor("lse_out", lse, (B, H, N), torch.float32, dev)
    if key_lengths is not None:
        _check_device_tensor("key_lengths", key_lengths, (B,), torch.int32, dev)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    if path not in _lib.PATHS:
        raise ValueError(f"path must be one of {sorted(_lib.PATHS)}")
    kl_ptr = key_lengths.data_ptr() if key_lengths is not None else None
    lse_ptr = lse.data_ptr() if lse is not None else None
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        if (Hkv, Nk) == (H, N) and dt == _lib.DTYPE_F16:
            what = "attn_fwd_path"
            st = _lib.lib().attn_fwd_path(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, N, d,
                float(sm_scale), int(bool(causal)), kl_ptr, _lib.PATHS[path], stream)
        else:
            what = "attn_fwd_ex"
            st = _lib.lib().attn_fwd_ex(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, Hkv, N, Nk,
                d, dt, float(sm_scale), int(bool(causal)), kl_ptr, _lib.PATHS[path], stream)
    if st != _lib.ATTN_OK:
        raise _lib.AttnError(st, what)
    return (out, lse) if return_lse else out


def _dtype_code(q):
    if q.dtype == torch.float16:
        return _lib.DTYPE_F16
    if q.dtype == torch.bfloat16:
        return _lib.DTYPE_BF16
    if q.dtype == torch.float32:
        return _lib.DTYPE_F32
    raise TypeError(f"q must be torch.float16, torch.bfloat16 or torch.float32, got {q.dtype}")


def _shapes(q, k):
    """(B, H, N, d, H_kv, N_k) of q [B, H, N, d] and k [B, H_kv, N_k, d]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, H, N, d] and k, v [B, H_kv, N_k, d]")
    B, H, N, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or Hkv < 1 or H % Hkv != 0:
        raise ValueError("k, v must be [B, H_kv, N_k, d] with H a multiple of H_kv")
    return B, H, N, d, Hkv, Nk


def fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
                sm_scale: float | None = None, key_lengths: torch.Tensor | None = None,
                return_lse: bool = False, out: torch.Tensor | None = None,
                lse_out: torch.Tensor | None = None, n_splits: int = 0,
                workspace: torch.Tensor | None = None):
    """fwd() with the keys of every query tile pair split into n_splits ranges that run as
    separate work units and are merged exactly (attn_fwd_splitkv, attn_fwd_splitkv_ex for
    k, v of another shape than q). n_splits <= 0 chooses the count for the current device.
    workspace: a CUDA tensor of at least splitkv_workspace_bytes(...) bytes (allocated here
    when None). Device tensors only."""
    B, H, N, d, Hkv, Nk = _shapes(q, k)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("fwd_splitkv takes CUDA tensors")
    dt = _dtype_code(q)
    _check_device_tensor("q", q, (B, H, N, d), q.dtype, dev)
    for name, t in (("k", k), ("v", v)):
        _check_device_tensor(name, t, (B, Hkv, Nk, d), q.dtype, dev)
    if out is None:
        out = torch.empty_like(q)
    _check_device_tensor("out", out, (B, H, N, d), q.dtype, dev)
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, H, N), device=dev,
                                                               dtype=torch.float32)
        _check_device_tensor("lse_out", lse, (B, H, N), torch.float32, dev)
    if key_lengths is not None:
        _check_device_tensor("key_lengths", key_lengths, (B,), torch.int32, dev)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    L = _lib.lib()
    with torch.cuda.device(dev):
        if n_splits <= 0:
            n_splits = L.attn_splitkv_auto_splits_ex(B, H, Hkv, N, Nk, d, int(bool(causal)))
        need = L.attn_splitkv_workspace_bytes(B, H, N, d, int(n_splits))
        if need == 0:
            raise ValueError(f"invalid split-KV sizes (n_splits={n_splits})")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the device of q")
        stream = torch.cuda.current_stream(dev).cuda_stream
        lse_ptr = lse.data_ptr() if lse is not None else None
        kl_ptr = key_lengths.data_ptr() if key_lengths is not None else None
        ws_bytes = workspace.numel() * workspace.element_size()
        if (Hkv, Nk) == (H, N) and dt == _lib.DTYPE_F16:
            what = "attn_fwd_splitkv"
            st = L.attn_fwd_splitkv(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, N, d,
                float(sm_scale), int(bool(causal)), kl_ptr, int(n_splits), workspace.data_ptr(),
                ws_bytes, stream)
        else:
            what = "attn_fwd_splitkv_ex"
            st = L.attn_fwd_splitkv_ex(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, Hkv, N,
                Nk, d, dt, float(sm_scale), int(bool(causal)), kl_ptr, int(n_splits),
                workspace.data_ptr(), ws_bytes, stream)
    if st != _lib.ATTN_OK:
        raise _lib.AttnError(st, what)
    return (out, lse) if return_lse else out


def splitkv_workspace_bytes(B: int, H: int, N: int, d: int, n_splits: int) -> int:
    """Workspace bytes fwd_splitkv needs (0 for invalid sizes)."""
    return int(_lib.lib().attn_splitkv_workspace_bytes(B, H, N, d, n_splits))


def fwd_naive(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
              sm_scale: float | None = None, key_lengths: torch.Tensor | None = None,
              return_lse: bool = False, out: torch.Tensor | None = None,
              lse_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """The naive three-pass forward (attn_fwd_naive): S and P written to and read back from
    `workspace`, a CUDA tensor of at least naive_workspace_bytes(B, H, N) bytes (allocated here
    when None). The library's comparison baseline; fp16 self-attention, device tensors only."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("fwd_naive takes CUDA tensors")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_device_tensor(name, t, (B, H, N, d), torch.float16, dev)
    if out is None:
        out = torch.empty_like(q)
    _check_device_tensor("out", out, (B, H, N, d), torch.float16, dev)
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, H, N), device=dev,
                                                               dtype=torch.float32)
        _check_device_tensor("lse_out", lse, (B, H, N), torch.float32, dev)
    if key_lengths is not None:
        _check_device_tensor("key_lengths", key_lengths, (B,), torch.int32, dev)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    L = _lib.lib()
    need = naive_workspace_bytes(B, H, N)
    if need == 0:
        raise ValueError("invalid sizes for the naive forward")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the device of q")
    with torch.cuda.device(dev):
        st = L.attn_fwd_naive(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
            lse.data_ptr() if lse is not None else None, B, H, N, d, float(sm_scale),
            int(bool(causal)), key_lengths.data_ptr() if key_lengths is not None else None,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            torch.cuda.current_stream(dev).cuda_stream)
    if st != _lib.ATTN_OK:
        raise _lib.AttnError(st, "attn_fwd_naive")
    return (out, lse) if return_lse else out


def naive_workspace_bytes(B: int, H: int, N: int) -> int:
    """Workspace bytes fwd_naive needs (0 for invalid sizes)."""
    return int(_lib.lib().attn_naive_workspace_bytes(B, H, N))


# Host problems at least this large (Q, K, V and O together) are copied and computed in pieces.
_HOST_CHUNK_MIN_BYTES = 64 << 20
_HOST_PIECES = 8


def _host_pieces(q, k):
    """Independent pieces of a host problem, at most _HOST_PIECES: (q index, k/v index, batch
    index) triples, each a run of batches, or a run of key/value heads (with their query-head
    groups) of one batch, so that every piece is a contiguous block of q, k, v and o. None when
    the problem is small or cannot be split."""
    B, H = q.shape[0], q.shape[1]
    Hkv = k.shape[1]
    total = (q.numel() * 2 + k.numel() * 2) * q.element_size()
    if total < _HOST_CHUNK_MIN_BYTES or B * Hkv < 2:
        return None
    if B >= _HOST_PIECES:
        cut = [B * i // _HOST_PIECES for i in range(_HOST_PIECES + 1)]
        return [((slice(cut[i], cut[i + 1]),), (slice(cut[i], cut[i + 1]),), slice(cut[i], cut[i + 1]))
                for i in range(_HOST_PIECES)]
    g = H // Hkv
    per = max(1, min(Hkv, _HOST_PIECES // B)) # pieces per batch
    cut = [Hkv * i // per for i in range(per + 1)]
    return [((slice(b, b + 1), slice(cut[i] * g, cut[i + 1] * g)), (slice(b, b + 1), slice(cut[i], cut[i + 1])),
             slice(b, b + 1)) for b in range(B) for i in range(per)]


_host_streams = {}


def _pipeline_streams(dev):
    """(input copies, kernels, output copies) streams of a device, created once."""
    key = dev.index
    if key not in _host_streams:
        _host_streams[key] = tuple(torch.cuda.Stream(dev) for _ in range(3))
    return _host_streams[key]


def _fwd_host(q, k, v, *, causal, sm_scale, key_lengths, return_lse, out, lse_out, path):
    """Host tensors in, host tensors out. Large problems go as a pipeline of independent
    (batch, head) pieces: the input copies run back to back on one stream, each piece's kernel
    on a second once its inputs are in, and its output copy on a third once it is done, so the
    copies overlap the kernels and each other. The result is the same as one call."""
    dev = torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if return_lse and lse_out is None:
        lse_out = torch.empty(q.shape[:3], dtype=torch.float32, pin_memory=True)
    pieces = _host_pieces(q, k)
    cur = torch.cuda.current_stream(dev)
    if pieces is None:
        qd, kd, vd = (x.to(dev, non_blocking=True) for x in (q, k, v))
        kld = key_lengths.to(dev, non_blocking=True) if key_lengths is not None else None
        res = fwd(qd, kd, vd, causal=causal, sm_scale=sm_scale, key_lengths=kld,
                  return_lse=return_lse, path=path)
        o_dev, lse_dev = res if return_lse else (res, None)
        out.copy_(o_dev, non_blocking=True)
        if return_lse:
            lse_out.copy_(lse_dev, non_blocking=True)
        cur.synchronize()
        return (out, lse_out) if return_lse else out
    s_in, s_run, s_out = _pipeline_streams(dev)
    for st in (s_in, s_run, s_out):
        st.wait_stream(cur)
    keep = []  # device tensors of every piece, alive until the streams are done
    for qs, ks, bs in pieces:
        with torch.cuda.stream(s_in):
            qd = q[qs].to(dev, non_blocking=True)
            kd = k[ks].to(dev, non_blocking=True)
            vd = v[ks].to(dev, non_blocking=True)
            kld = key_lengths[bs].to(dev, non_blocking=True) if key_lengths is not None else None
            loaded = torch.cuda.Event()
            loaded.record(s_in)
        s_run.wait_event(loaded)
        with torch.cuda.stream(s_run):
            res = fwd(qd, kd, vd, causal=causal, sm_scale=sm_scale, key_lengths=kld,
                      return_lse=return_lse, path=path)
            o_dev, lse_dev = res if return_lse else (res, None)
            done = torch.cuda.Event()
            done.record(s_run)
        s_out.wait_event(done)
        with torch.cuda.stream(s_out):
            out[qs].copy_(o_dev, non_blocking=True)
            if return_lse:
                lse_out[qs].copy_(lse_dev, non_blocking=True)
        keep.append((qd, kd, vd, kld, o_dev, lse_dev))
    s_out.synchronize()
    for st in (s_in, s_run):
        st.synchronize()
    return (out, lse_out) if return_lse else out


def auto_path(N: int, d: int) -> str:
    """Name of the kernel the "auto" path runs for sequence length N and head dimension d."""
    code = _lib.lib().attn_auto_path(int(N), int(d))
    for name, c in _lib.PATHS.items():
        if c == code and name != "auto":
            return name
    raise ValueError(f"unsupported head dimension {d}")


def auto_path_ex(H: int, H_kv: int, N_q: int, N_k: int, d: int, dtype: str = "f16",
                 causal: bool = False) -> str:
    """Name of the kernel the "auto" path runs for H query heads over H_kv key/value heads, N_q
    query rows over N_k keys, head dimension d and element type "f16", "bf16" or "f32"."""
    dt = {"f16": _lib.DTYPE_F16, "bf16": _lib.DTYPE_BF16, "f32": _lib.DTYPE_F32}[dtype]
    code = _lib.lib().attn_auto_path_ex(int(H), int(H_kv), int(N_q), int(N_k), int(d), dt,
                                        int(bool(causal)))
    for name, c in _lib.PATHS.items():
        if c == code and name != "auto":
            return name
    raise ValueError("unsupported shape or element type")


def read_device_status() -> int:
    """Synchronizes the current stream and returns (and clears) the device status word."""
    stream = torch.cuda.current_stream().cuda_stream
    return _lib.lib().attn_read_device_status(stream)
