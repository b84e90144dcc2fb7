"""Partition of a host problem into the pieces of the end-to-end copy pipeline (CPU only).

api._host_pieces cuts a host problem into independent blocks. Each block is a run of batches,
or a run of key/value heads of one batch together with their query-head groups. Every query
head and every key/value head must fall in exactly one piece, and a piece's query heads must be
the groups of its key/value heads. Every piece must be one contiguous block of q, k, v and o.
Meta tensors stand in for the host tensors, so no memory of the full size is allocated.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_attn_gb300 import api


def _meta(*shape):
    return torch.empty(shape, dtype=torch.float16, device="meta")


def _range(sl, n):
    start, stop, step = sl.indices(n)
    assert step == 1
    return start, stop


SHAPES = [
    # B, H, H_kv, N, N_k, d
    (4, 32, 32, 4096, 4096, 128),   # prefill: fewer batches than pieces, split by heads
    (4, 32, 8, 4096, 4096, 128),    # grouped-query prefill
    (1, 16, 16, 8192, 8192, 128),   # one batch, heads only
    (2, 32, 8, 1024, 16384, 128),   # chunk of queries over a long cache
    (8, 32, 8, 1, 8192, 128),       # decode: one query per head, batches only
    (50, 12, 12, 2048, 2048, 32),   # many batches: runs of batches
    (9, 3, 1, 16384, 16384, 64),    # B just above the piece count, one key/value head
    (3, 6, 3, 16384, 16384, 64),    # 3 batches x 2 pieces each
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}kv{s[2]}Nq{s[3]}Nk{s[4]}d{s[5]}" for s in SHAPES])
def test_pieces_partition_the_problem(shape):
    B, H, Hkv, N, Nk, d = shape
    q, k = _meta(B, H, N, d), _meta(B, Hkv, Nk, d)
    pieces = api._host_pieces(q, k)
    assert pieces is not None, "problem large enough to be split"
    assert 2 <= len(pieces) <= api._HOST_PIECES
    G = H // Hkv
    q_seen = np.zeros((B, H), np.int32)
    kv_seen = np.zeros((B, Hkv), np.int32)
    for qs, ks, bs in pieces:
        b0, b1 = _range(bs, B)
        assert _range(qs[0], B) == (b0, b1) and _range(ks[0], B) == (b0, b1)
        if len(qs) == 1:
            # whole batches: every head of each
            assert len(ks) == 1
            q_seen[b0:b1, :] += 1
            kv_seen[b0:b1, :] += 1
        else:
            # one batch, a run of key/value heads with their query-head groups
            assert b1 - b0 == 1
            g0, g1 = _range(ks[1], Hkv)
            h0, h1 = _range(qs[1], H)
            assert (h0, h1) == (g0 * G, g1 * G), "query heads are the groups of the piece's K/V heads"
            assert g1 > g0
            q_seen[b0, h0:h1] += 1
            kv_seen[b0, g0:g1] += 1
        # each piece is one contiguous block of q (and so of o), k and v
        for t, sl in ((q, qs), (k, ks)):
            blk = t[sl]
            assert blk.is_contiguous() and blk.numel() > 0
    assert (q_seen == 1).all(), "every query head in exactly one piece"
    assert (kv_seen == 1).all(), "every key/value head in exactly one piece"


def test_small_or_unsplittable_problems_run_whole():
    # below the size threshold (the reranking batch: 39 MB of Q, K, V and O)
    assert api._host_pieces(_meta(2, 2, 128, 64), _meta(2, 2, 128, 64)) is None
    assert api._host_pieces(_meta(50, 12, 256, 32), _meta(50, 12, 256, 32)) is None
    # one batch with one key/value head cannot be cut into independent pieces
    assert api._host_pieces(_meta(1, 8, 65536, 128), _meta(1, 1, 65536, 128)) is None


def test_threshold_counts_q_k_v_and_o():
    # the size test counts Q, K, V and O: just under and at the threshold
    limit = api._HOST_CHUNK_MIN_BYTES
    d, H = 64, 2
    n_tok = limit // (4 * 2 * d * H)        # tokens per batch at which 4 tensors of fp16 hit it
    B = 2
    N_at = n_tok // B
    assert api._host_pieces(_meta(B, H, N_at, d), _meta(B, H, N_at, d)) is not None
    assert api._host_pieces(_meta(B, H, N_at - 1, d), _meta(B, H, N_at - 1, d)) is None
