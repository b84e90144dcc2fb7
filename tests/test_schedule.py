"""Host-side unit schedule of the tiled kernel (CPU only, through attn_debug_schedule).

A unit is (batch * head, pair of 128-row Q tiles), numbered in the kernel's unit order: head
blocks of `head_block` heads, inside a block the pairs from the last one down and the heads of
the block next to each other. These tests derive every expectation from that definition and
the causal tile counts, not from the library:
- the dynamic order is a permutation that keeps the unit order up to a head-block boundary and
  sorts the rest heaviest first, over at most three head blocks;
- the static table deals every unit exactly once, largest-first, so per-CTA loads differ by at
  most one unit's weight;
- the dynamic schedule starts at three units per multiprocessor;
- bad arguments are refused.
"""
import ctypes

import numpy as np
import pytest

from exact_scaled_dot_attn_gb300 import _lib

KBM = 128  # query rows per Q tile = keys per K/V tile


def schedule(BH, N, Nk, d, G=1, causal=1, sms=152, cap=None):
    L = _lib.lib()
    n_pairs = (N + 2 * KBM - 1) // (2 * KBM)
    cap = BH * n_pairs if cap is None else cap
    units = np.full(max(cap, 1), -1, dtype=np.int32)
    off = np.zeros(sms + 1, dtype=np.int32)
    n = ctypes.c_int(-1)
    hb = ctypes.c_int(-1)
    r = L.attn_debug_schedule(BH, N, Nk, d, G, causal, sms, units.ctypes.data, cap,
                              off.ctypes.data, ctypes.byref(n), ctypes.byref(hb))
    return r, units[:max(n.value, 0)], off, n.value, hb.value


def sorted_tail_start(units, per_block):
    """Head-block boundary from which the dynamic order leaves the unit order (the heaviest
    units of the first sorted block may keep their places)."""
    n = len(units)
    first = next((i for i in range(n) if units[i] != i), n)
    cut = first // per_block * per_block
    assert np.array_equal(units[:cut], np.arange(cut))
    return cut


def weights(BH, N, Nk, causal, hb):
    """(Q tile, K/V tile) steps of every unit in the unit order."""
    n_pairs = (N + 2 * KBM - 1) // (2 * KBM)
    per_block = hb * n_pairs
    w = np.zeros(BH * n_pairs, dtype=np.int64)
    for u in range(BH * n_pairs):
        blk, r = divmod(u, per_block)
        heads = min(hb, BH - blk * hb)
        pair = n_pairs - 1 - r // heads
        q0 = pair * 2 * KBM
        ends = []
        for t in range(2):
            if q0 + t * KBM >= N:
                ends.append(0)
                continue
            e = min(Nk, q0 + (t + 1) * KBM + Nk - N) if causal else Nk
            ends.append(max(0, e))
        w[u] = sum((e + KBM - 1) // KBM for e in ends)
    return w


def test_dynamic_order_prefill():
    BH, N, d = 128, 4096, 128  # 4 batches x 32 heads
    r, units, _, n, hb = schedule(BH, N, N, d)
    assert r == 1 and n == BH * 16
    assert hb == 8  # K and V of one head are 2 MB at N = 4096; a block holds 16 MB
    assert sorted(units.tolist()) == list(range(n))
    per_block = hb * 16
    cut = sorted_tail_start(units, per_block)
    assert 0 < n - cut <= 3 * per_block
    w = weights(BH, N, N, True, hb)
    tail = w[units[cut:]]
    assert np.all(tail[:-1] >= tail[1:])          # heaviest first
    assert sorted(units[cut:].tolist()) == list(range(cut, n))
    # the sorted share is about a fifth of the work (one head block of slack)
    assert w[cut:].sum() <= 0.2 * w.sum() + w[cut - per_block:cut].sum() + 1


def test_dynamic_tail_capped_at_three_blocks():
    BH, N, d = 32, 32768, 128  # one head per 16 MB block
    r, units, _, n, hb = schedule(BH, N, N, d)
    assert r == 1 and hb == 1 and n == 32 * 128
    cut = sorted_tail_start(units, 128)
    assert n - cut == 3 * 128  # 20 % of the work would span six blocks; the cap keeps three
    w = weights(BH, N, N, True, hb)
    tail = w[units[cut:]]
    assert np.all(tail[:-1] >= tail[1:])


def test_grouped_heads_widen_the_block():
    # 4 query heads per key/value head: a block holds 4x the query heads for the same K/V bytes
    _, _, _, _, hb1 = schedule(128, 4096, 4096, 128, G=1)
    _, _, _, _, hb4 = schedule(128, 4096, 4096, 128, G=4)
    assert hb4 == 4 * hb1


@pytest.mark.parametrize("causal", [0, 1])
def test_static_table_deals_every_unit_once(causal):
    BH, N, d, sms = 8, 8192, 64, 152  # 8 x 16 = 128 units: below 3 per SM
    r, units, off, n, hb = schedule(BH, N, N, d, causal=causal, sms=sms)
    assert r == 0
    grid = min(n, sms)
    assert off[0] == 0 and off[grid] == n and np.all(np.diff(off[:grid + 1]) >= 0)
    dealt = np.concatenate([units[off[c]:off[c + 1]] for c in range(grid)])
    assert sorted(dealt.tolist()) == list(range(n))
    w = weights(BH, N, N, causal, hb) + 8  # + the unit-start cost in tile steps
    loads = np.array([w[units[off[c]:off[c + 1]]].sum() for c in range(grid)])
    assert loads.max() - loads.min() <= w.max()


def test_static_table_several_units_per_cta():
    BH, N, d, sms = 32, 2048, 128, 152  # 32 x 8 = 256 units on 152 SMs
    r, units, off, n, hb = schedule(BH, N, N, d, sms=sms)
    assert r == 0 and n == 256
    dealt = np.concatenate([units[off[c]:off[c + 1]] for c in range(sms)])
    assert sorted(dealt.tolist()) == list(range(n))
    w = weights(BH, N, N, True, hb) + 8
    loads = np.array([w[units[off[c]:off[c + 1]]].sum() for c in range(sms)])
    assert loads.max() - loads.min() <= w.max()


def test_dynamic_threshold_is_three_units_per_sm():
    sms = 152
    r_lo, *_ = schedule(3 * sms - 1, 256, 256, 64, sms=sms)  # one pair per head
    r_hi, *_ = schedule(3 * sms, 256, 256, 64, sms=sms)
    assert (r_lo, r_hi) == (0, 1)


def test_large_launches_take_the_unit_order():
    # more units than the table holds (4096): the dynamic schedule runs units in their order
    r, units, _, n, _ = schedule(64, 32768, 32768, 64)
    assert r == 1 and n == 64 * 128
    assert np.array_equal(units, np.arange(n))


def test_bad_arguments():
    assert schedule(0, 4096, 4096, 128)[0] == -1
    assert schedule(4, 4096, 4096, 48)[0] == -1
    assert schedule(4, 4096, 4096, 128, sms=0)[0] == -1
    assert schedule(4, 4096, 4096, 128, sms=257)[0] == -1
    assert schedule(4, 4096, 4096, 128, causal=2)[0] == -1
    assert schedule(4, 4096, 4096, 128, cap=10)[0] == -1  # 64 units
