"""Automatic split-KV count (attn_splitkv_auto_splits[_ex]) on the host, at GB300's 152 SMs
(the count the library assumes where no device answers, and the count of the device itself).

The rule, from the header: a causal problem whose (Q tile pair) units already fill the SMs is not
split; otherwise equal ranges (SMs / pairs without the causal mask, about 2 * SMs / pairs with it) or
balanced runs over all pairs, whichever finishes sooner; never more than one range per two
128-key tiles, never more than 16, never fewer than 1. The decode counts checked here are the
ones the measured sweeps found fastest on GB300.
"""
import pytest
import torch

from exact_scaled_dot_attn_gb300 import _lib

SMS = 152


@pytest.fixture(scope="module")
def lib():
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != SMS:
        pytest.skip("counts below are for 152 SMs")
    return _lib.lib()


def pairs(B, H, Nq):
    return B * H * ((Nq + 255) // 256)


@pytest.mark.parametrize("B,H,N,d,causal", [
    (4, 32, 4096, 128, 1),    # prefill: 2048 pairs
    (50, 12, 256, 32, 0),     # reranking: 600 pairs
    (1, 32, 32768, 128, 1),   # long: 4096 pairs
])
def test_problems_that_fill_the_sms_are_not_split(lib, B, H, N, d, causal):
    assert pairs(B, H, N) >= SMS
    assert lib.attn_splitkv_auto_splits(B, H, N, d, causal) == 1


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,causal,expected", [
    (1, 1, 1, 32768, 32768, 1, 3),     # one causal head of 32768 (bench split_kv line)
    (8, 32, 8, 1, 8192, 1, 2),         # decoding, 64 packed groups (fastest in the sweep)
    (8, 32, 8, 8, 8192, 1, 2),         # a causal block of 8 draft queries, same groups
    (1, 32, 8, 1, 8192, 0, 16),        # 8 packed groups: 19 ranges wanted, 16 at most
])
def test_measured_decode_and_long_counts(lib, B, H, Hkv, Nq, Nk, causal, expected):
    assert lib.attn_splitkv_auto_splits_ex(B, H, Hkv, Nq, Nk, 128, causal) == expected


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk", [
    (1, 2, 2, 4096, 4096), (1, 4, 4, 2048, 2048), (2, 8, 2, 1, 1024), (1, 1, 1, 300, 300),
    (1, 1, 1, 1, 256), (1, 1, 1, 1, 128), (3, 6, 3, 17, 5000), (64, 32, 8, 1, 32768),
])
@pytest.mark.parametrize("causal", [0, 1])
def test_bounds(lib, B, H, Hkv, Nq, Nk, causal):
    s = lib.attn_splitkv_auto_splits_ex(B, H, Hkv, Nq, Nk, 64, causal)
    kv_tiles = (Nk + 127) // 128
    assert 1 <= s <= min(16, max(1, kv_tiles // 2))


def test_balanced_runs_fill_a_partial_last_wave(lib):
    # stress shape without the mask: 1024 pairs of 64 key tiles make 6.74 waves of whole pairs
    # (7 x (64 + 8) = 504 tile times); 152 runs of 432 tiles, each over at most 8 pairs, take
    # 432 + 8 x 8 = 496, so the launch uses balanced runs, two ranges per pair at most
    assert lib.attn_splitkv_auto_splits(2, 16, 8192, 64, 0) == 2
    # with the mask the pairs differ in length and only equal ranges apply: 1024 pairs fill the SMs
    assert lib.attn_splitkv_auto_splits(2, 16, 8192, 64, 1) == 1


def test_equal_ranges_without_the_mask(lib):
    # 32 pairs of 32 key tiles: four equal ranges make 128 units, one wave on 152 SMs; balanced
    # runs would need five or more ranges per pair and two units on most CTAs
    assert lib.attn_splitkv_auto_splits(1, 2, 4096, 128, 0) == SMS // 32


def test_invalid_sizes(lib):
    assert lib.attn_splitkv_auto_splits(0, 4, 4096, 128, 1) == -1
    assert lib.attn_splitkv_auto_splits(1, 4, 4096, 96, 1) == -1
    assert lib.attn_splitkv_auto_splits(1, 4, 0, 128, 1) == -1
