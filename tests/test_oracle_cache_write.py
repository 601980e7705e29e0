"""Pins of the oracle's paged cache write (no GPU)."""
import json
import os

import numpy as np

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import cache_write, gather_latent, slot_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cache_write_hand_case.json")


def test_hand_case():
    g = json.load(open(GOLDEN))
    nb, bs, e = g["num_blocks"], g["block_size"], g["entry_dim"]
    cache = np.array([[100 + 10 * s, 101 + 10 * s] for s in range(nb * bs)], dtype=np.int64).reshape(nb, bs, e)
    lat = np.array([[1000 + 10 * t, 1001 + 10 * t] for t in range(len(g["slot_mapping"]))], dtype=np.int64)
    out = cache_write(cache, lat, np.array(g["slot_mapping"], dtype=np.int64))
    np.testing.assert_array_equal(out.reshape(nb * bs, e), np.array(g["expected_flat"]))
    np.testing.assert_array_equal(cache.reshape(nb * bs, e)[0], [100, 101])   # input untouched


def test_round_trip_through_the_gather():
    # Writing a request's new positions at the slots the block table gives them, then
    # gathering those positions, returns the written rows (ties the write to the gather).
    rng = np.random.default_rng(3)
    nb, bs, e = 16, 4, 8
    cache = rng.integers(0, 1 << 16, size=(nb, bs, e)).astype(np.uint16)
    table = rng.permutation(nb)[:12].reshape(2, 6).astype(np.int32)
    starts, lens = [3, 10], [9, 7]           # positions [3, 12) of request 0, [10, 17) of request 1
    slots = np.array([slot_of(table, r, p, bs) for r in range(2) for p in range(starts[r], starts[r] + lens[r])])
    lat = rng.integers(0, 1 << 16, size=(len(slots), e)).astype(np.uint16)
    out = cache_write(cache, lat, slots)
    cu = wl.indptr_from_lengths(lens)
    back = gather_latent(out, table, cu, np.array(starts, dtype=np.int32))
    np.testing.assert_array_equal(back, lat)
    # every slot not written keeps its old row
    keep = np.setdiff1d(np.arange(nb * bs), slots)
    np.testing.assert_array_equal(out.reshape(-1, e)[keep], cache.reshape(-1, e)[keep])


def test_padding_slots_write_nothing():
    rng = np.random.default_rng(4)
    cache = rng.integers(0, 1 << 16, size=(5, 3, 4)).astype(np.uint16)
    lat = rng.integers(0, 1 << 16, size=(6, 4)).astype(np.uint16)
    np.testing.assert_array_equal(cache_write(cache, lat, np.full(6, -1, dtype=np.int64)), cache)


def test_repeated_slot_keeps_the_later_token():
    cache = np.zeros((2, 2, 1), dtype=np.int64)
    lat = np.array([[7], [8], [9]], dtype=np.int64)
    out = cache_write(cache, lat, np.array([3, 0, 3], dtype=np.int64))
    assert out.reshape(-1)[3] == 9 and out.reshape(-1)[0] == 8
