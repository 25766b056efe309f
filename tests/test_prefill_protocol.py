"""Host-side check of the persistent prefill kernel's barrier protocol (no
GPU): the discrete-event model in prefill_protocol_model runs every role's
waits, arrivals and commits over random item lists with random latencies and
interleavings, and must find no deadlock, aliased parity wait, buffer race
or stale read; with any one of the protocol's waits removed it must find a
violation, so each wait is shown to be needed and the checks to bite."""
import random

import pytest

import prefill_protocol_model as pm


def _cases(n, seed):
    rng = random.Random(seed)
    return [(pm.random_items(rng), rng.choice([0, 1, 2]), 1000 + i) for i in range(n)]


def test_protocol_holds_on_random_item_streams():
    for items, T, seed in _cases(400, 1):
        pm.run(items, T, seed)


def test_protocol_edge_streams():
    for items in ([(0, 1)], [(0, 1)] * 9, [(3, 4)], [(0, 1), (7, 8), (0, 1), (2, 3)],
                  [(5, 6), (5, 6), (5, 6)], [(8, 9)] * 3):
        for seed in range(40):
            pm.run(items, 2, seed)


@pytest.mark.parametrize("name", ["q_full", "q_empty", "prev_item_qk", "q_sf", "ones",
                                  "o_free", "hand_over", "epilogue", "p_bank", "rescale_o",
                                  "s_read", "k_full", "k_ring", "v_full", "v_ring", "s_full",
                                  "p_ready", "qk_own"])
def test_each_wait_is_needed(name):
    for items, T, seed in _cases(400, 2):
        try:
            pm.run(items, T, seed, drop=(name,))
        except pm.ProtocolError:
            return
    pytest.fail(f"dropping the {name!r} wait went unnoticed")
