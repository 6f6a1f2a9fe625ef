"""Pins of the scheduler oracle: hand-worked deals, brute-force coverage and
the makespan property LPT is for (CPU only)."""

import itertools

import numpy as np

from oracle import sched as S


def test_hand_worked_zigzag_three_sms_seven_tiles():
    # One head, tile_rows = 1: each sequence is one tile, work = its length.
    # Sorted by work (descending, stable): b = 3(9), 0(7), 5(7), 2(5), 6(4), 1(2), 4(1)
    # pass 0 left->right: SM0 <- b3, SM1 <- b0, SM2 <- b5
    # pass 1 right->left: SM2 <- b2, SM1 <- b6, SM0 <- b1
    # pass 2 left->right: SM0 <- b4
    lengths = [7, 2, 5, 9, 1, 7, 4]
    sm_ptr, tiles = S.schedule(lengths, H=1, tile_rows=1 << 20, num_sms=3)
    assert sm_ptr == [0, 3, 5, 7]
    assert [t[0] for t in tiles] == [3, 1, 4, 0, 6, 5, 2]
    assert all(t[1] == 0 and t[2] == 0 for t in tiles)


def test_naive_is_round_robin_in_enumeration_order():
    sm_ptr, tiles = S.schedule([300, 10], H=2, tile_rows=128, num_sms=4, zigzag=False)
    # enumeration: (0,0,0) (0,0,1) (0,0,2) (0,1,0) (0,1,1) (0,1,2) (1,0,0) (1,1,0)
    assert sm_ptr == [0, 2, 4, 6, 8]
    # SM s takes enumeration positions s and s + 4
    assert tiles == [(0, 0, 0), (0, 1, 1), (0, 0, 1), (0, 1, 2),
                     (0, 0, 2), (1, 0, 0), (0, 1, 0), (1, 1, 0)]


def test_every_tile_exactly_once_brute_force():
    for lengths in itertools.product([0, 1, 63, 64, 65, 200], repeat=3):
        for num_sms in (1, 2, 5):
            for zz in (True, False):
                sm_ptr, tiles = S.schedule(list(lengths), 2, 64, num_sms, zigzag=zz)
                want = sorted((b, h, m) for b, L in enumerate(lengths)
                              for h in range(2) for m in range(-(-L // 64)))
                assert sorted(tiles) == want
                assert sm_ptr[0] == 0 and sm_ptr[-1] == len(tiles)
                assert all(a <= b for a, b in zip(sm_ptr, sm_ptr[1:]))


def test_fixed_rows_and_work_for_broadcast_q():
    sm_ptr, tiles = S.schedule([5, 700, 64], H=1, tile_rows=256, num_sms=2, fixed_rows=256)
    # one Q tile per sequence; work = K/V length: order b1, b0... sorted 1(700), 2(64), 0(5)
    assert sorted(tiles) == [(0, 0, 0), (1, 0, 0), (2, 0, 0)]
    assert tiles[sm_ptr[0]] == (1, 0, 0)
    sm_ptr, tiles = S.schedule([5, 700], H=1, tile_rows=128, num_sms=3, fixed_work=256)
    assert len(tiles) == 1 + 6


def test_lpt_zigzag_beats_naive_on_stress_shape():
    rng = np.random.default_rng(3)
    lengths = list(np.concatenate([np.full(4, 16384), rng.integers(1, 257, 252)]))
    for sms in (148, 152):
        a = S.schedule(lengths, 4, 128, sms, zigzag=True)
        b = S.schedule(lengths, 4, 128, sms, zigzag=False)
        assert S.makespan(*a, lengths) <= S.makespan(*b, lengths)
