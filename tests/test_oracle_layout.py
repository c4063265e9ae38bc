"""Pins for the oracle's layout, positions and temporal causal mask.

Pinned against: hand-derived fixtures (tests/golden), closed forms stated by
the SimSD pages (identity order; counts), and a simulation of the decoding
process that derives each slot's visible set step by step.
"""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    P = B = None
    tau = positions = None
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "P":
                P = int(vals[0])
            elif key == "B":
                B = int(vals[0])
            elif key == "tau":
                tau = [int(v) for v in vals]
            elif key == "positions":
                positions = [int(v) for v in vals]
            elif key == "row":
                rows.append([int(v) for v in vals[1:]])
    return P, B, np.array(tau), np.array(positions), np.array(rows, np.uint8)


@pytest.mark.parametrize("name", ["mask_P2_B4_tau3142.txt", "mask_P1_B4_identity.txt"])
def test_golden_fixture(name):
    P, B, tau, positions, mask = read_golden(name)
    pos, m = oracle.layout(P, tau)
    np.testing.assert_array_equal(pos, positions)
    np.testing.assert_array_equal(m, mask)


def test_identity_order_closed_form():
    # identity tau: slot i sees D_1..D_{i-1} and D~_i..D~_B (plus prompt)
    for B in range(1, 10):
        for P in (0, 1, 5):
            _, m = oracle.layout(P, np.arange(1, B + 1))
            for i in range(B):
                row = m[B + i]
                assert row[:P].all()
                exp_D = np.array([j < i for j in range(B)], np.uint8)
                exp_S = np.array([j >= i for j in range(B)], np.uint8)
                np.testing.assert_array_equal(row[P:P + B], exp_D)
                np.testing.assert_array_equal(row[P + B:], exp_S)


def simulate_visible_sets(B, tau):
    """Walk the decoding steps: at step s the data tokens decoded at earlier
    steps are revealed and the slots not yet decoded are still masked.  The
    slot decoded at step s sees exactly that context; a data token decoded
    at step s sees the data tokens revealed up to and including step s."""
    slot_sees, data_sees = {}, {}
    revealed = set()
    for s in range(1, B + 1):
        unresolved = {j for j in range(B) if tau[j] >= s}
        (i,) = [j for j in range(B) if tau[j] == s]
        slot_sees[i] = (set(revealed), unresolved)
        revealed.add(i)
        data_sees[i] = set(revealed)
    return slot_sees, data_sees


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6])
def test_all_orders_match_decoding_simulation(B):
    P = 3
    for perm in itertools.permutations(range(1, B + 1)):
        tau = np.array(perm)
        _, m = oracle.layout(P, tau)
        slot_sees, data_sees = simulate_visible_sets(B, list(perm))
        for i in range(B):
            D_vis, S_vis = slot_sees[i]
            row = m[B + i]
            assert row[:P].all()
            assert {j for j in range(B) if row[P + j]} == D_vis
            assert {j for j in range(B) if row[P + B + j]} == S_vis
            drow = m[i]
            assert drow[:P].all()
            assert {j for j in range(B) if drow[P + j]} == data_sees[i]
            assert not drow[P + B:].any()


def test_counts_and_no_self_reference():
    rng = np.random.default_rng(7)
    for B in (1, 4, 8, 16, 32):
        for _ in range(5):
            tau = rng.permutation(B) + 1
            P = int(rng.integers(0, 40))
            _, m = oracle.layout(P, tau)
            tail = m[:, P:]
            # every slot row sees B new columns, every data row tau(i)
            np.testing.assert_array_equal(m[B:].sum(1), P + B)
            np.testing.assert_array_equal(m[:B].sum(1), P + tau)
            assert int(tail.sum()) == B * B + B * (B + 1) // 2
            for i in range(B):
                assert m[B + i, P + i] == 0          # slot never sees its own data token
                assert m[B + i, P + B + i] == 1      # but sees itself
                assert m[i, P + i] == 1


def test_positions_copy_rule():
    rng = np.random.default_rng(3)
    for B in (1, 4, 16):
        for P in (0, 64, 1000):
            pos, _ = oracle.layout(P, rng.permutation(B) + 1, with_mask=False)
            np.testing.assert_array_equal(pos[:P], np.arange(P))
            np.testing.assert_array_equal(pos[P:P + B], P + np.arange(B))
            np.testing.assert_array_equal(pos[P + B:], pos[P:P + B])
    # the tiny workload: prompt 0..63, D at 64..67, copied for the slots
    pos, _ = oracle.layout(64, [2, 4, 1, 3], with_mask=False)
    assert list(pos[64:68]) == [64, 65, 66, 67] and list(pos[68:]) == [64, 65, 66, 67]


@pytest.mark.parametrize("tau", [[1, 1, 2], [0, 1, 2], [1, 2, 4], [2, 3, 4]])
def test_rejects_non_permutation(tau):
    assert not oracle.tau_is_permutation(tau)
    with pytest.raises(oracle.OracleError):
        oracle.layout(4, tau)
