"""Host model of the grouped GEMM's stage barriers (csrc/gemm_w4.cu), run under random
interleavings of its three pipeline roles.

The kernel's roles per k-block i:
  * A producer (the dequantising warps): waits until the MMAs of k-block i - SA are
    done, writes A stage i % SA, arrives on a_full[i % SA];
  * B producer (the gather warps, deferring each arrival by D = SB - 2 k-blocks, or the
    TMA thread with D = 0): waits until the MMAs of k-block i - SB are done, fills token
    stage i % SB, arrives on its ready barrier for k-block i - D: b_full[.] or, merged
    (tiles of up to 64 rows with A in TMEM, SB = SA), on a_full[.];
  * MMA thread: waits a_full[i % SA] (and b_full[i % SB] when not merged), reads both
    stages, commits once to done[i % SD], SD = max(SA, SB).
An mbarrier only compares phase parity: a wait for phase n succeeds once the phase
count c has passed n (c & 1 != n & 1). The protocol is right only if every wait sees
c in {n, n + 1}, every arrival lands in the phase it belongs to, the MMA reads the
data of its own k-block, and no schedule deadlocks. The model checks all four.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # completed phases

    def arrive(self, n):
        assert n == self.phase, f"arrival for phase {n} while phase {self.phase} is open"
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def test(self, n):
        """mbarrier try_wait.parity for phase n, with the aliasing check."""
        assert self.phase in (n, n + 1), f"waiting for phase {n} at phase count {self.phase}"
        return (self.phase & 1) != (n & 1)


def run(SA, SB, merged, tma_b, n_iters, seed, merge_any=False):
    assert merge_any or not merged or SA == SB
    SD = max(SA, SB)
    D = 0 if tma_b else SB - 2
    a_full = [Barrier(2 if merged else 1) for _ in range(SA)]
    b_full = [Barrier(1) for _ in range(SB)]
    done = [Barrier(1) for _ in range(SD)]
    # merged: the token tile of k-block j arrives on the A barrier of k-block j
    b_ready = a_full if merged else b_full
    b_index = SA if merged else SB
    a_stage = [None] * SA
    b_stage = [None] * SB
    rng = random.Random(seed)
    st = dict(a=0, b=0, b_arrived=0, m=0)

    def wait_done(j):  # the MMAs of k-block j are complete
        return j < 0 or done[j % SD].test(j // SD)

    def step_a():
        i = st["a"]
        if i >= n_iters or not wait_done(i - SA):
            return False
        a_stage[i % SA] = i
        a_full[i % SA].arrive(i // SA)
        st["a"] += 1
        return True

    def step_b():
        i = st["b"]
        if i < n_iters:
            if not wait_done(i - SB):
                return False
            b_stage[i % SB] = i
            st["b"] += 1
            # arrivals trail the issues by D k-blocks (all of them at the end)
            while st["b_arrived"] <= st["b"] - 1 - D:
                j = st["b_arrived"]
                b_ready[j % b_index].arrive(j // b_index)
                st["b_arrived"] += 1
            return True
        if st["b_arrived"] < n_iters:
            j = st["b_arrived"]
            b_ready[j % b_index].arrive(j // b_index)
            st["b_arrived"] += 1
            return True
        return False

    def step_m():
        i = st["m"]
        if i >= n_iters:
            return False
        if not a_full[i % SA].test(i // SA):
            return False
        if not merged and not b_full[i % SB].test(i // SB):
            return False
        assert a_stage[i % SA] == i, f"MMA {i} read A of k-block {a_stage[i % SA]}"
        assert b_stage[i % SB] == i, f"MMA {i} read B of k-block {b_stage[i % SB]}"
        done[i % SD].arrive(i // SD)
        st["m"] += 1
        return True

    roles = [step_a, step_b, step_m]
    idle = 0
    while st["m"] < n_iters:
        r = rng.choice(roles)
        idle = 0 if r() else idle + 1
        assert idle < 10000, f"no role can move: {st}"
    return st


@pytest.mark.parametrize("SA,SB,merged,tma_b", [
    (2, 8, False, False),  # gate/up, 128-row tiles: A in shared memory, deep token ring
    (2, 3, False, False),  # 256-row gate/up tiles: three token stages
    (4, 8, False, True),   # down at 128 rows: A in TMEM, token tiles by TMA
    (4, 4, True, False),   # tiles of up to 64 rows, gathers on the merged barrier
    (4, 4, True, True),    # down at up to 64 rows, TMA on the merged barrier
    (3, 3, True, False),   # three stages, merged
])
def test_stage_barriers_hold_under_random_schedules(SA, SB, merged, tma_b):
    for seed in range(30):
        st = run(SA, SB, merged, tma_b, n_iters=97, seed=seed)
        assert st["a"] == st["b"] == st["m"] == 97


def test_the_model_catches_a_ring_too_shallow():
    """A completion ring shorter than the A stages lets the A producer wait on a
    barrier two phases ahead of it: the parity check must flag it."""
    def shallow(SA, SB, seed):
        # as run(), with SD one short of SA
        SD = SA - 1
        a_full = [Barrier(1) for _ in range(SA)]
        done = [Barrier(1) for _ in range(SD)]
        rng = random.Random(seed)
        a = m = 0
        while m < 60:
            if rng.random() < 0.5 and a < 60:
                j = a - SA
                if j < 0 or done[j % SD].test(j // SD):
                    a_full[a % SA].arrive(a // SA)
                    a += 1
            elif m < a and a_full[m % SA].test(m // SA):
                done[m % SD].arrive(m // SD)
                m += 1
    with pytest.raises(AssertionError):
        for seed in range(50):
            shallow(4, 4, seed)


def test_the_model_catches_a_merged_barrier_with_a_deeper_token_ring():
    """Merged, the token ring must not run ahead of the A ring: with 8 token stages
    over 4 A stages the gathers can arrive for a k-block whose A barrier is still on
    an earlier phase, and the model must flag it."""
    with pytest.raises(AssertionError):
        for seed in range(50):
            run(4, 8, True, False, n_iters=97, seed=seed, merge_any=True)
