"""Host model of the batch-1 decode kernel's cross-block protocol (csrc/decode.cu).

Per call every block reads the sync word and takes epoch = sync + 1 (0 skipped),
publishes its router partials as {value, epoch} words, polls every block's partials
until their epoch is this call's, publishes its h words the same way, polls every
block's h, and finishes; block 0 writes its epoch to the sync word as its last step.
Calls on one workspace run one after another (each launch waits for the previous
one's completion before its first read of that memory), while the blocks of one call
interleave arbitrarily. Nothing is reset between calls.

The model runs random interleavings and checks that every block of a call reads the
same epoch, that every poll returns that call's values (never an older call's), and
that no schedule stalls. The kernel's block 0 advances the sync word last; what makes
that safe is that by then it has polled a word every block published after reading
the sync word (already true after the router partials). The model plants the
ordering mistake the kernel avoids, block 0 advancing the sync word right after its
own read, and shows a slow block then picks up the next call's epoch.
"""
import random

import pytest


def run_calls(G, n_calls, seed, sync_early=False, start_sync=0):
    rng = random.Random(seed)
    sync = [start_sync]
    pub = [(0, None)] * G    # router partial words {epoch, value}
    pub_h = [(0, None)] * G  # h words
    for call in range(n_calls):
        value = ("call", call)
        # per block: a program of steps, run one step at a time in random order
        state = [dict(pc=0, epoch=None) for _ in range(G)]
        epochs = [None] * G

        def step(b):
            s = state[b]
            pc = s["pc"]
            if pc == 0:  # read the sync word
                e = (sync[0] + 1) & 0xFFFFFFFF
                s["epoch"] = e if e != 0 else 1
                epochs[b] = s["epoch"]
                if sync_early and b == 0:
                    sync[0] = s["epoch"]  # the planted mistake: advance before the others read
            elif pc == 1:
                pub[b] = (s["epoch"], value)
            elif pc == 2:  # poll every block's router partials
                if any(pub[o][0] != s["epoch"] for o in range(G)):
                    return False
                assert all(pub[o][1] == value for o in range(G)), "stale partial read"
            elif pc == 3:
                pub_h[b] = (s["epoch"], value)
            elif pc == 4:  # poll every block's h
                if any(pub_h[o][0] != s["epoch"] for o in range(G)):
                    return False
                assert all(pub_h[o][1] == value for o in range(G)), "stale h read"
            elif pc == 5:
                if b == 0 and not sync_early:
                    sync[0] = s["epoch"]  # the kernel's last step
            else:
                return False
            s["pc"] += 1
            return True

        idle = 0
        while any(s["pc"] < 6 for s in state):
            b = rng.randrange(G)
            idle = 0 if step(b) else idle + 1
            assert idle < 20000, f"call {call} stalled: {[s['pc'] for s in state]}"
        assert len(set(epochs)) == 1, f"call {call}: blocks read epochs {sorted(set(epochs))}"
    return sync[0]


@pytest.mark.parametrize("G", [2, 3, 8])
def test_every_call_sees_its_own_epoch_and_values(G):
    for seed in range(40):
        assert run_calls(G, n_calls=6, seed=seed) == 6


def test_the_epoch_skips_zero_when_it_wraps():
    """A workspace whose sync word holds 0xFFFFFFFF wraps to epoch 1, never 0 (the
    value a zero-filled workspace's words carry)."""
    assert run_calls(3, n_calls=2, seed=1, start_sync=0xFFFFFFFF) == 2


def test_the_model_catches_an_early_epoch_advance():
    with pytest.raises(AssertionError):
        for seed in range(200):
            run_calls(4, n_calls=3, seed=seed, sync_early=True)
