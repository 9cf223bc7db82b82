"""A host model of the verify kernel's state-chunk ring and its waits.

The state warp streams each item's state as eight chunks, in order, into a
ring of N chunk slots; gemv warp g takes chunk 8 i + g of item i, and the
operand ring (kNumOp slots) lets a gemv warp run up to kNumOp - 1 items ahead
of the slowest one.  Each slot has a full barrier whose phases complete as the
slot's copies land; a parity wait for lap L of a slot succeeds when the
barrier's current (incomplete) phase has the other parity, which is right only
if the slot's lap L - 1 has already completed.

The model plays random schedules (random consumer order, random copy
latencies) and checks, at every successful wait, which copy the consumer
would read.  The parity-only wait can succeed one lap early at the ring sizes
the kernel uses (21 slots at C2, 18 in the fold variant); with the lap rule
(the producer records the lap it arms, a consumer first waits for its own
lap) every successful wait reads its own copy.  The kernel's wait is
warp_wait_chunk in csrc/kda_verify.cu."""
from __future__ import annotations

import random

import pytest

GEMV_WARPS = 8


def simulate(n_slots: int, n_op: int, items: int, seed: int, lap_rule: bool) -> int:
    """Returns how many successful chunk waits matched a phase other than the
    consumer's own lap (0 means the protocol held)."""
    rng = random.Random(seed)
    completed = [0] * n_slots        # phases completed per slot's full barrier
    consumed = [0] * n_slots         # laps released per slot (its empty barrier)
    lap = [-1] * n_slots             # lap last armed, as the producer records it
    in_flight = []                   # (slot, lap) copies issued, not landed
    issued = 0                       # chunks the producer has armed
    done_items = [0] * GEMV_WARPS    # items each gemv warp has finished
    waiting = [None] * GEMV_WARPS    # the chunk each gemv warp waits for
    wrong = 0
    total = items * GEMV_WARPS
    for _ in range(400 * total):
        if min(done_items) >= items:
            break
        action = rng.random()
        if action < 0.3 and issued < total:
            # the producer arms the next chunk once its slot's previous lap is released
            pos, L = issued % n_slots, issued // n_slots
            if consumed[pos] >= L:
                lap[pos] = L
                in_flight.append((pos, L))
                issued += 1
        elif action < 0.55 and in_flight:
            # a copy lands: any in-flight copy, not only the oldest
            k = rng.randrange(len(in_flight))
            pos, L = in_flight.pop(k)
            assert completed[pos] == L  # one copy per phase
            completed[pos] += 1
        else:
            g = rng.randrange(GEMV_WARPS)
            i = done_items[g]
            if i >= items or i >= min(done_items) + n_op:
                continue  # finished, or its operand slot is not filled yet
            pc = GEMV_WARPS * i + g
            pos, L = pc % n_slots, pc // n_slots
            if lap_rule and lap[pos] != L:
                continue  # the slot does not show this lap yet
            if (completed[pos] & 1) == (L & 1):
                continue  # parity wait: the current phase has this lap's parity
            if completed[pos] != L + 1:
                wrong += 1  # the wait matched another lap's phase
                continue    # (the kernel would read that slot now and release it early)
            consumed[pos] += 1
            done_items[g] += 1
    assert min(done_items) >= items, "the schedule did not finish"
    return wrong


@pytest.mark.parametrize("n_slots", [21, 18])
def test_parity_alone_can_alias_at_the_kernels_ring_sizes(n_slots):
    """With four operand slots a gemv warp can be 24 + chunks ahead of another,
    more than the ring: some schedule lets a parity-only wait succeed early."""
    assert sum(simulate(n_slots, 4, 40, seed, lap_rule=False) for seed in range(40)) > 0


@pytest.mark.parametrize("n_slots", [21, 18, 16, 20])
def test_the_lap_rule_never_waits_on_another_lap(n_slots):
    for seed in range(60):
        assert simulate(n_slots, 4, 40, seed, lap_rule=True) == 0


def test_a_shallow_operand_ring_does_not_need_the_lap_rule():
    """At most one item of lead (two operand slots, the windows of 8 on the CUDA
    cores) stays within a 16-slot ring: the parity wait alone holds."""
    for seed in range(40):
        assert simulate(16, 2, 40, seed, lap_rule=False) == 0
