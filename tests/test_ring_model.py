"""A model of the kernel's pipeline protocol, run under random schedules.

The model follows the kernel's barriers one for one:
  - ring of `slots = stages + release` buffers; `full[s]` completes when the
    producer's TMA data for a step has landed, `empty[s]` when the slot is
    handed back;
  - the producer waits on `empty` (parity of the previous use) before loading
    step j into slot j % slots;
  - the MMA thread waits on `full`, issues its MMAs (asynchronous: they finish
    later, in issue order), and commits step i's completion to the `empty`
    barrier of step i - release;
  - two TMEM accumulators: the MMA waits on `tmem_empty[t % 2]` before tile t
    overwrites it and commits `tmem_full` after its last step; the epilogue
    reads it asynchronously and arrives on `tmem_empty`.

Checked: no slot is overwritten while an MMA that reads it has not finished,
no accumulator is overwritten while the epilogue still reads it, every run
finishes (no deadlock), and the first reuse of slot 0 matches the pages'
example for max_concurrent_steps / delay_release ("JAX Pallas Mosaic GPU
快速上手", section "深入emit_pipeline的关键参数": with (2, 1) the buffer of
iteration 0 is reused at iteration 3, with plain double buffering at 2).
A variant that releases on MMA *issue* instead of completion (the race the
pages warn of when delay_release is left out) is shown to be caught.
"""
import random

import pytest


class Barrier:
    """mbarrier phases as a completion count; wait(parity) as the kernel does."""

    def __init__(self):
        self.completed = 0

    def arrive(self):
        self.completed += 1

    def passed(self, parity):
        # try_wait.parity(P) succeeds once the phase with parity P completed:
        # the current (incomplete) phase index is `completed`.
        return (self.completed & 1) != parity


def simulate(stages, release, tiles, k_steps, seed, release_on_issue=False, record=None):
    rng = random.Random(seed)
    slots = stages + release
    full = [Barrier() for _ in range(slots)]
    empty = [Barrier() for _ in range(slots)]
    tfull = [Barrier(), Barrier()]
    tempty = [Barrier(), Barrier()]
    total = tiles * k_steps

    slot_data = [None] * slots          # step whose data the slot holds
    pending_reads = [0] * slots         # MMAs issued on the slot, not finished
    inflight_loads = []                 # (slot, step) landing later
    mma_queue = []                      # issued MMAs in order: (step, slot)
    commits = []                        # (after_step, barrier) arrive once MMAs <= after_step done
    done_mma = -1                       # last finished MMA step
    acc_owner = [None, None]            # tile whose partial sums the accumulator holds
    acc_reading = [False, False]        # epilogue still reading
    epi_queue = []                      # tiles ready for the epilogue, in order

    prod = {"j": 0}
    mma = {"i": 0, "tile_open": False}
    epi = {"t": 0, "reading": None}
    first_reuse = {}

    def producer_step():
        j = prod["j"]
        if j >= total:
            return False
        s, use = j % slots, j // slots
        if not empty[s].passed((use & 1) ^ 1):
            return False
        # safety: the previous content of this slot is no longer being read
        assert pending_reads[s] == 0, f"slot {s} overwritten at step {j} while an MMA reads it"
        if slot_data[s] is not None and s == 0 and 0 not in first_reuse:
            first_reuse[0] = j
        inflight_loads.append((s, j))
        prod["j"] += 1
        return True

    def load_lands():
        if not inflight_loads:
            return False
        s, j = inflight_loads.pop(rng.randrange(len(inflight_loads)))
        slot_data[s] = j
        full[s].arrive()
        return True

    def mma_issue():
        i = mma["i"]
        if i >= total:
            return False
        t, kb = divmod(i, k_steps)
        acc = t & 1
        if kb == 0 and not mma["tile_open"]:
            if not tempty[acc].passed(((t >> 1) & 1) ^ 1):
                return False
            assert not acc_reading[acc], f"accumulator {acc} overwritten while the epilogue reads tile {acc_owner[acc]}"
            acc_owner[acc] = t
            mma["tile_open"] = True
        s, use = i % slots, i // slots
        if not full[s].passed(use & 1):
            return False
        assert slot_data[s] == i, f"MMA step {i} found step {slot_data[s]} in slot {s}"
        pending_reads[s] += 1
        mma_queue.append((i, s))
        if i >= release:
            rs = (i - release) % slots
            if release_on_issue:
                empty[rs].arrive()      # wrong: hands the buffer back before the MMA ran
            else:
                commits.append((i, empty[rs]))
        if kb == k_steps - 1:
            commits.append((i, ("tfull", t)))
            mma["tile_open"] = False
        mma["i"] += 1
        return True

    def mma_finish():
        nonlocal done_mma
        if not mma_queue:
            return False
        i, s = mma_queue.pop(0)
        pending_reads[s] -= 1
        done_mma = i
        while commits and commits[0][0] <= done_mma:
            _, target = commits.pop(0)
            if isinstance(target, tuple):
                t = target[1]
                epi_queue.append(t)
                tfull[t & 1].arrive()
            else:
                target.arrive()
        return True

    def epilogue_start():
        t = epi["t"]
        if epi["reading"] is not None or t >= tiles:
            return False
        acc = t & 1
        if not tfull[acc].passed((t >> 1) & 1):
            return False
        assert acc_owner[acc] == t
        acc_reading[acc] = True
        epi["reading"] = t
        return True

    def epilogue_finish():
        t = epi["reading"]
        if t is None:
            return False
        acc_reading[t & 1] = False
        tempty[t & 1].arrive()
        epi["reading"] = None
        epi["t"] += 1
        return True

    actions = [producer_step, load_lands, mma_issue, mma_finish, epilogue_start, epilogue_finish]
    for _ in range(100 * (total + tiles) + 1000):
        if epi["t"] == tiles:
            break
        order = actions[:]
        rng.shuffle(order)
        if not any(a() for a in order):
            raise RuntimeError("deadlock")
    else:
        raise RuntimeError("did not finish")
    if record is not None:
        record.update(first_reuse)
    return True


CONFIGS = [(s, r) for s in range(1, 7) for r in range(0, 3) if r < s]


@pytest.mark.parametrize("stages,release", CONFIGS)
def test_protocol_is_race_free_and_finishes(stages, release):
    for seed in range(40):
        simulate(stages, release, tiles=5, k_steps=7, seed=seed)
    simulate(stages, release, tiles=9, k_steps=1, seed=123)  # one step per tile


def test_pages_example_first_reuse():
    """(max_concurrent_steps=2, delay_release=1): buffer of iteration 0 is
    reused at iteration 3; (2, 0): at iteration 2."""
    rec = {}
    simulate(2, 1, tiles=1, k_steps=8, seed=0, record=rec)
    assert rec[0] == 3
    rec = {}
    simulate(2, 0, tiles=1, k_steps=8, seed=0, record=rec)
    assert rec[0] == 2


def test_release_on_issue_is_a_race():
    """Handing a buffer back when its MMA is issued rather than when it has
    finished lets the producer overwrite data still being read."""
    caught = 0
    for seed in range(200):
        try:
            simulate(2, 0, tiles=3, k_steps=6, seed=seed, release_on_issue=True)
        except AssertionError:
            caught += 1
    assert caught > 0


def test_no_load_in_flight_deadlocks():
    """With no load allowed in flight (stages = 0, so slots = release) the step
    that would release a buffer needs data that has no buffer to land in: the
    model deadlocks.  The planner is stricter still and, as emit_pipeline
    does, refuses any stages <= release."""
    with pytest.raises(RuntimeError, match="deadlock"):
        simulate(0, 1, tiles=1, k_steps=4, seed=0)
