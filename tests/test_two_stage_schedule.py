"""The two-stage launch's item lists (host logic, no GPU): every item placed exactly once, and
the lists can always be run to the end. A first-stage item never waits; a down item waits
until every first-stage item of its band has run. Running the lists in any interleaving, a
list whose next item is ready always exists until all are done: no circular wait, with every
pair resident."""
import pytest

import feed_forward_gemm_gb300 as fm

# (bands, first-stage N tiles, down N tiles, K steps per first-stage and down tile)
SHAPES = [(32, 24, 3, 12, 48),        # GPT-2-small GeGLU block, 8192 tokens
          (32, 12, 3, 12, 48),        # 768/3072 MLP
          (16, 16, 16, 64, 64),       # 4096-wide MLP, 4096 tokens
          (2, 24, 3, 12, 48),         # 512 tokens
          (1, 1, 1, 1, 1),
          (64, 16, 16, 16, 64),       # 16384 tokens
          (7, 9, 5, 3, 40)]


def check_schedule(num_m, num_n1, num_n2, pairs, start, items):
    n1, n2 = num_m * num_n1, num_m * num_n2
    assert sorted(items) == list(range(n1 + n2))          # each item exactly once
    assert start[0] == 0 and start[-1] == len(items)
    assert all(a <= b for a, b in zip(start, start[1:]))
    queues = [items[start[p]:start[p + 1]] for p in range(pairs)]
    left = [num_n1] * num_m                                # first-stage items still to run
    pos = [0] * pairs
    done = 0
    while done < n1 + n2:
        progressed = False
        for p in range(pairs):
            while pos[p] < len(queues[p]):
                t = queues[p][pos[p]]
                if t < n1:
                    left[t // num_n1] -= 1
                elif left[(t - n1) // num_n2]:
                    break                                   # waits for its band
                pos[p] += 1
                done += 1
                progressed = True
        assert progressed, "every list waits on a band no other list can complete"


@pytest.mark.parametrize("num_m,num_n1,num_n2,kb1,kb2", SHAPES)
@pytest.mark.parametrize("pairs", [76, 36, 5, 1])
def test_two_stage_lists_cover_every_item_and_never_deadlock(num_m, num_n1, num_n2, kb1, kb2,
                                                             pairs):
    start, items = fm.fmlp_test_two_stage_schedule(num_m, num_n1, num_n2, kb1, kb2, pairs)
    check_schedule(num_m, num_n1, num_n2, pairs, start, items)


def test_the_checker_catches_a_circular_wait():
    """A planted bad schedule: each list holds a down item ahead of the first-stage item the
    other list's down item needs."""
    # 2 bands, 1 first-stage tile each (items 0, 1), 1 down tile each (items 2, 3)
    start, items = [0, 2, 4], [2, 1, 3, 0]
    with pytest.raises(AssertionError):
        check_schedule(2, 1, 1, 2, start, items)


def test_schedule_shapes_out_of_range_are_refused():
    with pytest.raises(fm.FmlpError) as e:
        fm.fmlp_test_two_stage_schedule(65, 24, 3, 12, 48, 76)
    assert e.value.status == fm.FMLP_ERR_SHAPE
    with pytest.raises(fm.FmlpError):
        fm.fmlp_test_two_stage_schedule(32, 24, 3, 12, 48, 129)      # more pairs than lists
    with pytest.raises(fm.FmlpError):
        fm.fmlp_test_two_stage_schedule(64, 64, 32, 12, 48, 76)     # more than 2048 items
