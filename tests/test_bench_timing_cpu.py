"""Host logic of the benchmark's timing hygiene: a sub-benchmark whose step
touches less memory than L2 cycles over enough disjoint buffer copies that
the memory touched between two uses of one copy is about three times L2, so
no step finds the previous step's data there."""
import bench


def test_rotation_covers_three_times_l2():
    for step_bytes in (10**6, 34 * 10**6, 74 * 10**6, 135 * 10**6):
        n = bench.rotation(step_bytes)
        assert n * step_bytes >= 3 * bench.L2_BYTES or n == 8
        assert (n - 1) * step_bytes < 3 * bench.L2_BYTES  # no more copies than needed


def test_rotation_is_one_for_steps_larger_than_three_l2():
    assert bench.rotation(3 * bench.L2_BYTES) == 1
    assert bench.rotation(10**10) == 1


def test_rotation_respects_the_cap():
    assert bench.rotation(1, most=5) == 5
    assert bench.rotation(0) == 8


def test_cycling_runs_each_copy_in_turn():
    seen = []
    step = bench.cycling([lambda i=i: seen.append(i) for i in range(3)])
    for _ in range(7):
        step()
    assert seen == [0, 1, 2, 0, 1, 2, 0]
