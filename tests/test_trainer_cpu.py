"""Host logic of the training loop: the learning-rate schedule and the reselection cadence."""
import math

import pytest

from sparse_moe_fine_gb300.trainer import cosine_lr, reselect_due


def test_cosine_schedule_endpoints_and_shape():
    peak, total = 2e-4, 100
    assert cosine_lr(0, total, peak) == pytest.approx(peak)
    assert cosine_lr(total, total, peak) == pytest.approx(0.0, abs=1e-15)
    assert cosine_lr(total // 2, total, peak) == pytest.approx(peak / 2)
    # monotone non-increasing after warm-up
    vals = [cosine_lr(s, total, peak) for s in range(1, total + 1)]
    assert all(a >= b - 1e-18 for a, b in zip(vals, vals[1:]))
    # past the end it stays at the floor
    assert cosine_lr(total + 10, total, peak, floor=1e-6) == pytest.approx(1e-6)


def test_cosine_schedule_with_warmup():
    peak, total, warm = 1.0, 110, 10
    assert cosine_lr(1, total, peak, warm) == pytest.approx(0.1)
    assert cosine_lr(10, total, peak, warm) == pytest.approx(1.0)
    assert cosine_lr(60, total, peak, warm) == pytest.approx(0.5)
    assert cosine_lr(35, total, peak, warm) == pytest.approx(0.5 * (1 + math.cos(math.pi / 4)))


def test_reselect_cadence():
    assert [s for s in range(1, 201) if reselect_due(s, 50)] == [50, 100, 150, 200]
    assert not any(reselect_due(s, 0) for s in range(1, 10))
