"""Pins of the lane-candidate NMS oracle ("nms_kernel.cu 파일 분석 -2": 77
values per lane candidate, visited in score order, a symmetric comparison by
absolute values against a similarity threshold; the page stops before the
comparison, and the readings are in nms_oracle.c): closed forms of the
distance (a constant offset, rows outside the common span ignored, no common
rows), the row span's parsing, the strict threshold, a hand-worked chain, the
tie rule, and an exact-rational brute force of the greedy definition on
integer lanes."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def lane(x, start=0, length=72):
    p = np.zeros(77, np.float32)
    p[2] = start
    p[4] = length
    p[5:] = np.broadcast_to(np.asarray(x, np.float32), (72,))
    p[3] = p[5 + int(max(0, min(71, np.floor(start))))] if np.isfinite(start) else 0
    return p


def test_constant_offset_is_the_distance():
    r = np.arange(72, dtype=np.float32)
    for d in (0.0, 0.5, 5.0, 37.25):
        assert oracle.lane_distance(lane(100 + r), lane(100 + r + d)) == np.float32(d)
        assert oracle.lane_distance(lane(100 + r + d), lane(100 + r)) == np.float32(d)  # symmetric


def test_only_common_rows_count():
    """a covers rows [0, 40), b rows [20, 72): only rows 20..39 count; b's
    values above row 20 are far away and must not matter."""
    r = np.arange(72, dtype=np.float32)
    xb = 100 + r + 3
    xb[:20] = 1e6
    a = lane(100 + r, 0, 40)
    b = lane(xb, 20, 52)
    assert oracle.lane_distance(a, b) == np.float32(3)
    # mean of unequal offsets: rows 20..39 differ by 1 (10 rows) and 4 (10 rows): 50 / 20 = 2.5
    xc = 100 + r
    xc[20:30] += 1
    xc[30:40] += 4
    assert oracle.lane_distance(a, lane(xc, 20, 52)) == np.float32(2.5)


def test_no_common_rows_never_suppress():
    a = lane(np.full(72, 50.0), 0, 30)
    b = lane(np.full(72, 50.0), 30, 42)
    assert oracle.lane_distance(a, b) == np.float32(np.inf)
    props = np.stack([a, b])
    assert oracle.lane_nms(props, np.array([0.9, 0.8], np.float32), 1e30).tolist() == [0, 1]


def test_row_span_parsing():
    """Rows are [floor(start), floor(start) + floor(length)) clipped to
    [0, 72): start 10.7, length 5.9 is rows 10..14; start -3, length 10 is
    rows 0..6; start 70, length 9 is rows 70, 71; NaN or infinite values give
    no rows."""
    r = np.arange(72, dtype=np.float32)
    base = lane(r * 0)  # all rows, x = 0
    x = np.zeros(72, np.float32)
    x[10:15] = 8  # only rows 10..14 differ by 8
    x[15:] = 1000
    x[:10] = 1000
    assert oracle.lane_distance(base, lane(x, 10.7, 5.9)) == np.float32(8)
    y = np.full(72, 1000, np.float32)
    y[:7] = 2
    assert oracle.lane_distance(base, lane(y, -3, 10)) == np.float32(2)
    z = np.full(72, 1000, np.float32)
    z[70:] = 6
    assert oracle.lane_distance(base, lane(z, 70, 9)) == np.float32(6)
    for bad in (np.nan, np.inf, -np.inf, 3e6):
        p = lane(r * 0)
        p[2] = bad
        assert oracle.lane_distance(base, p) == np.float32(np.inf)
        q = lane(r * 0)
        q[4] = bad
        assert oracle.lane_distance(base, q) == np.float32(np.inf)


def test_threshold_is_strict():
    r = np.arange(72, dtype=np.float32)
    props = np.stack([lane(r), lane(r + 5)])
    s = np.array([0.9, 0.8], np.float32)
    assert oracle.lane_nms(props, s, 5.0).tolist() == [0, 1]  # distance == thr keeps
    assert oracle.lane_nms(props, s, float(np.nextafter(np.float32(5), np.float32(6)))).tolist() == [0]


def test_chain_hand_worked():
    """A (0.9), B (0.8), C (0.7): d(A,B) = 6, d(B,C) = 6, d(A,C) = 12 at
    threshold 10: B goes with A; C is 6 from the dropped B only and stays."""
    r = np.arange(72, dtype=np.float32)
    props = np.stack([lane(200 + r), lane(206 + r), lane(212 + r)])
    s = np.array([0.9, 0.8, 0.7], np.float32)
    assert oracle.lane_nms(props, s, 10.0).tolist() == [0, 2]
    assert oracle.lane_nms(props, s, 13.0).tolist() == [0]
    assert oracle.lane_nms(props, s, 6.0).tolist() == [0, 1, 2]
    assert oracle.lane_nms(props, s, 10.0, max_out=1).tolist() == [0]


def test_equal_scores_lower_index_first():
    r = np.arange(72, dtype=np.float32)
    props = np.stack([lane(300 + r), lane(100 + r), lane(101 + r), lane(100.5 + r)])
    s = np.full(4, 0.5, np.float32)
    assert oracle.lane_nms(props, s, 2.0).tolist() == [0, 1]


def _exact_greedy(xs, spans, scores, thr):
    """The greedy definition with exact rationals: visit by descending score
    (ties to the lower index), drop a lane whose mean |dx| over the common
    rows with a kept lane is below thr."""
    order = sorted(range(len(scores)), key=lambda i: (-scores[i], i))
    kept = []
    for i in order:
        ok = True
        for k in kept:
            lo, hi = max(spans[i][0], spans[k][0]), min(spans[i][1], spans[k][1])
            if hi <= lo:
                continue
            d = Fraction(sum(abs(int(xs[i][r]) - int(xs[k][r])) for r in range(lo, hi)), hi - lo)
            if d < thr:
                ok = False
                break
        if ok:
            kept.append(i)
    return kept


@pytest.mark.parametrize("seed", range(60))
def test_brute_force_integer_lanes(seed):
    """Integer x's (so the binary32 sums are exact) and half-integer
    thresholds (so the binary32 mean lies on the same side of the threshold
    as the exact one: a mean of k <= 72 integers differs from m + 1/2 by at
    least 1/144, far more than an ulp)."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 14))
    base = rng.integers(0, 60, n)
    xs = base[:, None] + rng.integers(-3, 4, (n, 72))
    starts = rng.integers(0, 60, n)
    lens = rng.integers(1, 40, n)
    spans = [(int(a), int(min(72, a + b))) for a, b in zip(starts, lens)]
    scores = rng.choice([0.25, 0.5, 0.75], n).astype(np.float32)
    props = np.stack([lane(xs[i].astype(np.float32), starts[i], lens[i]) for i in range(n)])
    for thr in (0.5, 2.5, 7.5, 20.5):
        assert oracle.lane_nms(props, scores, thr).tolist() == _exact_greedy(xs, spans, scores.tolist(),
                                                                             Fraction(thr))
