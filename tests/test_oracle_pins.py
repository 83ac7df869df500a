"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or plain mathematics
fix: hand-worked cases with exact rational IoUs (tests/golden), closed-form
special cases, library routines (numpy's stable argsort), an exhaustive
brute-force characterisation of the greedy result on tiny inputs with exact
rational arithmetic, and invariants.  A plausible slip in the oracle (a dropped
term, a wrong comparison, a flipped tie rule, fused multiply-add) fails at
least one of them.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- golden cases

def test_six_box_hand_worked():
    g = _golden("six_box.json")
    b = np.array(g["boxes"], np.float32)
    s = np.array(g["scores"], np.float32)
    for case in g["cases"]:
        got = oracle.nms_single(b, s, case["iou_thr"])
        assert got.tolist() == case["keep"], case


def test_six_box_exact_ious():
    g = _golden("six_box.json")
    b = np.array(g["boxes"], np.float32)
    expect = {(0, 1): 0.6, (0, 2): 1 / 3, (0, 5): 0.5, (1, 2): 0.6, (1, 5): 1 / 3,
              (2, 5): 0.2, (3, 4): 1.0}
    for (i, j), v in expect.items():
        assert oracle.iou(b[i], b[j]) == np.float32(v)


def test_iou_exactly_at_threshold_is_kept():
    g = _golden("at_threshold.json")
    for case in g["cases"]:
        got = oracle.nms_single(np.array(case["boxes"], np.float32),
                                np.array(case["scores"], np.float32), case["iou_thr"])
        assert got.tolist() == case["keep"], case


def test_equal_scores_priority():
    g = _golden("equal_scores.json")
    for case in g["cases"]:
        got = oracle.nms_single(np.array(case["boxes"], np.float32),
                                np.array(case["scores"], np.float32), case["iou_thr"])
        assert got.tolist() == case["keep"], case


def _bit_layout_boxes(g):
    n = g["n"]
    b = np.zeros((n, 4), np.float32)
    for k in range(n):
        b[k] = [20 * k, 100, 20 * k + 10, 110]
    b[3] = [0, 0, 10, 10]
    b[4] = [0, 0, 10, 9]
    b[5] = [200, 0, 210, 10]
    b[32] = [200, 0, 210, 9]
    b[34] = [200, 1, 210, 10]
    return b


def test_mask_bit_layout_matches_pages_example():
    g = _golden("bit_layout.json")
    b = _bit_layout_boxes(g)
    m = oracle.mask(b, g["iou_thr"])
    got = sorted((i, 64 * w + k) for i in range(m.shape[0]) for w in range(m.shape[1])
                 for k in range(64) if (int(m[i, w]) >> k) & 1)
    assert got == sorted(tuple(x) for x in g["expected_set_bits"])
    # The pages' 32-bit view: word 1 of row 5 is 0b101 (boxes 32 and 34).
    words32 = m.view(np.uint32)
    assert words32[5, 1] == 0b101
    assert words32[3, 0] == 1 << 4


# ------------------------------------------------------------- closed forms

def _random_boxes(rng, n, span=100.0, wmax=30.0):
    c = rng.uniform(0, span, (n, 2))
    wh = rng.uniform(1, wmax, (n, 2))
    return np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)


@pytest.mark.parametrize("seed", range(5))
def test_threshold_at_least_one_is_stable_argsort(seed):
    rng = np.random.default_rng(seed)
    n = 200
    b = _random_boxes(rng, n)
    s = (np.floor(rng.uniform(0, 1, n) * 16) / 16).astype(np.float32)  # many ties
    expect = np.argsort(-s.astype(np.float64), kind="stable")
    for thr in (1.0, 1.5, np.inf):
        assert oracle.nms_single(b, s, thr).tolist() == expect.tolist()


@pytest.mark.parametrize("seed", range(5))
def test_negative_threshold_keeps_only_top(seed):
    rng = np.random.default_rng(seed)
    b = _random_boxes(rng, 50)
    s = (np.floor(rng.uniform(0, 1, 50) * 4) / 4).astype(np.float32)
    top = int(np.argsort(-s.astype(np.float64), kind="stable")[0])
    assert oracle.nms_single(b, s, -0.01).tolist() == [top]


def test_disjoint_boxes_all_kept_in_score_order():
    rng = np.random.default_rng(7)
    n = 300
    x = np.arange(n, dtype=np.float32) * 10
    b = np.stack([x, np.zeros(n), x + 5, np.full(n, 5.0)], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    assert oracle.nms_single(b, s, 0.0).tolist() == np.argsort(-s, kind="stable").tolist()


def test_identical_boxes_keep_one():
    b = np.tile(np.array([[3, 4, 13, 24]], np.float32), (40, 1))
    s = np.linspace(0.1, 0.9, 40).astype(np.float32)
    assert oracle.nms_single(b, s, 0.99).tolist() == [39]


@pytest.mark.parametrize("seed", range(3))
def test_max_out_is_prefix(seed):
    rng = np.random.default_rng(seed)
    b = _random_boxes(rng, 400)
    s = rng.uniform(0, 1, 400).astype(np.float32)
    full = oracle.nms_single(b, s, 0.5)
    for k in (1, 5, 37, len(full) - 1, len(full), len(full) + 10):
        if k <= 0:
            continue
        assert oracle.nms_single(b, s, 0.5, max_out=k).tolist() == full[:k].tolist()


def test_score_order_special_values():
    s = np.array([np.nan, -0.0, 0.0, -np.inf, 1.0, 1.0, np.inf, np.nan, -1.0], np.float32)
    # +inf first; the two 1.0 by index; -0 and +0 tie (index order); -1; -inf; NaNs last.
    assert oracle.score_order(s).tolist() == [6, 4, 5, 1, 2, 8, 3, 0, 7]


def test_prefilter_is_strict():
    b = _random_boxes(np.random.default_rng(1), 6, span=1000.0)
    s = np.array([0.25, 0.5, 0.25, 0.2500001, 0.1, np.nan], np.float32)
    got = oracle.nms_single(b, s, 0.5, score_thr=0.25)
    assert sorted(got.tolist()) == [1, 3]


def test_nan_box_never_suppresses():
    b = np.array([[0, 0, 10, 10], [0, 0, 10, 10], [np.nan, 0, 10, 10]], np.float32)
    s = np.array([0.5, 0.4, 0.9], np.float32)
    assert oracle.nms_single(b, s, 0.5).tolist() == [2, 0]


def test_iou_is_bitwise_symmetric():
    rng = np.random.default_rng(3)
    a = _random_boxes(rng, 2000, wmax=60)
    c = _random_boxes(rng, 2000, wmax=60)
    for i in range(2000):
        x, y = oracle.iou(a[i], c[i]), oracle.iou(c[i], a[i])
        assert x.tobytes() == y.tobytes()


def test_iou_has_no_fused_multiply_add():
    """The canonical IoU rounds w*h to binary32 before the subtraction.  Find
    inputs where an FMA-contracted union (sum - w*h with one rounding) gives a
    different binary32 IoU, and check the oracle gives the two-rounding one.
    The reference values here come from numpy float32 arithmetic, whose
    operations are individually rounded (numpy never contracts)."""
    rng = np.random.default_rng(11)
    found = 0
    for _ in range(200000):
        a = rng.uniform(0, 1, 4).astype(np.float32)
        a[2:] += a[:2]
        b = (a + rng.uniform(-0.3, 0.3, 4).astype(np.float32)).astype(np.float32)
        b[2] = max(b[2], b[0] + np.float32(0.01))
        b[3] = max(b[3], b[1] + np.float32(0.01))
        f = np.float32
        aa = f(f(a[2] - a[0]) * f(a[3] - a[1]))
        ab = f(f(b[2] - b[0]) * f(b[3] - b[1]))
        w = max(f(min(a[2], b[2]) - max(a[0], b[0])), f(0))
        h = max(f(min(a[3], b[3]) - max(a[1], b[1])), f(0))
        inter = f(w * h)
        s = f(aa + ab)
        uni_two = f(s - inter)
        uni_fma = f(np.float64(s) - np.float64(w) * np.float64(h))  # one rounding
        if uni_two == uni_fma:
            continue
        two = f(inter / uni_two)
        fma = f(inter / uni_fma)
        if two == fma:
            continue
        assert oracle.iou(a, b) == two
        found += 1
        if found >= 20:
            break
    assert found >= 5


# ------------------------------------------- exhaustive brute force, tiny N

def _exact_iou(a, b):
    aa = (a[2] - a[0]) * (a[3] - a[1])
    ab = (b[2] - b[0]) * (b[3] - b[1])
    w = max(min(a[2], b[2]) - max(a[0], b[0]), 0)
    h = max(min(a[3], b[3]) - max(a[1], b[1]), 0)
    inter = w * h
    return Fraction(inter, aa + ab - inter)


def _characterised_keep(boxes, scores, cls, thr):
    """The unique subset K such that no member is suppressed by an earlier
    member and every non-member is suppressed by an earlier member (earlier =
    higher score, ties to the lower index; suppression needs the same class and
    an exact rational IoU strictly above the threshold).  Found by enumerating
    every subset."""
    n = len(boxes)
    order = sorted(range(n), key=lambda i: (-scores[i], i))
    rank = {i: r for r, i in enumerate(order)}
    sup = [[False] * n for _ in range(n)]
    for k in range(n):
        for j in range(n):
            if rank[k] < rank[j] and cls[k] == cls[j] and _exact_iou(boxes[k], boxes[j]) > thr:
                sup[k][j] = True
    sols = []
    for mask in range(1 << n):
        K = [i for i in range(n) if mask >> i & 1]
        ok = all(not sup[k][j] for k in K for j in K)
        ok = ok and all(any(sup[k][j] for k in K) for j in range(n) if not mask >> j & 1)
        if ok:
            sols.append(sorted(K, key=lambda i: rank[i]))
    assert len(sols) == 1  # the greedy result is unique
    return sols[0]


@pytest.mark.parametrize("thr_s", ["0.3", "0.45", "0.5", "0.7"])
def test_brute_force_tiny_grid(thr_s):
    """Integer boxes on a 0..8 grid: every binary32 step of the IoU is exact
    except the final division, and a ratio with denominator <= 128 is either
    equal to the threshold or at least 1/2560 away from it, so the binary32
    decision equals the exact rational one."""
    rng = np.random.default_rng(int(float(thr_s) * 100))
    thr = Fraction(thr_s)
    for trial in range(150):
        n = int(rng.integers(1, 9))
        x1 = rng.integers(0, 7, n)
        y1 = rng.integers(0, 7, n)
        x2 = x1 + rng.integers(1, 3, n)
        y2 = y1 + rng.integers(1, 3, n)
        boxes = [tuple(int(v) for v in r) for r in zip(x1, y1, x2, y2)]
        scores = [float(v) for v in rng.choice([0.25, 0.5, 0.75], n)]
        cls = [int(v) for v in rng.integers(0, 2, n)]
        expect = _characterised_keep(boxes, scores, cls, thr)
        b = np.array(boxes, np.float32)
        s = np.array(scores, np.float32)
        c = np.array(cls, np.int32)
        keep, counts = oracle.nms(b, s, float(thr_s), class_ids=c,
                                  batch_offsets=np.array([0, n], np.int64))
        assert keep[: counts[0]].tolist() == expect, (boxes, scores, cls)


# ------------------------------------------------------- batched = composition

@pytest.mark.parametrize("seed", range(3))
def test_batched_equals_per_class_runs_merged(seed):
    rng = np.random.default_rng(100 + seed)
    B, C, per = 4, 5, 120
    n = B * per
    b = _random_boxes(rng, n, span=60.0, wmax=25.0)
    s = (np.floor(rng.uniform(0, 1, n) * 64) / 64).astype(np.float32)
    cls = rng.integers(0, C, n).astype(np.int32)
    off = np.arange(0, n + 1, per, dtype=np.int64)
    for max_out, score_thr in ((0, None), (17, 0.3), (1000, 0.1)):
        keep, counts = oracle.nms(b, s, 0.45, class_ids=cls, batch_offsets=off,
                                  score_thr=score_thr, max_out=max_out)
        for img in range(B):
            lo, hi = off[img], off[img + 1]
            merged = []
            for c in range(C):
                idx = np.array([i for i in range(lo, hi) if cls[i] == c], np.int64)
                if len(idx) == 0:
                    continue
                sub = oracle.nms_single(b[idx], s[idx], 0.45, score_thr=score_thr)
                merged.extend(int(idx[k]) for k in sub)
            merged.sort(key=lambda i: (-float(s[i]), i))
            if max_out > 0:
                merged = merged[:max_out]
            base = img * max_out if max_out > 0 else lo
            assert keep[base: base + counts[img]].tolist() == merged
