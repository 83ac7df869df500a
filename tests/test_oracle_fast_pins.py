"""Pins of the Fast NMS oracle to facts that do not come from the oracle.

Fast NMS ("YOLOv5后处理GPU移植实战", section 2.2) drops a box when any box of
higher priority and the same class overlaps it beyond the threshold, kept or
not.  Pinned by the hand-worked cases of tests/golden/fast_nms.json (exact
rational IoUs, including the three equal boxes of section 2.1), by an
exhaustive exact-rational check of that definition on tiny integer grids, and
by invariants relating it to greedy NMS.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "fast_nms.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_golden_cases(case):
    b = np.array(case["boxes"], np.float32)
    s = np.array(case["scores"], np.float32)
    assert oracle.nms_single(b, s, case["iou_thr"], fast=True).tolist() == case["keep"]
    assert oracle.nms_single(b, s, case["iou_thr"]).tolist() == case["greedy_keep"]


def _exact_iou(a, b):
    aa = (a[2] - a[0]) * (a[3] - a[1])
    ab = (b[2] - b[0]) * (b[3] - b[1])
    w = max(min(a[2], b[2]) - max(a[0], b[0]), 0)
    h = max(min(a[3], b[3]) - max(a[1], b[1]), 0)
    inter = w * h
    return Fraction(inter, aa + ab - inter)


@pytest.mark.parametrize("thr_s", ["0.3", "0.5", "0.7"])
def test_definition_on_tiny_grids(thr_s):
    """Integer boxes on a 0..8 grid (the binary32 decisions equal the exact
    rational ones there): the kept set is exactly the boxes with no earlier
    same-class box over the threshold, in priority order."""
    rng = np.random.default_rng(int(float(thr_s) * 1000) + 7)
    thr = Fraction(thr_s)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        x1 = rng.integers(0, 7, n)
        y1 = rng.integers(0, 7, n)
        x2 = x1 + rng.integers(1, 3, n)
        y2 = y1 + rng.integers(1, 3, n)
        boxes = [tuple(int(v) for v in r) for r in zip(x1, y1, x2, y2)]
        scores = [float(v) for v in rng.choice([0.25, 0.5, 0.75], n)]
        cls = [int(v) for v in rng.integers(0, 2, n)]
        order = sorted(range(n), key=lambda i: (-scores[i], i))
        expect = [j for r, j in enumerate(order)
                  if not any(cls[k] == cls[j] and _exact_iou(boxes[k], boxes[j]) > thr for k in order[:r])]
        keep, counts = oracle.nms(np.array(boxes, np.float32), np.array(scores, np.float32), float(thr_s),
                                  class_ids=np.array(cls, np.int32),
                                  batch_offsets=np.array([0, n], np.int64), fast=True)
        assert keep[: counts[0]].tolist() == expect


@pytest.mark.parametrize("seed", range(3))
def test_fast_is_a_subset_of_greedy_in_the_same_order(seed):
    """A box with no higher-priority box over the threshold is kept by greedy
    NMS too, so Fast NMS keeps a subsequence of the greedy answer."""
    rng = np.random.default_rng(seed)
    n = 300
    c = rng.uniform(0, 200, (n, 2))
    wh = rng.uniform(5, 40, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    for thr in (0.3, 0.5, 0.7):
        fast = oracle.nms_single(b, s, thr, fast=True).tolist()
        greedy = oracle.nms_single(b, s, thr).tolist()
        it = iter(greedy)
        assert all(x in it for x in fast)
        assert len(fast) <= len(greedy)


def test_chain_keeps_only_the_head():
    """a overlaps b, b overlaps c, a misses c: greedy keeps a and c, Fast NMS
    only a (c is dropped by b although b was dropped)."""
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1]], np.float32)
    s = np.array([0.9, 0.8, 0.7], np.float32)
    # IoU(a,b) = IoU(b,c) = 7/13 > 0.5, IoU(a,c) = 4/16 = 0.25
    assert oracle.nms_single(b, s, 0.5).tolist() == [0, 2]
    assert oracle.nms_single(b, s, 0.5, fast=True).tolist() == [0]


def test_no_chains_equals_greedy():
    """When every dropped box overlaps only kept boxes (pairs of equal boxes
    far apart), Fast NMS and greedy agree."""
    rng = np.random.default_rng(4)
    pts = rng.permutation(100)[:40]
    base = np.stack([pts * 20.0, np.zeros(40), pts * 20.0 + 10, np.full(40, 10.0)], 1)
    b = np.concatenate([base, base]).astype(np.float32)
    s = rng.uniform(0, 1, 80).astype(np.float32)
    assert oracle.nms_single(b, s, 0.5, fast=True).tolist() == oracle.nms_single(b, s, 0.5).tolist()


def test_max_out_and_prefilter():
    """max_out keeps a prefix; the pre-filter is strict."""
    rng = np.random.default_rng(9)
    n = 200
    c = rng.uniform(0, 100, (n, 2))
    wh = rng.uniform(5, 20, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    full = oracle.nms_single(b, s, 0.5, fast=True).tolist()
    assert oracle.nms_single(b, s, 0.5, fast=True, max_out=7).tolist() == full[:7]
    thr = float(np.median(s))
    filt = oracle.nms_single(b, s, 0.5, fast=True, score_thr=thr).tolist()
    assert all(s[i] > np.float32(thr) for i in filt)
