"""The multi-core CPU baseline (oracle/cpu_baseline.c, OpenMP bitmask and
resolve) that bench.py times beside the GPU path: it must give exactly the
oracle's keep lists and counts.  Pinned to the hand-worked cases of
tests/golden ("NMS CUDA代码学习", intro and section 算法与数据流; the
at-threshold containments; "YOLOv5后处理GPU移植实战" section 2.1's equal
scores) and to the oracle on the five benchmark workloads (seed 0) and on
tiny grids with ties, NaN scores, degenerate boxes, classes and images."""
import json
import os

import numpy as np
import pytest

import oracle
from greedy_iou_nms_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _single(b, s, thr, **kw):
    keep, counts = oracle.cpu_baseline_nms(np.asarray(b, np.float32), np.asarray(s, np.float32), thr, **kw)
    return keep[: counts[0]].tolist()


def test_threads_reported():
    assert oracle.cpu_baseline_threads() >= 1


def test_six_box_golden():
    g = _golden("six_box.json")
    for c in g["cases"]:
        assert _single(g["boxes"], g["scores"], c["iou_thr"]) == c["keep"], c["why"]


def test_at_threshold_golden():
    g = _golden("at_threshold.json")
    for c in g["cases"]:
        assert _single(c["boxes"], c["scores"], c["iou_thr"]) == c["keep"]


def test_equal_scores_golden():
    g = _golden("equal_scores.json")
    for c in g["cases"]:
        assert _single(c["boxes"], c["scores"], c["iou_thr"]) == c["keep"]


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_workloads_match_oracle(name):
    wl = W.make(name, 0)
    kw = dict(class_ids=wl.class_ids, batch_offsets=wl.batch_offsets, score_thr=wl.score_thr, max_out=wl.max_out)
    got_k, got_c = oracle.cpu_baseline_nms(wl.boxes, wl.scores, wl.iou_thr, **kw)
    exp_k, exp_c = oracle.nms(wl.boxes, wl.scores, wl.iou_thr, **kw)
    assert got_c.tolist() == exp_c.tolist()
    assert got_k.tolist() == exp_k.tolist()


@pytest.mark.parametrize("seed", range(40))
def test_tiny_grids_match_oracle(seed):
    """Integer boxes on an 8 x 8 grid with three score levels: many exact
    ties and IoUs exactly at the threshold; NaN and -0 scores, zero-area and
    inverted boxes; two images of up to three classes, with and without a
    pre-filter and max_out."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    xy = rng.integers(0, 8, (n, 2))
    wh = rng.integers(-1, 5, (n, 2))
    b = np.concatenate([xy, xy + wh], 1).astype(np.float32)
    s = rng.choice([0.25, 0.5, 0.75], n).astype(np.float32)
    if n > 3:
        s[1] = np.nan
        s[2] = -0.0
    cls = rng.integers(0, 3, n).astype(np.int32)
    cut = int(rng.integers(0, n + 1))
    off = np.array([0, cut, n], np.int64)
    for thr in (0.0, 1 / 3, 0.5, 0.7):
        for kw in ({}, {"max_out": 3}, {"score_thr": 0.3}):
            assert oracle.cpu_baseline_nms(b, s, thr, **kw)[0].tolist() == oracle.nms(b, s, thr, **kw)[0].tolist()
            kb = dict(kw, class_ids=cls, batch_offsets=off)
            gk, gc = oracle.cpu_baseline_nms(b, s, thr, **kb)
            ek, ec = oracle.nms(b, s, thr, **kb)
            assert gc.tolist() == ec.tolist() and gk.tolist() == ek.tolist()
