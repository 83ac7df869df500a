"""Pins of the Matrix NMS oracle ("Fastest Matrix NMS in the West (Part 2)",
section "What do we need to compute?" and section "Optimization 4") to facts
that do not come from the oracle: closed forms (disjoint boxes, a pair at an
exact IoU, identical boxes), a hand-worked three-box chain with exact rational
IoUs, the page's own restatement of the drop rule (a box goes when some
father's candidate decayed score is below the threshold), and invariants."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def test_disjoint_boxes_keep_their_scores():
    b = np.array([[0, 0, 1, 1], [5, 5, 6, 6], [10, 0, 11, 1], [0, 10, 1, 11]], np.float32)
    s = np.array([0.9, 0.2, 0.6, 0.4], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.3)
    assert keep.tolist() == [0, 2, 3]
    assert fs.tolist() == [np.float32(0.9), np.float32(0.6), np.float32(0.4)]
    # the threshold is inclusive for keeping: final score == t stays
    keep, _ = oracle.matrix_nms(b, s, np.float32(0.4))
    assert keep.tolist() == [0, 2, 3]


@pytest.mark.parametrize("sigma", [0.5, 2.0])
def test_pair_at_exact_iou(sigma):
    """IoU([0,0,4,4], [0,0,4,2]) = 8/16 = 0.5 exactly: the second box decays by
    exp(-0.25/sigma); the first (no father) keeps its score."""
    b = np.array([[0, 0, 4, 4], [0, 0, 4, 2]], np.float32)
    s = np.array([0.9, 0.8], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, sigma=sigma)
    assert keep.tolist() == [0, 1]
    assert fs[0] == np.float32(0.9)
    assert fs[1] == np.float32(float(np.float32(0.8)) * math.exp(-0.25 / float(np.float32(sigma))))


def test_identical_boxes():
    """k identical boxes: the first keeps its score; every other one decays by
    exp(-1/sigma) (its top father overlaps it at 1 and has no father itself;
    the other fathers overlap at 1 with their own maximum 1, decay 1)."""
    k = 6
    b = np.tile(np.array([[3, 3, 9, 7]], np.float32), (k, 1))
    s = np.linspace(0.9, 0.4, k).astype(np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0)
    assert keep.tolist() == list(range(k))
    assert fs[0] == s[0]
    for j in range(1, k):
        assert fs[j] == np.float32(float(s[j]) * math.exp(-2.0))


def test_chain_hand_worked():
    """a=[0,0,10,1], b=[3,0,13,1], c=[6,0,16,1]: IoU(a,b) = IoU(b,c) = 7/13,
    IoU(a,c) = 1/4.  O_max: a 0, b 7/13, c 7/13.  Decays (sigma 1/2): b gets
    exp(-2 (7/13)^2) from a; c gets min(exp(-2 (1/4)^2) from a, exp(0) from b)."""
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1]], np.float32)
    s = np.array([0.9, 0.8, 0.7], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0)
    r = float(Fraction(7, 13))
    exp_b = float(np.float32(0.8)) * math.exp(-2 * r * r)
    exp_c = float(np.float32(0.7)) * math.exp(-2 * 0.25 * 0.25)
    assert keep.tolist() == [0, 1, 2]
    assert abs(fs[1] - exp_b) <= 2e-7 and abs(fs[2] - exp_c) <= 2e-7  # binary32 IoUs of 7/13
    assert fs[0] == np.float32(0.9)
    # final scores: a 0.9, b ~0.448, c ~0.618; a threshold between b and c
    # drops b only, one between c and a keeps a only
    assert exp_b < exp_c < 0.9
    assert oracle.matrix_nms(b, s, (exp_b + exp_c) / 2)[0].tolist() == [0, 2]
    assert oracle.matrix_nms(b, s, (exp_c + 0.9) / 2)[0].tolist() == [0]


def _clustered(rng, n):
    c = rng.uniform(0, 200, (max(n // 6, 1), 2))[rng.integers(0, max(n // 6, 1), n)] + rng.normal(0, 5, (n, 2))
    wh = rng.uniform(8, 40, (n, 2))
    return np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32), rng.uniform(0, 1, n).astype(np.float32)


@pytest.mark.parametrize("seed", range(3))
def test_pages_exists_restatement(seed):
    """Section "Optimization 4": since scores are non-negative, s_j min_i d_ij < t
    exactly when some father i has s_j d_ij < t.  The drop decisions of the
    oracle (a minimum, then one comparison) equal that existence form,
    evaluated here pair by pair from the binary32 IoUs."""
    rng = np.random.default_rng(seed)
    n = 60
    b, s = _clustered(rng, n)
    t = 0.25
    keep, _ = oracle.matrix_nms(b, s, t)
    order = oracle.score_order(s)
    O = np.zeros((n, n))
    for p in range(n):
        for q in range(p):
            O[q, p] = float(oracle.iou(b[order[q]], b[order[p]]))
    omax = np.array([max([O[q, p] for q in range(p)], default=0.0) for p in range(n)])
    kept = []
    for p in range(n):
        sj = float(s[order[p]])
        drop = sj < t if p == 0 else any(sj * math.exp((omax[q] ** 2 - O[q, p] ** 2) / 0.5) < t for q in range(p))
        if not drop:
            kept.append(int(order[p]))
    assert keep.tolist() == kept


@pytest.mark.parametrize("seed", range(2))
def test_invariants(seed):
    rng = np.random.default_rng(10 + seed)
    b, s = _clustered(rng, 200)
    # a very wide Gaussian decays nothing
    keep, fs = oracle.matrix_nms(b, s, 0.0, sigma=1e7)
    order = oracle.score_order(s)
    assert keep.tolist() == order.tolist()
    assert np.allclose(fs, s[order], rtol=1e-6)
    # decayed scores never exceed the scores; a higher threshold keeps a subset
    keep, fs = oracle.matrix_nms(b, s, 0.0)
    assert np.all(fs <= s[keep])
    k2, _ = oracle.matrix_nms(b, s, 0.3)
    assert set(k2.tolist()) <= set(keep.tolist())
    assert [x for x in keep.tolist() if x in set(k2.tolist())] == k2.tolist()
    # max_out keeps a prefix; the pre-filter is strict
    k3, f3 = oracle.matrix_nms(b, s, 0.1, max_out=9)
    kf, ff = oracle.matrix_nms(b, s, 0.1)
    assert k3.tolist() == kf.tolist()[:9] and f3.tolist() == ff.tolist()[:9]
    kp, _ = oracle.matrix_nms(b, s, 0.0, score_thr=0.5)
    assert all(s[i] > np.float32(0.5) for i in kp)


# ------------------------------------------------------------- linear decay
#
# The page names a linear decay without printing it; the reading is
# d_ij = (1 - O_ij) / (1 - O_max,i), the linear kernel with the same
# compensation.  Pins by closed forms and hand-worked rationals.

def test_linear_disjoint_and_exact_pair():
    b = np.array([[0, 0, 1, 1], [5, 5, 6, 6], [10, 0, 11, 1]], np.float32)
    s = np.array([0.9, 0.2, 0.6], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, decay="linear")
    assert keep.tolist() == [0, 2, 1] and fs.tolist() == [np.float32(0.9), np.float32(0.6), np.float32(0.2)]
    # IoU 1/2 exactly, father without fathers: decay (1 - 1/2) / 1
    b = np.array([[0, 0, 4, 4], [0, 0, 4, 2]], np.float32)
    s = np.array([0.9, 0.8], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, decay="linear")
    assert keep.tolist() == [0, 1]
    assert fs[1] == np.float32(float(np.float32(0.8)) * 0.5)
    assert oracle.matrix_nms(b, s, np.float32(0.8) * np.float32(0.5), decay="linear")[0].tolist() == [0, 1]
    assert oracle.matrix_nms(b, s, np.nextafter(np.float32(0.4), np.float32(1)), decay="linear")[0].tolist() == [0]


def test_linear_identical_boxes():
    """The second box overlaps its top father at 1: decay 0.  Later fathers
    that overlap their own father at 1 give 0/0 (ignored) or x/0 (no effect)."""
    k = 5
    b = np.tile(np.array([[3, 3, 9, 7]], np.float32), (k, 1))
    s = np.linspace(0.9, 0.5, k).astype(np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, decay="linear")
    assert keep.tolist() == list(range(k))
    assert fs[0] == s[0] and all(f == 0.0 for f in fs[1:])
    assert oracle.matrix_nms(b, s, 1e-30, decay="linear")[0].tolist() == [0]


def test_linear_father_with_full_overlap():
    """A and A' identical (O_max of A' is 1), C overlaps both at IoU 1/2: the
    A' term is 0.5/0 = +inf and does not count; C decays by 1/2 from A."""
    b = np.array([[0, 0, 4, 4], [0, 0, 4, 4], [0, 0, 4, 2]], np.float32)
    s = np.array([0.9, 0.8, 0.7], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, decay="linear")
    assert keep.tolist() == [0, 1, 2]
    assert fs[1] == 0.0 and fs[2] == np.float32(float(np.float32(0.7)) * 0.5)


def test_linear_chain_hand_worked():
    """a=[0,0,10,1], b=[3,0,13,1], c=[6,0,16,1]: IoU(a,b) = IoU(b,c) = 7/13,
    IoU(a,c) = 1/4; O_max of b is 7/13.  b decays by 1 - 7/13 = 6/13 (from a);
    c by min(1 - 1/4 (from a), (1 - 7/13) / (1 - 7/13) = 1 (from b)) = 3/4."""
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1]], np.float32)
    s = np.array([0.9, 0.8, 0.7], np.float32)
    keep, fs = oracle.matrix_nms(b, s, 0.0, decay="linear")
    o = float(np.float32(7 / 13))  # the binary32 IoU of the two 7/13 pairs
    assert keep.tolist() == [0, 1, 2]
    assert fs[1] == np.float32(float(np.float32(0.8)) * (1.0 - o))
    assert fs[2] == np.float32(float(np.float32(0.7)) * 0.75)
    assert abs(float(fs[1]) - 0.8 * 6 / 13) < 1e-6


@pytest.mark.parametrize("seed", range(2))
def test_linear_exists_restatement(seed):
    """The existence form of the drop rule ("Optimization 4") with the linear
    decay, pair by pair from the binary32 IoUs (NaN terms never drop)."""
    rng = np.random.default_rng(20 + seed)
    n = 60
    b, s = _clustered(rng, n)
    t = 0.25
    keep, _ = oracle.matrix_nms(b, s, t, decay="linear")
    order = oracle.score_order(s)
    O = np.zeros((n, n))
    for p in range(n):
        for q in range(p):
            O[q, p] = float(oracle.iou(b[order[q]], b[order[p]]))
    omax = np.array([max([O[q, p] for q in range(p)], default=0.0) for p in range(n)])
    kept = []
    for p in range(n):
        sj = float(s[order[p]])
        drop = sj < t
        for q in range(p):
            den = 1.0 - omax[q]
            if den > 0 and sj * ((1.0 - O[q, p]) / den) < t:
                drop = True
        if not drop:
            kept.append(int(order[p]))
    assert keep.tolist() == kept


# ------------------------------------------ box-by-box form (large images)

def _decide_all(b, s, t, **kw):
    pos = np.arange(len(s) if kw.get("score_thr") is None else int((np.asarray(s) > kw["score_thr"]).sum()))
    idx, kept, fs = oracle.matrix_decide_at(b, s, t, pos, **kw)
    return idx[kept], fs[kept]


@pytest.mark.parametrize("sigma", [0.5, 2.0])
def test_decide_at_closed_forms(sigma):
    """The box-by-box form on the closed forms above: the pair at IoU exactly
    1/2 decays by exp(-0.25/sigma) (Gaussian) and by exactly 1/2 (linear);
    disjoint boxes keep their scores; identical boxes decay by exp(-2) after
    the first (sigma 1/2)."""
    b = np.array([[0, 0, 4, 4], [0, 0, 4, 2]], np.float32)
    s = np.array([0.9, 0.8], np.float32)
    idx, kept, fs = oracle.matrix_decide_at(b, s, 0.0, [1, 0], sigma=sigma)
    assert idx.tolist() == [1, 0] and kept.tolist() == [True, True]
    assert fs[0] == np.float32(float(np.float32(0.8)) * math.exp(-0.25 / float(np.float32(sigma))))
    assert fs[1] == np.float32(0.9)
    idx, kept, fs = oracle.matrix_decide_at(b, s, 0.0, [1], decay="linear")
    assert fs[0] == np.float32(0.4)
    d = np.array([[0, 0, 1, 1], [5, 5, 6, 6], [10, 0, 11, 1], [0, 10, 1, 11]], np.float32)
    sd = np.array([0.9, 0.2, 0.6, 0.4], np.float32)
    idx, kept, fs = oracle.matrix_decide_at(d, sd, 0.3, [0, 1, 2, 3])
    assert idx.tolist() == [0, 2, 3, 1] and kept.tolist() == [True, True, True, False]
    assert fs.tolist() == sd[[0, 2, 3, 1]].tolist()
    k = 6
    same = np.tile(np.array([[3, 3, 9, 7]], np.float32), (k, 1))
    ss = np.linspace(0.9, 0.4, k).astype(np.float32)
    idx, kept, fs = oracle.matrix_decide_at(same, ss, 0.0, np.arange(k))
    assert fs[0] == ss[0]
    assert all(fs[j] == np.float32(float(ss[j]) * math.exp(-2.0)) for j in range(1, k))


def test_decide_at_chain_hand_worked():
    """The three-box chain: c's decay is min(exp(-2 (1/4)^2), exp(0)) from
    fathers a and b, b's exp(-2 (7/13)^2)."""
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1]], np.float32)
    s = np.array([0.9, 0.8, 0.7], np.float32)
    _, _, fs = oracle.matrix_decide_at(b, s, 0.0, [0, 1, 2])
    r = float(Fraction(7, 13))
    # within 2e-7: the binary32 IoU of 7/13 is not 7/13 itself
    assert abs(fs[1] - float(s[1]) * math.exp(-2 * r * r)) <= 2e-7
    assert abs(fs[2] - float(s[2]) * math.exp(-2 * 0.0625)) <= 2e-7
    assert fs[0] == np.float32(0.9)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("decay", ["gaussian", "linear"])
def test_decide_at_matches_whole_image(seed, decay):
    """On clustered images with identical boxes, NaN boxes, a pre-filter and
    two thresholds, the box-by-box form keeps exactly the boxes the whole-image
    evaluation keeps, with the same final scores bit for bit."""
    rng = np.random.default_rng(seed)
    n = 300
    c = rng.uniform(0, 200, (12, 2))[rng.integers(0, 12, n)] + rng.normal(0, 4, (n, 2))
    wh = rng.uniform(5, 30, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    b[::23] = b[0]
    b[5] = np.nan
    s = rng.uniform(0, 1, n).astype(np.float32)
    for t in (0.05, 0.3):
        for thr in (None, 0.4):
            k, fs = oracle.matrix_nms(b, s, t, decay=decay, score_thr=thr)
            k2, fs2 = _decide_all(b, s, t, decay=decay, score_thr=thr)
            assert k2.tolist() == k.tolist()
            assert fs2.tobytes() == fs.tobytes()
