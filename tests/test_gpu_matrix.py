"""GPU parity of Matrix NMS (nms_matrix_run) with the oracle: kept indices
and their order bit-exact, final scores within 4 binary32 ulp (the binary32
exponential's bound), on hand-worked cases, the workloads' shapes, clusters,
the pre-filter, max_out and thresholds."""
import math

import numpy as np
import pytest

import oracle
import greedy_iou_nms_gb300 as g
from greedy_iou_nms_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    g.load()


def _check(boxes, scores, t, **kw):
    b = torch.from_numpy(np.ascontiguousarray(boxes, np.float32)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    k, fs = g.matrix_nms(b, s, t, **kw)
    ek, efs = oracle.matrix_nms(boxes, scores, t, **kw)
    assert k.cpu().numpy().tolist() == ek.tolist()
    got = fs.cpu().numpy().astype(np.float64)
    ulp = np.spacing(np.abs(efs).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - efs) <= 4 * ulp + 1e-38)


def test_hand_worked():
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1], [0, 0, 4, 4], [0, 0, 4, 2]], np.float32)
    s = np.array([0.9, 0.8, 0.7, 0.6, 0.5], np.float32)
    for t in (0.0, 0.3, 0.45, 0.62):
        _check(b, s, t)


@pytest.mark.parametrize("name", ["single_n1000_ties", "single_n8192"])
@pytest.mark.parametrize("t", [0.05, 0.2])
def test_workload_shapes(name, t):
    wl = W.make(name, 0)
    _check(wl.boxes, wl.scores, t)


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 3000])
@pytest.mark.parametrize("sigma", [0.5, 2.0])
def test_clusters(n, sigma):
    rng = np.random.default_rng(n)
    k = max(n // 10, 1)
    c = rng.uniform(0, 500, (k, 2))[rng.integers(0, k, n)] + rng.normal(0, 5, (n, 2))
    wh = rng.uniform(10, 50, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check(b, s, 0.1, sigma=sigma)
    _check(b, s, 0.1, sigma=sigma, max_out=max(n // 7, 1))
    _check(b, s, 0.1, sigma=sigma, score_thr=0.3)


@pytest.mark.parametrize("decay", ["gaussian", "linear"])
def test_overlap_filter_edges(decay):
    """Pairs at the edges of the packed overlap filter: boxes that touch (a
    zero difference), nested boxes, degenerate boxes, and groups scaled by
    2^-45 and 2^45 (outside the filter's coordinate range, so those units
    test every pair exactly), next to ordinary ones in the same units."""
    rng = np.random.default_rng(7)
    x = rng.integers(0, 40, 300).astype(np.float32)
    y = rng.integers(0, 40, 300).astype(np.float32)
    w = rng.integers(0, 6, 300).astype(np.float32)  # zero widths too
    h = rng.integers(1, 6, 300).astype(np.float32)
    b = np.stack([x, y, x + w, y + h], 1)  # integer grid: many touching edges
    nest = np.array([[0, 0, 100, 100], [10, 10, 90, 90], [20, 20, 80, 80], [30, 30, 70, 70]], np.float32)
    tiny = (b[:100] * np.float32(2.0 ** -45)).astype(np.float32)
    huge = (b[100:200] * np.float32(2.0 ** 45)).astype(np.float32)
    allb = np.concatenate([b, nest, tiny, huge]).astype(np.float32)
    s = rng.uniform(0, 1, len(allb)).astype(np.float32)
    for t in (0.01, 0.1):
        if decay == "gaussian":
            _check(allb, s, t)
        else:
            _check_linear(allb, s, t)


@pytest.mark.parametrize("max_out", [1, 64, 100, 1000])
@pytest.mark.parametrize("decay", ["gaussian", "linear"])
def test_max_out_prefix(max_out, decay):
    """max_out decides the leading 2*max_out boxes first: a prefix that holds
    max_out kept boxes (spread boxes), one that does not (a stack of
    overlapping boxes ahead of the spread ones, decayed below the threshold),
    and a pre-filter that leaves fewer boxes than the prefix."""
    rng = np.random.default_rng(max_out + 17)
    n = 5000
    c = rng.uniform(0, 3000, (n, 2))
    wh = rng.uniform(5, 20, (n, 2))
    spread = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0.3, 0.9, n).astype(np.float32)
    stack = np.tile(np.array([[100, 100, 140, 140]], np.float32), (2500, 1)) + rng.uniform(0, 1, (2500, 1))
    b = np.concatenate([stack.astype(np.float32), spread])
    s2 = np.concatenate([rng.uniform(0.95, 1.0, 2500), s]).astype(np.float32)
    chk = _check if decay == "gaussian" else _check_linear
    chk(spread, s, 0.2, max_out=max_out)
    chk(b, s2, 0.2, max_out=max_out)
    chk(b, s2, 0.2, max_out=max_out, score_thr=0.955)


@pytest.mark.parametrize("decay", ["gaussian", "linear"])
def test_pair_list(decay):
    """From 16384 boxes pass A lists the overlapping pairs and pass B takes
    the list (20000 clustered boxes); with more overlapping pairs than the
    list holds (16384 boxes in a few tight stacks) pass B walks the units."""
    chk = _check if decay == "gaussian" else _check_linear
    rng = np.random.default_rng(31)
    n = 20000
    c = rng.uniform(0, 4000, (400, 2))[rng.integers(0, 400, n)] + rng.normal(0, 8, (n, 2))
    wh = rng.uniform(8, 40, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    chk(b, s, 0.2)
    chk(b, s, 0.2, score_thr=0.3)  # fewer candidates than the launch's bound
    n = 16384
    c = rng.uniform(0, 200, (4, 2))[rng.integers(0, 4, n)] + rng.normal(0, 2, (n, 2))
    b = np.concatenate([c - 20, c + 20], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    chk(b, s, 0.01)


def test_identical_boxes_and_empty():
    b = np.tile(np.array([[1, 1, 5, 5]], np.float32), (200, 1))
    s = np.linspace(1.0, 0.2, 200).astype(np.float32)
    _check(b, s, 0.05)
    _check(b, s, float(np.float32(0.9) * np.float32(math.exp(-2.0))))
    k, fs = g.matrix_nms(torch.zeros((0, 4), device="cuda"), torch.zeros(0, device="cuda"), 0.1)
    assert len(k) == 0


# ------------------------------------------------------------- linear decay

def _check_linear(boxes, scores, t, **kw):
    """Linear decay: indices and order bit-exact, final scores exactly the
    binary64 value rounded to binary32 (both sides take the same binary64
    quotient, minimum and product)."""
    b = torch.from_numpy(np.ascontiguousarray(boxes, np.float32)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    k, fs = g.matrix_nms(b, s, t, decay="linear", **kw)
    ek, efs = oracle.matrix_nms(boxes, scores, t, decay="linear", **kw)
    assert k.cpu().numpy().tolist() == ek.tolist()
    assert fs.cpu().numpy().tolist() == efs.tolist()


def test_linear_hand_worked():
    b = np.array([[0, 0, 10, 1], [3, 0, 13, 1], [6, 0, 16, 1], [0, 0, 4, 4], [0, 0, 4, 4], [0, 0, 4, 2]],
                 np.float32)
    s = np.array([0.9, 0.8, 0.7, 0.6, 0.55, 0.5], np.float32)
    for t in (0.0, 0.2, 0.3, 0.37, 0.5):
        _check_linear(b, s, t)


@pytest.mark.parametrize("name", ["single_n1000_ties", "single_n8192", "single_n32768_maxout1000"])
@pytest.mark.parametrize("t", [0.05, 0.2])
def test_linear_workload_shapes(name, t):
    wl = W.make(name, 0)
    _check_linear(wl.boxes, wl.scores, t, max_out=wl.max_out)


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 3000])
def test_linear_clusters(n):
    rng = np.random.default_rng(100 + n)
    k = max(n // 10, 1)
    c = rng.uniform(0, 500, (k, 2))[rng.integers(0, k, n)] + rng.normal(0, 5, (n, 2))
    wh = rng.uniform(10, 50, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    b[::17] = b[::17][0]  # a group of identical boxes: fathers that overlap their own father fully
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check_linear(b, s, 0.1)
    _check_linear(b, s, 0.1, max_out=max(n // 7, 1))
    _check_linear(b, s, 0.1, score_thr=0.3)


def test_linear_identical_boxes():
    b = np.tile(np.array([[1, 1, 5, 5]], np.float32), (200, 1))
    s = np.linspace(1.0, 0.2, 200).astype(np.float32)
    _check_linear(b, s, 0.0)
    _check_linear(b, s, 1e-30)


# ------------------------------------------------ the benchmark's full sizes

@pytest.mark.parametrize("name,nrand", [("stress_n65536_dense", 96), ("stress_n65536_sparse", 384)])
@pytest.mark.parametrize("decay", ["gaussian", "linear"])
def test_full_size_sampled(name, nrand, decay):
    """The 65536-box stress images at the benchmark's threshold (t = 0.1):
    the whole output satisfies what holds at any size (kept boxes in score
    order, final scores in [t, score]); sampled positions are checked one by
    one against the oracle's box-by-box form: random positions, the first
    boxes and the kept boxes closest to t.  Kept or not must agree; a kept
    box's final score is within 4 ulp (Gaussian) or exact (linear)."""
    t = 0.1
    wl = W.make(name, 0)
    n = wl.n
    k, fs = g.matrix_nms(torch.from_numpy(wl.boxes).cuda(), torch.from_numpy(wl.scores).cuda(), t, decay=decay)
    k = k.cpu().numpy()
    fs = fs.cpu().numpy()
    order = oracle.score_order(wl.scores)
    pos_of = np.empty(n, np.int64)
    pos_of[order] = np.arange(n)
    kp = pos_of[k]
    assert np.all(np.diff(kp) > 0)
    assert np.all(fs >= np.float32(t)) and np.all(fs <= wl.scores[k])
    rng = np.random.default_rng(5)
    pos = np.unique(np.concatenate([rng.choice(n, nrand, replace=False), np.arange(16),
                                    kp[np.argsort(fs, kind="stable")[:32]]]))
    idx, kept, efs = oracle.matrix_decide_at(wl.boxes, wl.scores, t, pos, decay=decay)
    assert np.isin(idx, k).tolist() == kept.tolist()
    got = dict(zip(k.tolist(), fs.tolist()))
    g_fs = np.array([got[i] for i in idx[kept].tolist()], np.float64)
    e_fs = efs[kept].astype(np.float64)
    if decay == "linear":
        assert g_fs.tolist() == e_fs.tolist()
    else:
        ulp = np.spacing(np.abs(efs[kept])).astype(np.float64)
        assert np.all(np.abs(g_fs - e_fs) <= 4 * ulp)


def test_gaussian_maxout_config():
    """The 32768-box image with max_out 1000 (Gaussian, t = 0.1) against the
    whole-image oracle."""
    wl = W.make("single_n32768_maxout1000", 0)
    _check(wl.boxes, wl.scores, 0.1, max_out=wl.max_out)
