"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element (keep indices, their order and the counts are integers: bit-exact).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import greedy_iou_nms_gb300 as g
from greedy_iou_nms_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    g.load()


def _gpu_nms(boxes, scores, thr, **kw):
    b = torch.from_numpy(np.ascontiguousarray(boxes, np.float32)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    cls = kw.pop("class_ids", None)
    off = kw.pop("batch_offsets", None)
    if cls is not None:
        kw["class_ids"] = torch.from_numpy(np.ascontiguousarray(cls, np.int32)).cuda()
    if off is not None:
        kw["batch_offsets"] = torch.from_numpy(np.ascontiguousarray(off, np.int64)).cuda()
    out = g.nms(b, s, thr, **kw)
    if isinstance(out, list):
        return [o.cpu().numpy() for o in out]
    return out.cpu().numpy()


def _check_single(boxes, scores, thr, max_out=0, score_thr=None):
    got = _gpu_nms(boxes, scores, thr, max_out=max_out, score_thr=score_thr)
    exp = oracle.nms_single(boxes, scores, thr, max_out=max_out, score_thr=score_thr)
    assert got.dtype == np.int64
    assert got.tolist() == exp.tolist()
    return got


def _check_workload(wl):
    keep, counts = oracle.nms(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids,
                              batch_offsets=wl.batch_offsets, score_thr=wl.score_thr,
                              max_out=wl.max_out)
    if wl.batch_offsets is None and wl.class_ids is None:
        got = _gpu_nms(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out, score_thr=wl.score_thr)
        assert len(got) == counts[0]
        assert got.tolist() == keep[: counts[0]].tolist()
        return
    got = _gpu_nms(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids,
                   num_classes=wl.num_classes, batch_offsets=wl.batch_offsets,
                   score_thr=wl.score_thr, max_out=wl.max_out)
    if wl.batch_offsets is None:
        got = [got]
    for b in range(wl.batch):
        base = b * wl.max_out if wl.max_out > 0 else int(wl.batch_offsets[b])
        assert got[b].tolist() == keep[base: base + counts[b]].tolist(), b


# ------------------------------------------------------------- golden cases

def test_golden_six_box():
    gd = json.load(open(os.path.join(GOLDEN, "six_box.json")))
    b = np.array(gd["boxes"], np.float32)
    s = np.array(gd["scores"], np.float32)
    for case in gd["cases"]:
        assert _gpu_nms(b, s, case["iou_thr"]).tolist() == case["keep"]


@pytest.mark.parametrize("name", ["at_threshold.json", "equal_scores.json"])
def test_golden_cases(name):
    gd = json.load(open(os.path.join(GOLDEN, name)))
    for case in gd["cases"]:
        got = _gpu_nms(np.array(case["boxes"], np.float32), np.array(case["scores"], np.float32),
                       case["iou_thr"])
        assert got.tolist() == case["keep"], case


def test_mask_bit_layout_golden():
    gd = json.load(open(os.path.join(GOLDEN, "bit_layout.json")))
    from test_oracle_pins import _bit_layout_boxes
    b = torch.from_numpy(_bit_layout_boxes(gd)).cuda()
    m = g.iou_mask(b, gd["iou_thr"]).cpu().numpy().view(np.uint64)
    got = sorted((i, 64 * w + k) for i in range(m.shape[0]) for w in range(m.shape[1])
                 for k in range(64) if (int(m[i, w]) >> k) & 1)
    assert got == sorted(tuple(x) for x in gd["expected_set_bits"])


# ------------------------------------------------------------ mask parity

def _sorted_random(n, seed, span=300.0, wmax=60.0, int_grid=False):
    rng = np.random.default_rng(seed)
    if int_grid:
        c = rng.integers(0, 20, (n, 2)).astype(np.float32)
        wh = rng.integers(1, 6, (n, 2)).astype(np.float32)
        return np.concatenate([c, c + wh], 1).astype(np.float32)
    c = rng.uniform(0, span, (n, 2))
    wh = rng.uniform(2, wmax, (n, 2))
    return np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)


@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 255, 256, 257, 700, 1000])
@pytest.mark.parametrize("thr", [0.5, 0.3])
def test_mask_parity(n, thr):
    b = _sorted_random(n, n + int(thr * 10), span=80.0 + n / 4)
    m = g.iou_mask(torch.from_numpy(b).cuda(), thr).cpu().numpy().view(np.uint64)
    ref = oracle.mask(b, thr)
    Wn = ref.shape[1]
    assert m.shape[1] >= Wn
    for i in range(n):
        w0 = i // 64
        assert np.array_equal(m[i, w0:Wn], ref[i, w0:Wn]), i
        assert not m[i, Wn:].any()


def test_mask_parity_integer_grid_ties():
    # Integer boxes give many IoUs exactly at 0.5 or at simple ratios: the
    # division-free test must hand those to the exact division.
    for seed in range(3):
        b = _sorted_random(600, seed, int_grid=True)
        for thr in (0.5, 0.25, 1 / 3, 0.6):
            m = g.iou_mask(torch.from_numpy(b).cuda(), thr).cpu().numpy().view(np.uint64)
            ref = oracle.mask(b, thr)
            for i in range(b.shape[0]):
                w0 = i // 64
                assert np.array_equal(m[i, w0:ref.shape[1]], ref[i, w0:])


def _canonical_iou32(a, b):
    """Canonical binary32 IoU of two boxes, used only to pick thresholds."""
    f = np.float32
    xx1, yy1 = max(f(a[0]), f(b[0])), max(f(a[1]), f(b[1]))
    xx2, yy2 = min(f(a[2]), f(b[2])), min(f(a[3]), f(b[3]))
    w, h = max(f(xx2 - xx1), f(0)), max(f(yy2 - yy1), f(0))
    inter = f(w * h)
    aa, ab = f(f(a[2] - a[0]) * f(a[3] - a[1])), f(f(b[2] - b[0]) * f(b[3] - b[1]))
    return f(inter / f(f(aa + ab) - inter))


def _mask_equal(b, thr):
    m = g.iou_mask(torch.from_numpy(np.ascontiguousarray(b, np.float32)).cuda(), thr).cpu().numpy().view(np.uint64)
    ref = oracle.mask(b, thr)
    for i in range(b.shape[0]):
        w0 = i // 64
        assert np.array_equal(m[i, w0:ref.shape[1]], ref[i, w0:]), (i, thr)


def test_mask_parity_nested_and_threshold_ulps():
    # Boxes nested in one axis or both (the filter's width and height bounds
    # are loosest there), with thresholds equal to, and one ulp either side
    # of, IoUs that occur in the set: every such pair sits on the strict
    # comparison's edge and must come out exactly as the definition says.
    rng = np.random.default_rng(21)
    n = 700
    big = np.array([0, 0, 200, 200], np.float32)
    c = rng.uniform(10, 190, (n, 2))
    wh = rng.uniform(1, 200, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    b[::5] = big
    b[1::7, 0], b[1::7, 2] = 0, 200          # spans the big box in x
    b[2::9, 1], b[2::9, 3] = 0, 200          # spans it in y
    picks = [_canonical_iou32(b[i], b[j]) for i, j in rng.integers(0, n, (40, 2)) if i != j]
    picks = [p for p in picks if 0.01 < p < 0.99][:8]
    assert picks
    for p in picks:
        for thr in (p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(1))):
            _mask_equal(b, float(thr))


@pytest.mark.parametrize("scale", [2.0 ** -40, 2.0 ** -20, 2.0 ** 20, 2.0 ** 40])
def test_mask_parity_scaled_coordinates(scale):
    # The same boxes at scales where every area is well inside the filter's
    # range (2^-20, 2^20) and where areas leave it (2^-40, 2^40: the tiles
    # then take the canonical test for every pair).
    b = (_sorted_random(500, 33, span=120.0) * np.float32(scale)).astype(np.float32)
    for thr in (0.5, 0.3):
        _mask_equal(b, thr)


# ------------------------------------------------------- workload parity

SINGLE = ["single_n1000_ties", "single_n8192", "single_n32768_maxout1000"]


@pytest.mark.parametrize("name", SINGLE)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_single_workloads(name, seed):
    _check_workload(W.make(name, seed))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_yolo_batched(seed):
    _check_workload(W.yolo_batched(seed))


@pytest.mark.parametrize("name", ["stress_n65536_dense", "stress_n65536_sparse"])
def test_stress_full_size(name):
    _check_workload(W.make(name, 0))


@pytest.mark.parametrize("n", [10, 100, 1024, 4096, 8192])
@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("thr", [0.5, 0.7])
def test_pages_random_sweep(n, seed, thr):
    """"NMS CUDA代码学习", section 实测数据: N in {10,100,1024,4096,8192} x 3 seeds x
    thresholds {0.5, 0.7}, scores with artificial ties."""
    rng = np.random.default_rng(1000 * seed + n)
    b = _sorted_random(n, seed + 7 * n, span=40.0 + 3 * math.sqrt(n) * 8, wmax=80.0)
    s = (np.floor(rng.uniform(0, 1, n) * 64) / 64).astype(np.float32)
    _check_single(b, s, thr)


# ------------------------------------------------------------- edge cases

def test_empty_and_single():
    assert _gpu_nms(np.zeros((0, 4), np.float32), np.zeros(0, np.float32), 0.5).tolist() == []
    assert _gpu_nms(np.array([[0, 0, 1, 1]], np.float32), np.array([0.3], np.float32), 0.5).tolist() == [0]


def test_special_scores_and_boxes():
    rng = np.random.default_rng(5)
    n = 500
    b = _sorted_random(n, 5, span=50.0)
    s = rng.uniform(0, 1, n).astype(np.float32)
    s[::7] = np.nan
    s[1::11] = -0.0
    s[2::11] = 0.0
    s[3::13] = -np.inf
    s[4::17] = np.inf
    b[5::19] = b[5::19][:, [2, 3, 0, 1]]          # inverted boxes (negative width/height)
    b[6::23, 2] = b[6::23, 0]                     # zero width
    b[7::29, 0] = np.nan                          # NaN coordinate
    for thr in (0.5, 0.0, -0.5, 1.0, 0.999):
        _check_single(b, s, thr)


@pytest.mark.parametrize("thr", [-1.0, 0.0, 1.0, 2.0, 1e-30, 1e30, math.inf, -math.inf])
def test_extreme_thresholds(thr):
    b = _sorted_random(300, 9, span=60.0)
    s = np.random.default_rng(9).uniform(0, 1, 300).astype(np.float32)
    _check_single(b, s, thr)


def test_identical_boxes_and_ties():
    b = np.tile(np.array([[3, 4, 13, 24]], np.float32), (700, 1))
    s = np.full(700, 0.5, np.float32)
    assert _gpu_nms(b, s, 0.5).tolist() == [0]
    s = (np.arange(700) % 3).astype(np.float32)
    _check_single(b, s, 0.99)


@pytest.mark.parametrize("n", [8192, 20000])
@pytest.mark.parametrize("levels", [1, 3, 16, 256])
def test_score_runs_of_ties(n, levels):
    # Runs of equal scores (one value, a few, quantised) over one sort chunk
    # and over several (merged by index across chunk boundaries), with a
    # sprinkle of infinities and NaN among them.
    wl = W.single_8192(5)
    rng = np.random.default_rng(levels)
    b = np.concatenate([wl.boxes] * ((n + 8191) // 8192))[:n]
    s = (rng.integers(0, levels, n) / levels + 0.25).astype(np.float32)
    s[rng.choice(n, 5, replace=False)] = [np.inf, -np.inf, np.nan, np.inf, np.nan]
    _check_single(b, s, 0.5)


@pytest.mark.parametrize("max_out", [1, 2, 63, 64, 65, 500, 5000])
def test_max_out_single(max_out):
    wl = W.single_8192(3)
    _check_single(wl.boxes, wl.scores, 0.5, max_out=max_out)


@pytest.mark.parametrize("score_thr", [0.0, 0.25, 0.5, 0.99, 2.0])
def test_prefilter_single(score_thr):
    wl = W.single_8192(4)
    _check_single(wl.boxes, wl.scores, 0.5, score_thr=score_thr)
    _check_single(wl.boxes, wl.scores, 0.5, score_thr=score_thr, max_out=100)


def test_batched_large_segments_and_empty_images():
    """Segments above 64 boxes take the one-CTA path; empty images and
    classes must come out empty."""
    rng = np.random.default_rng(21)
    sizes = [0, 300, 5, 0, 2000, 64, 65, 129]
    n = sum(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    b = _sorted_random(n, 21, span=150.0, wmax=50.0)
    s = (np.floor(rng.uniform(0, 1, n) * 32) / 32).astype(np.float32)
    cls = rng.integers(0, 3, n).astype(np.int32)
    cls[off[4]:off[5]] = 0  # one 2000-box single-class segment
    for max_out, score_thr in ((0, None), (50, 0.2), (3000, None)):
        wl = W.Workload("t", b, s, 0.5, class_ids=cls, batch_offsets=off, num_classes=3,
                        score_thr=score_thr, max_out=max_out)
        _check_workload(wl)


def test_batched_without_classes_and_single_image_with_classes():
    wl = W.single_8192(6)
    off = np.array([0, 1000, 1000, 5000, 8192], np.int64)
    _check_workload(W.Workload("t", wl.boxes, wl.scores, 0.5, batch_offsets=off))
    cls = np.random.default_rng(6).integers(0, 4, wl.n).astype(np.int32)
    _check_workload(W.Workload("t", wl.boxes, wl.scores, 0.5, class_ids=cls, num_classes=4,
                               max_out=700))


def test_device_side_validation():
    b = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    s = torch.ones(4, dtype=torch.float32, device="cuda")
    bad_off = torch.tensor([0, 3, 2, 4], dtype=torch.int64, device="cuda")
    with pytest.raises(g.NmsError) as e:
        g.nms(b, s, 0.5, batch_offsets=bad_off)
    assert e.value.code == g.NMS_ERR_INVALID_ARG
    bad_cls = torch.tensor([0, 1, 5, 0], dtype=torch.int32, device="cuda")
    with pytest.raises(g.NmsError) as e:
        g.nms(b, s, 0.5, class_ids=bad_cls, num_classes=2)
    assert e.value.code == g.NMS_ERR_INVALID_ARG


def test_repeat_runs_are_identical():
    """"NMS CUDA代码学习", section 三重 bug 诊断: run the same input 10 times;
    any cross-block race shows up as differing results."""
    for name in ("single_n8192", "yolo_batched"):
        wl = W.make(name, 1)
        outs = []
        for _ in range(10):
            if wl.class_ids is None:
                outs.append(_gpu_nms(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out).tolist())
            else:
                r = _gpu_nms(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids,
                             num_classes=wl.num_classes, batch_offsets=wl.batch_offsets,
                             score_thr=wl.score_thr, max_out=wl.max_out)
                outs.append([x.tolist() for x in r])
        assert all(o == outs[0] for o in outs)


def test_workspace_reuse_and_stream():
    """Calls on a side stream reusing one workspace give the same answers."""
    wl1, wl2 = W.single_1000(0), W.single_1000(1)
    ws = g.Workspace(1000)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for wl in (wl1, wl2, wl1):
            b = torch.from_numpy(wl.boxes).cuda()
            s = torch.from_numpy(wl.scores).cuda()
            got = g.nms(b, s, wl.iou_thr, workspace=ws).cpu().numpy()
            assert got.tolist() == oracle.nms_single(wl.boxes, wl.scores, wl.iou_thr).tolist()


# -------------------------------------------------------- resolve on its own

@pytest.mark.parametrize("n,span,max_out", [(1, 10.0, 0), (70, 30.0, 0), (1000, 100.0, 0),
                                            (5000, 300.0, 0), (20000, 900.0, 0),
                                            (20000, 900.0, 777), (4096, 64.0, 0)])
def test_resolve_mask_parity(n, span, max_out):
    """nms_resolve_mask on the library's own mask of score-sorted boxes equals
    the oracle's greedy result (as sorted positions)."""
    b = _sorted_random(n, n, span=span, wmax=40.0)
    s = np.linspace(1.0, 0.0, n, dtype=np.float32)  # already in score order, no ties
    exp = oracle.nms_single(b, s, 0.5, max_out=max_out)
    m = g.iou_mask(torch.from_numpy(b).cuda(), 0.5)
    got = g.resolve_mask(m, max_out=max_out).cpu().numpy()
    assert got.tolist() == exp.tolist()


def test_resolve_long_chains():
    """Boxes sliding by a small step: every box overlaps its next neighbours,
    so decisions inside a tile form long dependency chains."""
    n = 3000
    x = np.arange(n, dtype=np.float32) * 0.3
    b = np.stack([x, np.zeros(n), x + 1.0, np.ones(n)], 1).astype(np.float32)
    s = np.linspace(1.0, 0.0, n, dtype=np.float32)
    for thr in (0.5, 0.3, 0.8):
        exp = oracle.nms_single(b, s, thr)
        got = g.resolve_mask(g.iou_mask(torch.from_numpy(b).cuda(), thr)).cpu().numpy()
        assert got.tolist() == exp.tolist()
        assert _gpu_nms(b, s, thr).tolist() == exp.tolist()


def test_largest_single_image():
    """n = NMS_MAX_SINGLE_N (2^18): the widest chunk bitmaps and the largest
    shared-memory layout of the resolve; dense clusters keep the oracle quick."""
    n = g.NMS_MAX_SINGLE_N
    rng = np.random.default_rng(77)
    centres = rng.uniform(0, 4000, (800, 2))
    c = centres[rng.integers(0, 800, n)] + rng.normal(0, 2, (n, 2))
    wh = rng.uniform(20, 40, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check_single(b, s, 0.5)


def _parallel_chains(n_chains, length, step=0.3):
    """n_chains separate rows of unit boxes sliding by `step`; box k of every
    chain is visited before box k+1 of any chain, so the dependencies form
    n_chains chains of `length` links that all advance together."""
    k = np.repeat(np.arange(length), n_chains)
    c = np.tile(np.arange(n_chains), length)
    x = (k * step).astype(np.float32)
    y = (c * 10.0).astype(np.float32)
    b = np.stack([x, y, x + 1.0, y + 1.0], 1).astype(np.float32)
    s = (1.0 - np.arange(length * n_chains) / (length * n_chains)).astype(np.float32)
    perm = np.random.default_rng(length).permutation(len(s))
    return b[perm], s[perm]


@pytest.mark.parametrize("n_chains,length", [(100, 60), (64, 200), (64, 400), (8, 700), (1, 40)])
def test_dependency_chains_of_many_links(n_chains, length):
    """Chains deep enough to take many rounds of the sparse-graph resolve (and
    the longest ones past its round limit, where the walk takes over).  64
    chains of 400 links (25600 boxes, a round limit of 416, about 25 K pairs
    in one CTA) take about 306 passes (320 links took 257), past the wrap
    of the pass number that the per-box bytes hold."""
    b, s = _parallel_chains(n_chains, length)
    for thr in (0.5, 0.3):
        _check_single(b, s, thr)
    _check_single(b, s, 0.5, max_out=len(s) // 3)
    _check_single(b, s, 0.5, score_thr=0.25)


def test_pairs_concentrated_on_few_targets():
    """Many pairs ending in a narrow range of sorted positions (400 identical
    low-score boxes under 7792 scattered ones, ~80k pairs): more than one
    CTA's shared memory holds, so the first passes run over the list in
    global memory."""
    rng = np.random.default_rng(5)
    g_side = 89
    gx, gy = np.meshgrid(np.arange(g_side), np.arange(g_side))
    cx = (gx.ravel()[:7792] * 50.0).astype(np.float32)
    cy = (gy.ravel()[:7792] * 50.0).astype(np.float32)
    sparse = np.stack([cx, cy, cx + 10, cy + 10], 1)
    dup = np.tile(np.array([[10000.0, 10000.0, 10020.0, 10020.0]], np.float32), (400, 1))
    b = np.concatenate([sparse, dup]).astype(np.float32)
    s = np.concatenate([rng.uniform(0.5, 1.0, 7792), rng.uniform(0.0, 0.5, 400)]).astype(np.float32)
    p = rng.permutation(len(s))
    _check_single(b[p], s[p], 0.5)


def _clusters(n, k, jitter, seed, wh=(20.0, 40.0), span=3000.0):
    rng = np.random.default_rng(seed)
    centres = rng.uniform(0, span, (k, 2))
    c = centres[rng.integers(0, k, n)] + rng.normal(0, jitter, (n, 2))
    size = rng.uniform(wh[0], wh[1], (n, 2))
    b = np.concatenate([c - size / 2, c + size / 2], 1).astype(np.float32)
    return b, rng.uniform(0, 1, n).astype(np.float32)


@pytest.mark.parametrize("n,k,jitter,thr", [(8192, 100, 2.0, 0.5), (12000, 300, 6.0, 0.5),
                                            (16384, 600, 6.0, 0.5), (4000, 20, 10.0, 0.3),
                                            (4000, 4, 6.0, 0.3), (4000, 2, 6.0, 0.3)])
def test_lists_beyond_one_cta_up_to_16384_boxes(n, k, jitter, thr):
    """Clustered boxes whose pair list exceeds one CTA's shared memory (43 K
    to 49 K pairs) at no more than 16384 boxes: 67 K, 69 K, 151 K, 272 K and
    1.4 M pairs, where the first passes run over the list in global memory,
    compacting it in place, and the rest in shared memory once the
    survivors fit; and about 4 M pairs at 4000 boxes in two clusters, more
    than the list holds (1.57 M), where the walk decides.  Also with
    max_out, whose first stage must leave the list intact for the second."""
    b, s = _clusters(n, k, jitter, seed=n + k)
    _check_single(b, s, thr)
    _check_single(b, s, thr, max_out=n // 3)
    _check_single(b, s, thr, max_out=50)


def test_deep_chains_beyond_one_cta():
    """40 chains of 400 unit boxes sliding by 0.1 at threshold 0.3: five
    pairs a box (80 K pairs, more than one CTA holds) and well over a
    hundred passes, so the passes from global memory give up and the walk
    decides over the mask (which the in-place compaction leaves intact)."""
    b, s = _parallel_chains(40, 400, step=0.1)
    _check_single(b, s, 0.3)
    _check_single(b, s, 0.5)


@pytest.mark.parametrize("max_out,score_thr", [(100, None), (40, 0.3), (1, None), (3000, None)])
def test_max_out_needs_the_rest_of_the_mask(max_out, score_thr):
    """Heavy suppression (tight clusters): the leading 2*max_out boxes hold
    fewer than max_out kept boxes, so the rest of the mask and a second
    resolve are needed; small max_out values stop in the first part."""
    rng = np.random.default_rng(11)
    n = 6000
    centres = rng.uniform(0, 3000, (120, 2))
    c = centres[rng.integers(0, 120, n)] + rng.normal(0, 2, (n, 2))
    wh = rng.uniform(20, 40, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check_single(b, s, 0.5, max_out=max_out, score_thr=score_thr)


@pytest.mark.parametrize("zero_copy", [True, False])
def test_host_pipeline_matches_oracle(zero_copy):
    """HostPipeline, with the kernels moving the data across the host link
    (zero_copy: a copy kernel stages the pinned input, the resolve writes the
    pinned output) or with one packed host->device copy in and one
    device->host copy out: the kept indices equal the oracle's, for
    several sizes in one pipeline (the tail of the buffers is reused), and a
    later call sees new inputs written into the same buffer."""
    pipe = g.HostPipeline(9000, zero_copy=zero_copy)
    assert pipe.zero_copy == zero_copy  # pinned torch memory is mapped here
    for name, seed in (("single_n8192", 0), ("single_n1000_ties", 2), ("single_n8192", 1)):
        wl = W.make(name, seed)
        pipe.load(wl.boxes, wl.scores)
        got = pipe.run(wl.iou_thr, wl.score_thr, wl.max_out)
        exp = oracle.nms_single(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out)
        assert got.tolist() == exp.tolist()
        assert pipe.out_bytes(wl.max_out) == 8 * (1 + (len(exp) if zero_copy else wl.boxes.shape[0]))
    for mo in (5, 0):  # max_out through the captured graphs
        wl = W.make("single_n1000_ties", 3)
        pipe.load(wl.boxes, wl.scores)
        exp = oracle.nms_single(wl.boxes, wl.scores, wl.iou_thr, max_out=mo)
        assert pipe.run(wl.iou_thr, None, mo).tolist() == exp.tolist()
    pipe.set_n(0)
    assert len(pipe.run(0.5)) == 0


@pytest.mark.parametrize("nbytes,offset", [(163840, 0), (20 * 1001 + 4, 0), (37, 3), (16, 16)])
def test_copy_entry(nbytes, offset):
    """nms_copy: from mapped pinned host memory and from device memory into a
    device buffer, 16-byte words when the pointers and size allow and bytes
    otherwise (odd sizes, misaligned ends); the bytes around the range stay."""
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes + 64, dtype=np.uint8)).pin_memory()
    hsrc = g.nms_mapped_pointer(src.data_ptr())
    dsrc = src.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for s_addr in (hsrc + offset, dsrc.data_ptr() + offset):
        dst = torch.full((nbytes + 64,), 7, dtype=torch.uint8, device="cuda")
        assert g.nms_copy(dst.data_ptr() + offset, s_addr, nbytes, stream) == g.NMS_OK
        torch.cuda.synchronize()
        out = dst.cpu().numpy()
        assert np.array_equal(out[offset:offset + nbytes], src.numpy()[offset:offset + nbytes])
        assert (out[:offset] == 7).all() and (out[offset + nbytes:] == 7).all()
    assert g.nms_copy(dsrc.data_ptr(), hsrc, 0, stream) == g.NMS_OK  # nothing to do


def test_mapped_pointer():
    """nms_mapped_pointer: pinned host memory maps (offsets carry over),
    device memory and pageable memory do not."""
    pinned = torch.empty(64, dtype=torch.float32).pin_memory()
    base = g.nms_mapped_pointer(pinned.data_ptr())
    assert base is not None
    assert g.nms_mapped_pointer(pinned.data_ptr() + 16) == base + 16
    assert g.nms_mapped_pointer(torch.empty(64, device="cuda").data_ptr()) is None
    assert g.nms_mapped_pointer(np.zeros(64, np.float32).ctypes.data) is None


@pytest.mark.parametrize("max_out", [0, 150])
def test_pair_list_beyond_one_cta(max_out):
    """20000 boxes in tight clusters (~10^6 pairs over the threshold): more
    pairs than one CTA's shared memory holds, so all SMs take the rounds."""
    rng = np.random.default_rng(21)
    n = 20000
    centres = rng.uniform(0, 6000, (200, 2))
    c = centres[rng.integers(0, 200, n)] + rng.normal(0, 1.5, (n, 2))
    wh = rng.uniform(20, 30, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check_single(b, s, 0.5, max_out=max_out)
