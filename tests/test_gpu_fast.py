"""GPU parity of Fast NMS (nms_fast_run) with the oracle: kept indices, their
order and the counts, bit-exact, on the golden cases, every workload (one
image and batched, class-aware), the pre-filter, max_out, edge cases and
large segments."""
import json
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


def _fast(boxes, scores, thr, **kw):
    b = torch.from_numpy(np.ascontiguousarray(boxes, np.float32)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    cls = kw.pop("class_ids", None)
    off = kw.pop("batch_offsets", None)
    if cls is not None:
        kw["class_ids"] = torch.from_numpy(np.ascontiguousarray(cls, np.int32)).cuda()
    if off is not None:
        kw["batch_offsets"] = torch.from_numpy(np.ascontiguousarray(off, np.int64)).cuda()
    out = g.nms(b, s, thr, fast=True, **kw)
    if isinstance(out, list):
        return [o.cpu().numpy() for o in out]
    return out.cpu().numpy()


def _check_single(boxes, scores, thr, max_out=0, score_thr=None):
    got = _fast(boxes, scores, thr, max_out=max_out, score_thr=score_thr)
    exp = oracle.nms_single(boxes, scores, thr, max_out=max_out, score_thr=score_thr, fast=True)
    assert got.tolist() == exp.tolist()


def test_golden_cases():
    with open(os.path.join(GOLDEN, "fast_nms.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = _fast(np.array(c["boxes"], np.float32), np.array(c["scores"], np.float32), c["iou_thr"])
        assert got.tolist() == c["keep"], c["name"]


@pytest.mark.parametrize("name", [n for n in W.CONFIGS])
@pytest.mark.parametrize("seed", [0, 1])
def test_workloads(name, seed):
    wl = W.make(name, seed)
    keep, counts = oracle.nms(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids,
                              batch_offsets=wl.batch_offsets, score_thr=wl.score_thr,
                              max_out=wl.max_out, fast=True)
    if wl.batch_offsets is None and wl.class_ids is None:
        got = _fast(wl.boxes, wl.scores, wl.iou_thr, max_out=wl.max_out, score_thr=wl.score_thr)
        assert got.tolist() == keep[: counts[0]].tolist()
        return
    got = _fast(wl.boxes, wl.scores, wl.iou_thr, class_ids=wl.class_ids, num_classes=wl.num_classes,
                batch_offsets=wl.batch_offsets, score_thr=wl.score_thr, max_out=wl.max_out)
    if wl.batch_offsets is None:
        got = [got]
    for b in range(wl.batch):
        base = b * wl.max_out if wl.max_out > 0 else int(wl.batch_offsets[b])
        assert got[b].tolist() == keep[base: base + counts[b]].tolist(), b


@pytest.mark.parametrize("n", [1, 33, 1000, 4096])
@pytest.mark.parametrize("thr", [0.3, 0.5, 0.7])
def test_random_clusters(n, thr):
    rng = np.random.default_rng(n)
    c = rng.uniform(0, 400, (max(n // 8, 1), 2))[rng.integers(0, max(n // 8, 1), n)] + rng.normal(0, 6, (n, 2))
    wh = rng.uniform(10, 60, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    _check_single(b, s, thr)
    _check_single(b, s, thr, max_out=max(n // 5, 1))
    _check_single(b, s, thr, score_thr=0.4)


@pytest.mark.parametrize("max_out", [1, 64, 100, 1000])
def test_max_out_prefix(max_out):
    """max_out runs the mask of the leading 2*max_out boxes first: a prefix
    that holds max_out kept boxes (spread boxes), one that does not (a stack
    of overlapping boxes ahead of the spread ones), and a pre-filter that
    leaves fewer boxes than the prefix."""
    rng = np.random.default_rng(max_out)
    n = 6000
    c = rng.uniform(0, 3000, (n, 2))
    wh = rng.uniform(5, 20, (n, 2))
    spread = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 0.9, n).astype(np.float32)
    _check_single(spread, s, 0.5, max_out=max_out)
    stack = np.tile(np.array([[100, 100, 140, 140]], np.float32), (3000, 1)) + rng.uniform(0, 1, (3000, 1))
    b = np.concatenate([stack.astype(np.float32), spread])
    s2 = np.concatenate([rng.uniform(0.95, 1.0, 3000), s]).astype(np.float32)
    _check_single(b, s2, 0.5, max_out=max_out)
    _check_single(b, s2, 0.5, max_out=max_out, score_thr=0.955)


def test_empty_and_ties():
    assert len(_fast(np.zeros((0, 4), np.float32), np.zeros(0, np.float32), 0.5)) == 0
    b = np.tile(np.array([[0, 0, 10, 10]], np.float32), (70, 1))
    s = np.full(70, 0.5, np.float32)
    _check_single(b, s, 0.5)


def test_batched_large_segments():
    """Segments above 64 boxes (one CTA per segment) test each box against every
    earlier box of its segment."""
    rng = np.random.default_rng(3)
    B, per = 3, 700
    offs = np.arange(0, (B + 1) * per, per, dtype=np.int64)
    n = B * per
    c = rng.uniform(0, 300, (n, 2))
    wh = rng.uniform(10, 50, (n, 2))
    b = np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)
    s = rng.uniform(0, 1, n).astype(np.float32)
    cls = rng.integers(0, 2, n).astype(np.int32)
    keep, counts = oracle.nms(b, s, 0.5, class_ids=cls, batch_offsets=offs, fast=True)
    got = _fast(b, s, 0.5, class_ids=cls, num_classes=2, batch_offsets=offs)
    for i in range(B):
        assert got[i].tolist() == keep[offs[i]: offs[i] + counts[i]].tolist()
