"""GPU parity of the front end (nms_decode_boxes7) and of NMS over
count-header buffers (nms_boxes7_run) with the oracle: every float of the
buffers bit-exact (header, rows, keep flags), on hand-made and YOLO-shaped
predictions, with the max_objects cut, greedy and Fast NMS."""
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


def _same(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    assert a.shape == b.shape
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), np.argwhere(a.view(np.uint32) != b.view(np.uint32))[:5]


def _random_preds(seed, batch, anchors, classes):
    rng = np.random.default_rng(seed)
    p = np.empty((batch, anchors, 5 + classes), np.float32)
    c = rng.uniform(0, 200, (batch, max(anchors // 8, 1), 2))
    idx = rng.integers(0, c.shape[1], (batch, anchors))
    cen = np.take_along_axis(c, idx[..., None].repeat(2, -1), 1) + rng.normal(0, 4, (batch, anchors, 2))
    p[..., 0:2] = cen
    p[..., 2:4] = rng.uniform(4, 40, (batch, anchors, 2))
    p[..., 4] = rng.uniform(0, 1, (batch, anchors))
    p[..., 5:] = rng.uniform(0, 1, (batch, anchors, classes)) ** 3
    p[..., 5:][rng.uniform(size=(batch, anchors, classes)) < 0.02] = 0.5  # ties for the argmax
    return p


@pytest.mark.parametrize("batch,anchors,classes", [(1, 1, 1), (2, 127, 3), (3, 1000, 80), (1, 4099, 7)])
@pytest.mark.parametrize("max_objects", [0, 5, 300, 5000])
def test_decode_parity(batch, anchors, classes, max_objects):
    p = _random_preds(batch * anchors + classes, batch, anchors, classes)
    for thr in (0.2, 0.6):
        got = g.decode_boxes7(torch.from_numpy(p).cuda(), thr, max_objects).cpu().numpy()
        _same(got, oracle.decode_boxes7(p, thr, max_objects))


def test_decode_special_values():
    p = _random_preds(7, 2, 300, 4)
    p[0, ::7, 4] = np.nan
    p[0, 1::11, 5] = np.nan  # first class score NaN: never a maximum, confidence NaN
    p[1, ::5, 5:] = 0.7      # all classes tied
    p[1, 3::13, 2] = -3.0    # negative width
    got = g.decode_boxes7(torch.from_numpy(p).cuda(), 0.1, 400).cpu().numpy()
    _same(got, oracle.decode_boxes7(p, 0.1, 400))


@pytest.mark.parametrize("fast", [False, True])
@pytest.mark.parametrize("max_objects,thr", [(1000, 0.05), (300, 0.05), (1000, 0.25)])
def test_yolo_front_end_and_nms(fast, max_objects, thr):
    p = W.yolo_raw(0, batch=4)
    buf = g.decode_boxes7(torch.from_numpy(p).cuda(), thr, max_objects)
    exp = oracle.decode_boxes7(p, thr, max_objects)
    _same(buf.cpu().numpy(), exp)
    g.boxes7_nms(buf, 80, 0.45, fast=fast)
    _same(buf.cpu().numpy(), oracle.boxes7_nms(exp, 0.45, fast=fast))


@pytest.mark.parametrize("fast", [False, True])
def test_boxes7_dense_clusters(fast):
    """Many overlapping candidates of few classes (long greedy chains)."""
    p = _random_preds(3, 3, 2000, 3)
    p[..., 2:4] *= 2.5
    exp = oracle.decode_boxes7(p, 0.05, 2000)
    buf = torch.from_numpy(exp.copy()).cuda()
    g.boxes7_nms(buf, 3, 0.4, fast=fast)
    _same(buf.cpu().numpy(), oracle.boxes7_nms(exp, 0.4, fast=fast))


def test_boxes7_headers_and_invalid_class():
    p = _random_preds(5, 3, 200, 4)
    exp = oracle.decode_boxes7(p, 0.1, 50)
    exp[0, 0] = 1000.0          # above max_objects: all 50 rows
    exp[1, 0] = 7.5             # not an integer: 7 rows
    exp[2, 0] = np.nan          # none
    buf = torch.from_numpy(exp.copy()).cuda()
    g.boxes7_nms(buf, 4, 0.5)
    ref = exp.copy()
    ref[2, 0] = 0.0
    ref = oracle.boxes7_nms(ref, 0.5)
    ref[2, 0] = np.nan
    _same(buf.cpu().numpy(), ref)
    bad = exp.copy()
    bad[0, 1 + 5] = 9.0         # class beyond num_classes
    with pytest.raises(g.NmsError):
        g.boxes7_nms(torch.from_numpy(bad).cuda(), 4, 0.5)


def test_decode_no_anchors_and_repeat():
    p = np.zeros((3, 0, 9), np.float32)
    out = g.decode_boxes7(torch.from_numpy(p).cuda(), 0.1, 4).cpu().numpy()
    _same(out, oracle.decode_boxes7(p, 0.1, 4))
    # repeated calls with one workspace give the same buffers (the per-image
    # completion counters are reset by every call)
    q = _random_preds(9, 5, 3000, 20)
    t = torch.from_numpy(q).cuda()
    first = g.decode_boxes7(t, 0.3, 700).cpu().numpy()
    for _ in range(3):
        _same(g.decode_boxes7(t, 0.3, 700).cpu().numpy(), first)
    _same(first, oracle.decode_boxes7(q, 0.3, 700))
