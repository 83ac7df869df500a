"""Pins of the front-end oracle: the [count, 7-float rows] buffer of
"YOLOv5后处理GPU移植实战" (section 1.1 layout, section 1.2 slot counter with
the max_objects cut) filled from YOLO-shaped predictions, and NMS over such a
buffer (section 2.2: priority by confidence, then the lower position).  Values
are worked by hand; the decode itself is not printed on the page, so its
pins fix the readings (confidence = objectness x the largest class score,
first class among equal maxima, strict threshold, centre +- half size)."""
import numpy as np

import oracle


def _preds(rows, classes):
    p = np.zeros((1, len(rows), 5 + classes), np.float32)
    for a, r in enumerate(rows):
        p[0, a, :len(r)] = r
    return p


def test_decode_hand_worked():
    q = float(np.nextafter(np.float32(0.25), np.float32(1)))
    p = _preds([
        [10, 20, 4, 6, 0.5, 0.2, 0.9, 0.9],     # class 1 (first of two maxima), conf 0.45
        [30, 30, 8, 8, 0.5, 0.5, 0.1, 0.0],     # conf 0.25 == threshold: not a candidate
        [5, 7, 3, 5, 1.0, 0.0, 0.0, q],         # conf just above 0.25, class 2
        [1, 1, 2, 2, np.nan, 0.9, 0.9, 0.9],    # NaN confidence: not a candidate
    ], 3)
    out = oracle.decode_boxes7(p, 0.25, 4)
    assert out.shape == (1, 29)
    assert out[0, 0] == 2
    r0 = out[0, 1:8].tolist()
    assert r0 == [8.0, 17.0, 12.0, 23.0, float(np.float32(0.5) * np.float32(0.9)), 1.0, 1.0]
    r1 = out[0, 8:15].tolist()
    assert r1 == [3.5, 4.5, 6.5, 9.5, np.float32(q), 2.0, 1.0]
    assert not out[0, 15:].any()


def test_decode_cut_at_max_objects():
    """Five candidates, three slots: the header counts all five, the rows hold
    the first three in anchor order, the rest of the buffer is untouched."""
    rows = [[10 * a, 0, 2, 2, 0.9, 1.0] for a in range(7)]
    rows[1][4] = rows[4][4] = 0.0  # two non-candidates
    out = oracle.decode_boxes7(_preds(rows, 1), 0.5, 3)
    assert out[0, 0] == 5
    assert out[0, 1:22].reshape(3, 7)[:, 0].tolist() == [-1.0, 19.0, 29.0]
    out0 = oracle.decode_boxes7(_preds(rows, 1), 0.5, 0)
    assert out0.shape == (1, 1) and out0[0, 0] == 5


def test_decode_images_independent():
    p = np.zeros((2, 2, 7), np.float32)
    p[0, 1] = [4, 4, 2, 2, 0.8, 0.1, 0.7]
    p[1, 0] = [6, 6, 2, 2, 0.9, 0.6, 0.2]
    out = oracle.decode_boxes7(p, 0.1, 2)
    assert out[:, 0].tolist() == [1.0, 1.0]
    assert out[0, 1:8].tolist() == [3.0, 3.0, 5.0, 5.0, float(np.float32(0.8) * np.float32(0.7)), 1.0, 1.0]
    assert out[1, 1:8].tolist() == [5.0, 5.0, 7.0, 7.0, float(np.float32(0.9) * np.float32(0.6)), 0.0, 1.0]


def _buf(rows, max_objects):
    b = np.zeros((1, 1 + 7 * max_objects), np.float32)
    b[0, 0] = len(rows)
    b[0, 1:1 + 7 * len(rows)] = np.array(rows, np.float32).reshape(-1)
    return b


def test_boxes7_greedy_and_fast():
    """A > B > C of one class, IoU(A,B) = IoU(B,C) = 1/3 > 0.3, IoU(A,C) = 0:
    greedy keeps A and C (B, the only box over C, is removed); Fast NMS keeps A
    only (C goes because B overlaps it, kept or not).  D, another class, on top
    of A stays.  E ties A's confidence at a later position: A wins the tie."""
    A = [0, 0, 4, 2, 0.9, 0, 1]
    B = [2, 0, 6, 2, 0.8, 0, 1]
    C = [4, 0, 8, 2, 0.7, 0, 1]
    D = [0, 0, 4, 2, 0.95, 3, 1]
    E = [0, 0, 4, 2, 0.9, 0, 1]
    g = oracle.boxes7_nms(_buf([A, B, C, D, E], 6), 0.3)
    assert g[0, 1:36].reshape(5, 7)[:, 6].tolist() == [1, 0, 1, 1, 0]
    f = oracle.boxes7_nms(_buf([A, B, C, D, E], 6), 0.3, fast=True)
    assert f[0, 1:36].reshape(5, 7)[:, 6].tolist() == [1, 0, 0, 1, 0]
    # rows past the count are untouched; a header above max_objects uses max_objects rows
    b = _buf([A, B], 3)
    b[0, 15:22] = 7.0
    assert (oracle.boxes7_nms(b, 0.3)[0, 15:22] == 7.0).all()
    b = _buf([A, B, C], 3)
    b[0, 0] = 9
    assert oracle.boxes7_nms(b, 0.3)[0, 1:22].reshape(3, 7)[:, 6].tolist() == [1, 0, 1]
