"""Seeded synthetic NMS workloads.

Pure data generation (numpy PCG64): boxes, scores, class ids and image offsets
with the shapes and value distributions of the five benchmark workloads.  No
step of the NMS method itself lives here; this module is shared by the tests,
the bench and the CPU oracle's callers because it only makes inputs.

Every value is drawn in float64 and cast to float32 once.  Boxes are
[cx - w/2, cy - h/2, cx + w/2, cy + h/2].  Cluster members pick their cluster
uniformly at random; cluster centres are uniform in the image.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


@dataclass
class Workload:
    name: str
    boxes: np.ndarray                      # float32 [n, 4] xyxy
    scores: np.ndarray                     # float32 [n]
    iou_thr: float
    class_ids: Optional[np.ndarray] = None  # int32 [n]
    batch_offsets: Optional[np.ndarray] = None  # int64 [B+1]
    num_classes: int = 1
    score_thr: Optional[float] = None
    max_out: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.scores.shape[0])

    @property
    def batch(self) -> int:
        return 1 if self.batch_offsets is None else int(self.batch_offsets.shape[0] - 1)

    @property
    def pairs(self) -> int:
        """IoU pairs of the upper triangle, summed over independent problems."""
        if self.batch_offsets is None and self.class_ids is None:
            return self.n * (self.n - 1) // 2
        return int(self.meta.get("pairs", 0))


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _xyxy(cx, cy, w, h) -> np.ndarray:
    return np.stack([cx - w / 2, cy - h / 2, cx + w / 2, cy + h / 2], 1).astype(np.float32)


def _clustered(rng, n, n_centres, image, jitter, wh_sampler):
    centres = rng.uniform(0, image, (n_centres, 2))
    member = rng.integers(0, n_centres, n)
    c = centres[member] + rng.normal(0, jitter, (n, 2))
    w, h = wh_sampler(rng, n)
    return _xyxy(c[:, 0], c[:, 1], w, h)


def single_1000(seed: int = 0) -> Workload:
    """N=1000: 40 clusters in a 640x640 image, jitter N(0,20), w,h ~ U(10,120);
    scores U(0,1) quantised to 1/256 (many exact ties); IoU threshold 0.5."""
    rng = _rng(seed)
    boxes = _clustered(rng, 1000, 40, 640.0, 20.0,
                       lambda r, n: (r.uniform(10, 120, n), r.uniform(10, 120, n)))
    scores = (np.floor(rng.uniform(0, 1, 1000) * 256) / 256).astype(np.float32)
    return Workload("single_n1000_ties", boxes, scores, 0.5)


def single_8192(seed: int = 0) -> Workload:
    """N=8192: 300 clusters in 1280x1280, jitter N(0,15), w,h ~ U(8,200);
    scores Beta(2,5); IoU threshold 0.5."""
    rng = _rng(seed)
    boxes = _clustered(rng, 8192, 300, 1280.0, 15.0,
                       lambda r, n: (r.uniform(8, 200, n), r.uniform(8, 200, n)))
    scores = rng.beta(2, 5, 8192).astype(np.float32)
    return Workload("single_n8192", boxes, scores, 0.5)


def single_32768(seed: int = 0) -> Workload:
    """N=32768: 1000 clusters in 2048x2048, jitter N(0,15), w,h log-uniform in
    [4,256]; scores U(0,1) with 1% (328) exact duplicates of another box's
    score; IoU threshold 0.7; at most 1000 outputs."""
    rng = _rng(seed)
    n = 32768

    def loguni(r, m):
        return (np.exp(r.uniform(np.log(4), np.log(256), m)),
                np.exp(r.uniform(np.log(4), np.log(256), m)))

    boxes = _clustered(rng, n, 1000, 2048.0, 15.0, loguni)
    scores = rng.uniform(0, 1, n).astype(np.float32)
    dup = rng.choice(n, 328, replace=False)
    src = rng.integers(0, n, 328)
    scores[dup] = scores[src]
    return Workload("single_n32768_maxout1000", boxes, scores, 0.7, max_out=1000)


def yolo_batched(seed: int = 0, batch: int = 16) -> Workload:
    """Batched class-aware: `batch` images x 25200 YOLO-640 candidates.
    For stride s in (8, 16, 32) (grids 80, 40, 20), anchor a in (0, 1, 2) and
    cell (gy, gx) in row-major order: centre ((gx+U)s, (gy+U)s), w,h =
    s * 2^a * exp(U(0, ln 4)); class U{0..79}; objectness score Beta(0.5, 8).
    Pre-filter score > 0.25, IoU threshold 0.45, at most 300 per image."""
    rng = _rng(seed)
    per = 3 * (80 * 80 + 40 * 40 + 20 * 20)
    boxes = []
    for b in range(batch):
        parts = []
        for s, g in ((8, 80), (16, 40), (32, 20)):
            for a in range(3):
                gy, gx = np.meshgrid(np.arange(g), np.arange(g), indexing="ij")
                gx = gx.reshape(-1).astype(np.float64)
                gy = gy.reshape(-1).astype(np.float64)
                m = g * g
                cx = (gx + rng.uniform(0, 1, m)) * s
                cy = (gy + rng.uniform(0, 1, m)) * s
                w = s * 2.0 ** a * np.exp(rng.uniform(0, np.log(4), m))
                h = s * 2.0 ** a * np.exp(rng.uniform(0, np.log(4), m))
                parts.append(_xyxy(cx, cy, w, h))
        boxes.append(np.concatenate(parts, 0))
    boxes = np.concatenate(boxes, 0)
    n = batch * per
    cls = rng.integers(0, 80, n).astype(np.int32)
    scores = rng.beta(0.5, 8, n).astype(np.float32)
    off = np.arange(0, n + 1, per, dtype=np.int64)
    wl = Workload(f"yolo_batched_{batch}x{per}", boxes, scores, 0.45, class_ids=cls,
                  batch_offsets=off, num_classes=80, score_thr=0.25, max_out=300)
    # IoU pairs actually examined: per (image, class) segment after the pre-filter.
    keep = scores > np.float32(0.25)
    seg = (np.repeat(np.arange(batch), per) * 80 + cls)[keep]
    sizes = np.bincount(seg, minlength=batch * 80).astype(np.int64)
    wl.meta["pairs"] = int((sizes * (sizes - 1) // 2).sum())
    wl.meta["candidates"] = int(keep.sum())
    return wl


def yolo_raw(seed: int = 0, batch: int = 16, classes: int = 80) -> np.ndarray:
    """YOLO-640 head output rows [batch, 25200, 5 + classes] float32, the
    shape an exported detector emits: (cx, cy, w, h) of the yolo_batched
    anchors (same layout and size law), objectness ~ Beta(0.5, 8), class
    scores ~ U(0, 0.3) except one class per anchor (U{0..classes-1}) at
    U(0.5, 1.0)."""
    wl = yolo_batched(seed, batch)
    rng = _rng(seed + 1000)
    n = wl.boxes.shape[0]
    b = wl.boxes.astype(np.float64)
    out = np.empty((n, 5 + classes), np.float32)
    out[:, 0] = (b[:, 0] + b[:, 2]) / 2
    out[:, 1] = (b[:, 1] + b[:, 3]) / 2
    out[:, 2] = b[:, 2] - b[:, 0]
    out[:, 3] = b[:, 3] - b[:, 1]
    out[:, 4] = rng.beta(0.5, 8, n)
    out[:, 5:] = rng.uniform(0, 0.3, (n, classes))
    cls = rng.integers(0, classes, n)
    out[np.arange(n), 5 + cls] = rng.uniform(0.5, 1.0, n)
    return out.reshape(batch, n // batch, 5 + classes)


def stress_dense(seed: int = 0) -> Workload:
    """N=65536 dense: 500 tight clusters in 8192x8192 (jitter N(0,3)), w,h ~
    U(20,48): about 95% of the boxes are suppressed.  Scores U(0,1); 0.5."""
    rng = _rng(seed)
    boxes = _clustered(rng, 65536, 500, 8192.0, 3.0,
                       lambda r, n: (r.uniform(20, 48, n), r.uniform(20, 48, n)))
    scores = rng.uniform(0, 1, 65536).astype(np.float32)
    return Workload("stress_n65536_dense", boxes, scores, 0.5)


def stress_sparse(seed: int = 0) -> Workload:
    """N=65536 sparse: centres uniform in 8192x8192, w,h ~ U(4,32): under 1%
    suppressed.  Scores U(0,1); IoU threshold 0.5."""
    rng = _rng(seed)
    c = rng.uniform(0, 8192, (65536, 2))
    w = rng.uniform(4, 32, 65536)
    h = rng.uniform(4, 32, 65536)
    boxes = _xyxy(c[:, 0], c[:, 1], w, h)
    scores = rng.uniform(0, 1, 65536).astype(np.float32)
    return Workload("stress_n65536_sparse", boxes, scores, 0.5)


CONFIGS = {
    "single_n1000_ties": single_1000,
    "single_n8192": single_8192,
    "single_n32768_maxout1000": single_32768,
    "yolo_batched": yolo_batched,
    "stress_n65536_dense": stress_dense,
    "stress_n65536_sparse": stress_sparse,
}

HEADLINE = "single_n8192"


def make(name: str, seed: int = 0) -> Workload:
    return CONFIGS[name](seed)


# ------------------------------------------------------------ lane candidates

LANE_VALUES = 77  # two class scores, start row, start x, length, 72 x samples
LANE_ROWS = 72


def lanes(seed: int = 0, n: int = 1000, true_lanes: int = 4, width: float = 640.0):
    """Lane candidates of one road image, shaped like an anchor-based lane
    detector's output before NMS: (props float32 [n, 77], scores float32 [n]).

    Four true lanes x(r) = x0 + a r + b r^2 over the 72 sample rows (r = 0 at
    the top), x0 ~ U(0.15, 0.85) width, a ~ U(-3, 3), b ~ U(-0.02, 0.02).  85%
    of the candidates follow a true lane (a whole-lane shift N(0, 12) px and
    per-row noise N(0, 2) px), the rest are random straight lanes; every
    candidate has a start row U{0..47} and a length U{16..72 - start}; x is
    quantised to 1/16 px.  The two class scores are (1 - s, s) with s, the
    score passed beside the candidates, ~ Beta(4, 2) for lane followers and
    Beta(1, 4) for the random ones.  Values 0, 1, 2, 3, 4: class scores,
    start row, x at the start row, length."""
    rng = _rng(seed)
    r = np.arange(LANE_ROWS, dtype=np.float64)
    x0 = rng.uniform(0.15, 0.85, true_lanes) * width
    a = rng.uniform(-3.0, 3.0, true_lanes)
    b = rng.uniform(-0.02, 0.02, true_lanes)
    follow = rng.uniform(0, 1, n) < 0.85
    which = rng.integers(0, true_lanes, n)
    shift = rng.normal(0, 12.0, n)
    noise = rng.normal(0, 2.0, (n, LANE_ROWS))
    rx0 = rng.uniform(0, width, n)
    ra = rng.uniform(-6.0, 6.0, n)
    x = np.where(follow[:, None],
                 x0[which, None] + a[which, None] * r + b[which, None] * r * r + shift[:, None] + noise,
                 rx0[:, None] + ra[:, None] * r)
    x = np.round(x * 16.0) / 16.0
    start = rng.integers(0, 48, n)
    length = np.array([rng.integers(16, LANE_ROWS - s + 1) for s in start])
    s = np.where(follow, rng.beta(4, 2, n), rng.beta(1, 4, n))
    props = np.zeros((n, LANE_VALUES), dtype=np.float64)
    props[:, 0] = 1 - s
    props[:, 1] = s
    props[:, 2] = start
    props[:, 3] = x[np.arange(n), start]
    props[:, 4] = length
    props[:, 5:] = x
    return props.astype(np.float32), s.astype(np.float32)
