"""Greedy IoU NMS oracle (TEST INFRASTRUCTURE ONLY).

A plain, slow, single-threaded CPU implementation of greedy hard NMS, written
in C (``nms_oracle.c``) and loaded with ctypes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package.  It shares no code with ``greedy_iou_nms_gb300``.

Every function restates the method as the pages define it; see the header of
``nms_oracle.c`` for the citations and the readings taken where the pages are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nms_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

# -ffp-contract=off: gcc contracts a*b+c into an FMA by default on aarch64,
# which would change the binary32 rounding of the canonical IoU.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None

# The multi-core bitmask baseline (cpu_baseline.c): its own library, built with
# OpenMP; bench.py's CPU-baseline leg and its pin tests use it.
_BASE_SRC = os.path.join(_HERE, "cpu_baseline.c")
_BASE_LIB = os.path.join(_HERE, "_build", "libcpubase.so")
BASE_CFLAGS = ["-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_base = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (idempotent)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i32p = ctypes.POINTER(ctypes.c_int32)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.oracle_iou.argtypes = [f32p, f32p]
        lib.oracle_iou.restype = ctypes.c_float
        lib.oracle_nms.argtypes = [f32p, f32p, ctypes.c_int64, i32p, i64p, ctypes.c_int32,
                                   ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_int32,
                                   i64p, i64p]
        lib.oracle_nms.restype = ctypes.c_int64
        lib.oracle_fast_nms.argtypes = lib.oracle_nms.argtypes
        lib.oracle_fast_nms.restype = ctypes.c_int64
        lib.oracle_matrix_nms.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_float, ctypes.c_int32, i64p, f32p]
        lib.oracle_matrix_nms.restype = ctypes.c_int64
        lib.oracle_matrix_decide_at.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_float, ctypes.c_float, i64p,
                                                ctypes.c_int64, i64p, ctypes.POINTER(ctypes.c_int32), f32p]
        lib.oracle_matrix_decide_at.restype = ctypes.c_int64
        lib.oracle_lane_distance.argtypes = [f32p, f32p]
        lib.oracle_lane_distance.restype = ctypes.c_float
        lib.oracle_lane_nms.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32, i64p]
        lib.oracle_lane_nms.restype = ctypes.c_int64
        lib.oracle_score_order.argtypes = [f32p, i64p, ctypes.c_int64]
        lib.oracle_score_order.restype = None
        lib.oracle_mask.argtypes = [f32p, ctypes.c_int64, ctypes.c_float, u64p]
        lib.oracle_mask.restype = None
        lib.oracle_decode_boxes7.argtypes = [f32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                             ctypes.c_int32, f32p]
        lib.oracle_decode_boxes7.restype = None
        _lib = lib
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def iou(a, b) -> np.float32:
    """Canonical binary32 IoU of two xyxy boxes."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return np.float32(_load().oracle_iou(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float)))


def score_order(scores) -> np.ndarray:
    """Greedy visiting order: stable descending score, NaN last."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    idx = np.arange(s.shape[0], dtype=np.int64)
    _load().oracle_score_order(_ptr(s, ctypes.c_float), _ptr(idx, ctypes.c_int64), s.shape[0])
    return idx


def nms(boxes, scores, iou_thr, *, class_ids=None, batch_offsets=None, score_thr=None,
        max_out=0, fast=False):
    """Greedy NMS (Fast NMS with fast=True).  Returns (keep, counts) exactly as
    the library lays them out: image b's kept indices sit at keep[b*max_out]
    (max_out > 0) or at keep[batch_offsets[b]] (no cap); counts[b] is their
    number.  For a single image, keep[:counts[0]] is the answer."""
    bx = np.ascontiguousarray(boxes, dtype=np.float32).reshape(-1, 4)
    sc = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    n = sc.shape[0]
    assert bx.shape[0] == n
    cls = None if class_ids is None else np.ascontiguousarray(class_ids, dtype=np.int32)
    off = None if batch_offsets is None else np.ascontiguousarray(batch_offsets, dtype=np.int64)
    batch = 1 if off is None else off.shape[0] - 1
    cap = batch * max_out if max_out > 0 else n
    keep = np.full(max(cap, 1), -1, dtype=np.int64)
    counts = np.zeros(batch, dtype=np.int64)
    fn = _load().oracle_fast_nms if fast else _load().oracle_nms
    total = fn(
        _ptr(bx, ctypes.c_float), _ptr(sc, ctypes.c_float), n,
        None if cls is None else _ptr(cls, ctypes.c_int32),
        None if off is None else _ptr(off, ctypes.c_int64), batch,
        float(np.float32(iou_thr)), 0 if score_thr is None else 1,
        float(np.float32(score_thr if score_thr is not None else 0.0)), int(max_out),
        _ptr(keep, ctypes.c_int64), _ptr(counts, ctypes.c_int64))
    if total < 0:
        raise ValueError("oracle_nms: invalid arguments")
    return keep[:cap], counts


def nms_single(boxes, scores, iou_thr, *, max_out=0, score_thr=None, fast=False) -> np.ndarray:
    """Single image, single class: the kept indices in score order."""
    keep, counts = nms(boxes, scores, iou_thr, max_out=max_out, score_thr=score_thr, fast=fast)
    return keep[: counts[0]].copy()


def matrix_nms(boxes, scores, decay_thr, *, sigma=0.5, decay="gaussian", score_thr=None, max_out=0):
    """Matrix NMS of one image with the Gaussian (exp((O_max^2 - O^2)/sigma))
    or the linear ((1 - O)/(1 - O_max)) decay: (kept indices in score order,
    their final scores as binary32)."""
    if decay not in ("gaussian", "linear"):
        raise ValueError("matrix_nms: decay must be 'gaussian' or 'linear'")
    bx = np.ascontiguousarray(boxes, dtype=np.float32).reshape(-1, 4)
    sc = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    n = sc.shape[0]
    keep = np.full(max(n, 1), -1, dtype=np.int64)
    fs = np.zeros(max(n, 1), dtype=np.float32)
    k = _load().oracle_matrix_nms(_ptr(bx, ctypes.c_float), _ptr(sc, ctypes.c_float), n,
                                  float(np.float32(sigma)), 1 if decay == "linear" else 0,
                                  0 if score_thr is None else 1,
                                  float(np.float32(score_thr if score_thr is not None else 0.0)),
                                  float(np.float32(decay_thr)), int(max_out),
                                  _ptr(keep, ctypes.c_int64), _ptr(fs, ctypes.c_float))
    if k < 0:
        raise ValueError("oracle_matrix_nms: invalid arguments")
    return keep[:k].copy(), fs[:k].copy()


def matrix_decide_at(boxes, scores, decay_thr, positions, *, sigma=0.5, decay="gaussian", score_thr=None):
    """Matrix NMS (no max_out) decided box by box at the given sorted
    positions: (input indices there, kept flags, final scores as binary32)."""
    if decay not in ("gaussian", "linear"):
        raise ValueError("matrix_decide_at: decay must be 'gaussian' or 'linear'")
    bx = np.ascontiguousarray(boxes, dtype=np.float32).reshape(-1, 4)
    sc = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    pos = np.ascontiguousarray(positions, dtype=np.int64).reshape(-1)
    k = pos.shape[0]
    idx = np.zeros(max(k, 1), dtype=np.int64)
    kept = np.zeros(max(k, 1), dtype=np.int32)
    fs = np.zeros(max(k, 1), dtype=np.float32)
    m = _load().oracle_matrix_decide_at(_ptr(bx, ctypes.c_float), _ptr(sc, ctypes.c_float), sc.shape[0],
                                        float(np.float32(sigma)), 1 if decay == "linear" else 0,
                                        0 if score_thr is None else 1,
                                        float(np.float32(score_thr if score_thr is not None else 0.0)),
                                        float(np.float32(decay_thr)), _ptr(pos, ctypes.c_int64), k,
                                        _ptr(idx, ctypes.c_int64), _ptr(kept, ctypes.c_int32),
                                        _ptr(fs, ctypes.c_float))
    if m < 0:
        raise ValueError("oracle_matrix_decide_at: invalid arguments")
    return idx[:k].copy(), kept[:k].astype(bool), fs[:k].copy()


LANE_VALUES = 77  # values of one lane candidate (see oracle_lane_nms)
LANE_ROWS = 72


def lane_distance(a, b) -> np.float32:
    """Distance of two lane candidates (77 values each): mean |x_a - x_b| over
    the rows both cover, +inf without common rows."""
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(LANE_VALUES)
    b = np.ascontiguousarray(b, dtype=np.float32).reshape(LANE_VALUES)
    return np.float32(_load().oracle_lane_distance(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float)))


def lane_nms(props, scores, thr, *, max_out=0) -> np.ndarray:
    """Greedy NMS of lane candidates [n, 77]: kept input indices in score
    order (a lane goes when its distance to a kept lane is below thr)."""
    pr = np.ascontiguousarray(props, dtype=np.float32).reshape(-1, LANE_VALUES)
    sc = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    n = sc.shape[0]
    keep = np.full(max(n, 1), -1, dtype=np.int64)
    k = _load().oracle_lane_nms(_ptr(pr, ctypes.c_float), _ptr(sc, ctypes.c_float), n, float(np.float32(thr)),
                                int(max_out), _ptr(keep, ctypes.c_int64))
    if k < 0:
        raise ValueError("oracle_lane_nms: invalid arguments")
    return keep[:k].copy()


def mask(boxes_sorted, iou_thr) -> np.ndarray:
    """Row-major [n][ceil(n/64)] uint64 suppression bitmask of score-sorted boxes."""
    bx = np.ascontiguousarray(boxes_sorted, dtype=np.float32).reshape(-1, 4)
    n = bx.shape[0]
    W = (n + 63) // 64
    m = np.zeros((n, max(W, 1)), dtype=np.uint64)
    _load().oracle_mask(_ptr(bx, ctypes.c_float), n, float(np.float32(iou_thr)),
                        _ptr(m, ctypes.c_uint64))
    return m[:, :W]


def decode_boxes7(preds, conf_thr, max_objects) -> np.ndarray:
    """The [count, 7-float rows] buffers of YOLO-shaped predictions
    [batch, anchors, 5 + classes]: float32 [batch, 1 + 7 * max_objects],
    unused rows zero."""
    p = np.ascontiguousarray(preds, dtype=np.float32)
    if p.ndim != 3 or p.shape[2] < 6 or max_objects < 0:
        raise ValueError("decode_boxes7: preds must be [batch, anchors, 5 + classes]")
    batch, anchors, width = p.shape
    out = np.zeros((batch, 1 + 7 * max_objects), dtype=np.float32)
    _load().oracle_decode_boxes7(_ptr(p, ctypes.c_float), batch, anchors, width - 5,
                                 float(np.float32(conf_thr)), int(max_objects), _ptr(out, ctypes.c_float))
    return out


def boxes7_nms(buffers, iou_thr, *, fast=False) -> np.ndarray:
    """keep_flag of every row of [count, 7-float rows] buffers after class-aware
    NMS in the buffer's own priority (confidence descending, then row
    position), greedy or Fast NMS ("YOLOv5后处理GPU移植实战", section 2.2):
    returns a copy of the buffers with row flags 1 (kept) or 0; rows past
    min(count, max_objects) are untouched."""
    out = np.array(buffers, dtype=np.float32, copy=True)
    batch, width = out.shape
    max_objects = (width - 1) // 7
    for b in range(batch):
        m = min(int(out[b, 0]), max_objects)
        rows = out[b, 1:1 + 7 * m].reshape(m, 7)
        keep, counts = nms(rows[:, :4], rows[:, 4], iou_thr, class_ids=rows[:, 5].astype(np.int32), fast=fast)
        flags = np.zeros(m, dtype=np.float32)
        flags[keep[:counts[0]]] = 1.0
        rows[:, 6] = flags
        out[b, 1:1 + 7 * m] = rows.reshape(-1)
    return out


def build_cpu_baseline(force: bool = False) -> str:
    """Compile the multi-core CPU baseline with gcc and OpenMP (idempotent)."""
    os.makedirs(os.path.dirname(_BASE_LIB), exist_ok=True)
    if force or not os.path.exists(_BASE_LIB) or os.path.getmtime(_BASE_LIB) < os.path.getmtime(_BASE_SRC):
        tmp = _BASE_LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *BASE_CFLAGS, "-o", tmp, _BASE_SRC, "-lm"])
        os.replace(tmp, _BASE_LIB)
    return _BASE_LIB


def _load_base():
    global _base
    if _base is None:
        lib = ctypes.CDLL(build_cpu_baseline())
        f32p = ctypes.POINTER(ctypes.c_float)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.cpu_baseline_threads.restype = ctypes.c_int
        lib.cpu_baseline_nms.argtypes = [f32p, f32p, ctypes.c_int64, i32p, i64p, ctypes.c_int32, ctypes.c_float,
                                         ctypes.c_int, ctypes.c_float, ctypes.c_int32, i64p, i64p]
        lib.cpu_baseline_nms.restype = ctypes.c_int64
        _base = lib
    return _base


def cpu_baseline_threads() -> int:
    """Threads the multi-core baseline runs on."""
    return int(_load_base().cpu_baseline_threads())


def cpu_baseline_nms(boxes, scores, iou_thr, *, class_ids=None, batch_offsets=None, score_thr=None, max_out=0):
    """Greedy NMS on all host cores (bitmask and resolve, cpu_baseline.c):
    (keep, counts) laid out as for nms()."""
    bx = np.ascontiguousarray(boxes, dtype=np.float32).reshape(-1, 4)
    sc = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    n = sc.shape[0]
    cls = None if class_ids is None else np.ascontiguousarray(class_ids, dtype=np.int32)
    off = None if batch_offsets is None else np.ascontiguousarray(batch_offsets, dtype=np.int64)
    B = 1 if off is None else off.shape[0] - 1
    cap = B * max_out if max_out > 0 else n  # the layout of nms()
    keep = np.full(max(cap, 1), -1, dtype=np.int64)
    counts = np.zeros(max(B, 1), dtype=np.int64)
    tot = _load_base().cpu_baseline_nms(_ptr(bx, ctypes.c_float), _ptr(sc, ctypes.c_float), n,
                                        None if cls is None else _ptr(cls, ctypes.c_int32),
                                        None if off is None else _ptr(off, ctypes.c_int64), B,
                                        float(np.float32(iou_thr)), 0 if score_thr is None else 1,
                                        float(np.float32(score_thr if score_thr is not None else 0.0)),
                                        int(max_out), _ptr(keep, ctypes.c_int64), _ptr(counts, ctypes.c_int64))
    if tot < 0:
        raise ValueError("cpu_baseline_nms: invalid arguments")
    return keep, counts
