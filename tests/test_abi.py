"""The C-ABI library: builds, loads, exports what include/gbnms.h declares, and
rejects bad arguments on the host before touching the device (no GPU needed)."""
import ctypes
import math
import os
import re

import pytest

import greedy_iou_nms_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    g.build()
    return g.load()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(nms_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert declared == set(g.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in ((0, "NMS_OK"), (1, "NMS_ERR_INVALID_ARG"), (2, "NMS_ERR_WORKSPACE"),
                       (3, "NMS_ERR_CAPACITY"), (4, "NMS_ERR_CUDA"), (5, "NMS_ERR_TIMEOUT")):
        assert g.nms_status_string(code) == name
    assert g.nms_status_string(99) == "NMS_ERR_UNKNOWN"


def test_workspace_size(lib):
    # Single path holds the mask: n * 4*ceil(n/256) words.
    for n in (0, 1, 255, 256, 257, 8192):
        ws = g.nms_workspace_size(n)
        assert ws >= 8 * n * g.nms_mask_row_words(n)
    assert g.nms_workspace_size(1 << 18) > 0
    with pytest.raises(g.NmsError) as e:
        g.nms_workspace_size((1 << 18) + 1)
    assert e.value.code == g.NMS_ERR_CAPACITY
    # Batched path: linear in n.
    b1 = g.nms_workspace_size(100000, 16, 80)
    b2 = g.nms_workspace_size(200000, 16, 80)
    assert b2 < 2.2 * b1
    with pytest.raises(g.NmsError):
        g.nms_workspace_size(-1)


def test_matrix_and_front_end_workspace_sizes(lib):
    # Matrix NMS: the pair list of pass A (about 96 pairs a box plus a floor,
    # 12 bytes each, never more than the pairs there are) dominates.
    for n in (2, 1000, 8192, 65536):
        ws = g.nms_matrix_workspace_size(n)
        pairs = min(n * (n - 1) // 2, 96 * n + (1 << 20))
        assert ws >= 12 * pairs + 40 * n
    assert g.nms_matrix_workspace_size(0) > 0
    with pytest.raises(g.NmsError) as e:
        g.nms_matrix_workspace_size((1 << 18) + 1)
    assert e.value.code == g.NMS_ERR_CAPACITY
    # Front end: 7 floats of staging per anchor slot, linear in batch.
    d1 = g.nms_decode_workspace_size(1, 25200)
    d16 = g.nms_decode_workspace_size(16, 25200)
    assert d1 >= 7 * 4 * 25200 and 15 * d1 <= d16 <= 17 * d1


def test_mapped_pointer_rejects_other_memory(lib):
    # NULL and ordinary (unregistered) host memory have no device mapping; the
    # query enqueues nothing and needs no GPU to say so.
    import numpy as np
    assert g.nms_mapped_pointer(0) is None
    assert g.nms_mapped_pointer(np.zeros(16, np.float32).ctypes.data) is None


def test_copy_entry_validation(lib):
    # NULL pointers with bytes to copy are refused on the host; nothing to
    # copy enqueues nothing (no GPU needed for either).
    assert g.nms_copy(0, 0, 0, 0) == g.NMS_OK
    assert g.nms_copy(0, 16, 16, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_copy(16, 0, 16, 0) == g.NMS_ERR_INVALID_ARG


def test_mask_row_words(lib):
    assert g.nms_mask_row_words(0) == 0
    assert g.nms_mask_row_words(1) == 4
    assert g.nms_mask_row_words(256) == 4
    assert g.nms_mask_row_words(257) == 8


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on these paths


def _run(**kw):
    a = dict(boxes=FAKE, scores=FAKE, n=10, class_ids=0, num_classes=0, batch_offsets=0, batch=0,
             iou_thr=0.5, score_thr=-math.inf, max_out=0, keep=FAKE, keep_cap=10, counts=FAKE,
             dev_status=0, workspace=FAKE, workspace_bytes=0, stream=0)
    a.update(kw)
    return g.nms_run(**a)


def test_host_validation(lib):
    ws = g.nms_workspace_size(10)
    assert _run(n=-1) == g.NMS_ERR_INVALID_ARG
    assert _run(iou_thr=math.nan, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(score_thr=math.nan, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(boxes=0, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(boxes=FAKE + 4, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG  # not 16-B aligned
    assert _run(keep=0, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(counts=0, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(class_ids=FAKE, num_classes=0, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(batch_offsets=FAKE, batch=0, workspace_bytes=ws) == g.NMS_ERR_INVALID_ARG
    assert _run(keep_cap=9, workspace_bytes=ws) == g.NMS_ERR_CAPACITY
    assert _run(workspace_bytes=ws - 1) == g.NMS_ERR_WORKSPACE
    assert _run(workspace=0, workspace_bytes=ws) == g.NMS_ERR_WORKSPACE
    assert _run(workspace=FAKE + 8, workspace_bytes=ws) == g.NMS_ERR_WORKSPACE
    assert _run(n=(1 << 18) + 1, keep_cap=1 << 19, workspace_bytes=1 << 40) == g.NMS_ERR_CAPACITY
    # batched capacity: batch * max_out
    wsb = g.nms_workspace_size(10, 4, 3)
    assert _run(class_ids=FAKE, num_classes=3, batch_offsets=FAKE, batch=4, max_out=5,
                keep_cap=19, workspace_bytes=wsb) == g.NMS_ERR_CAPACITY


def test_timed_entry_validates_like_nms_run(lib):
    """nms_run_timed checks its arguments exactly as nms_run does, before any
    event is touched (the event handles here are fake and never used)."""
    ws = g.nms_workspace_size(10)
    a = dict(boxes=FAKE, scores=FAKE, n=10, class_ids=0, num_classes=0, batch_offsets=0, batch=0,
             iou_thr=0.5, score_thr=-math.inf, max_out=0, keep=FAKE, keep_cap=10, counts=FAKE,
             dev_status=0, workspace=FAKE, workspace_bytes=ws, stream=0)
    fake_events = [FAKE, FAKE, FAKE, FAKE]
    for bad, code in ((dict(n=-1), g.NMS_ERR_INVALID_ARG), (dict(iou_thr=math.nan), g.NMS_ERR_INVALID_ARG),
                      (dict(keep_cap=9), g.NMS_ERR_CAPACITY), (dict(workspace_bytes=ws - 1), g.NMS_ERR_WORKSPACE)):
        kw = dict(a, **bad)
        assert g.nms_run_timed(**kw, events=fake_events) == code
        assert g.nms_run(**kw) == code


def test_mask_entry_validation(lib):
    assert g.nms_iou_mask(FAKE, -1, 0.5, FAKE, 0, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_iou_mask(FAKE, 10, math.nan, FAKE, 40, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_iou_mask(0, 10, 0.5, FAKE, 40, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_iou_mask(FAKE, 10, 0.5, FAKE, 39, 0) == g.NMS_ERR_CAPACITY
    assert g.nms_iou_mask(FAKE, (1 << 18) + 1, 0.5, FAKE, 1 << 40, 0) == g.NMS_ERR_CAPACITY
    assert g.nms_iou_mask(0, 0, 0.5, 0, 0, 0) == g.NMS_OK


def test_resolve_entries_reject_misaligned_pointers(lib):
    """Both resolve entry points refuse, on the host, a count or keep that is
    not 8-byte aligned and a perm that is not 4-byte aligned (the resolve
    stores int64 and loads int32 there)."""
    ws = 1 << 20  # 256-byte aligned fake device address, never dereferenced
    big = 1 << 40
    for perm, keep, count in ((FAKE + 2, FAKE, FAKE), (FAKE, FAKE + 4, FAKE), (FAKE, FAKE, FAKE + 4), (0, FAKE, FAKE + 1)):
        assert g.nms_resolve_mask(FAKE, 100, perm, 0, keep, count, ws, big, 0) == g.NMS_ERR_INVALID_ARG
        assert g.nms_resolve_mask_noalloc(FAKE, 100, perm, 0, keep, count, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_resolve_mask(FAKE + 8, 100, 0, 0, FAKE, FAKE, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_resolve_mask_noalloc(FAKE + 8, 100, 0, 0, FAKE, FAKE, 0) == g.NMS_ERR_INVALID_ARG


def test_workspace_sizes_grow_with_n(lib):
    """A workspace sized for n serves every smaller call: the sizes never
    shrink as n grows (the pair list's capacity, one CTA's pairs times a
    factor up to 16384 boxes and the all-SM path's above, included), and
    the lane workspace holds the prepass's planes and second list besides
    the single-image regions."""
    sizes = [1, 63, 64, 65, 1000, 3000, 8192, 8193, 16384, 16385, 32768, 65536]
    for f, top in ((g.nms_workspace_size, 1 << 18), (g.nms_lane_workspace_size, g.NMS_LANE_MAX_N)):
        prev = 0
        for n in [x for x in sizes if x <= top]:
            b = f(n)
            assert b >= prev, (f.__name__, n)
            prev = b
    for n in (1000, 3000, 16384):
        assert g.nms_lane_workspace_size(n) > g.nms_workspace_size(n)


def test_lane_entry_validation(lib):
    ws = 1 << 20
    big = 1 << 40
    assert g.nms_lane_workspace_size(1000) > 0
    with pytest.raises(g.NmsError):
        g.nms_lane_workspace_size(g.NMS_LANE_MAX_N + 1)
    assert g.nms_lane_run(FAKE, FAKE, -1, 15.0, 0, FAKE, 10, FAKE, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(FAKE, FAKE, 10, math.nan, 0, FAKE, 10, FAKE, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(0, FAKE, 10, 15.0, 0, FAKE, 10, FAKE, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(FAKE + 2, FAKE, 10, 15.0, 0, FAKE, 10, FAKE, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(FAKE, FAKE, 10, 15.0, 0, FAKE + 4, 10, FAKE, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(FAKE, FAKE, 10, 15.0, 0, FAKE, 10, FAKE + 4, 0, ws, big, 0) == g.NMS_ERR_INVALID_ARG
    assert g.nms_lane_run(FAKE, FAKE, 10, 15.0, 0, FAKE, 9, FAKE, 0, ws, big, 0) == g.NMS_ERR_CAPACITY
    assert g.nms_lane_run(FAKE, FAKE, 10, 15.0, 3, FAKE, 3, FAKE, 0, 0, big, 0) == g.NMS_ERR_WORKSPACE
    assert g.nms_lane_run(FAKE, FAKE, 10, 15.0, 0, FAKE, 10, FAKE, 0, ws, 16, 0) == g.NMS_ERR_WORKSPACE
    assert g.nms_lane_run(FAKE, FAKE, g.NMS_LANE_MAX_N + 1, 15.0, 0, FAKE, big, FAKE, 0, ws, big, 0) == \
        g.NMS_ERR_CAPACITY


def test_no_cpu_fallback_when_library_missing(monkeypatch):
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", "/nonexistent/libgbnms.so")
    with pytest.raises(RuntimeError):
        g.load()


def test_matrix_entry_validation(lib):
    ws = g.nms_matrix_workspace_size(10)
    a = dict(boxes=FAKE, scores=FAKE, n=10, decay=g.NMS_DECAY_GAUSSIAN, sigma=0.5, score_thr=-math.inf,
             decay_thr=0.1, max_out=0,
             keep=FAKE, keep_scores=0, keep_cap=10, count=FAKE, dev_status=0, workspace=FAKE,
             workspace_bytes=ws, stream=0)
    for bad, code in ((dict(n=-1), g.NMS_ERR_INVALID_ARG), (dict(sigma=0.0), g.NMS_ERR_INVALID_ARG),
                      (dict(sigma=-1.0), g.NMS_ERR_INVALID_ARG), (dict(sigma=math.inf), g.NMS_ERR_INVALID_ARG),
                      (dict(decay_thr=math.nan), g.NMS_ERR_INVALID_ARG), (dict(boxes=FAKE + 4), g.NMS_ERR_INVALID_ARG),
                      (dict(keep_cap=9), g.NMS_ERR_CAPACITY), (dict(max_out=3, keep_cap=2), g.NMS_ERR_CAPACITY),
                      (dict(workspace_bytes=ws - 1), g.NMS_ERR_WORKSPACE), (dict(n=(1 << 18) + 1, keep_cap=1 << 19), g.NMS_ERR_CAPACITY),
                      (dict(decay=2), g.NMS_ERR_INVALID_ARG), (dict(decay=-1), g.NMS_ERR_INVALID_ARG),
                      (dict(decay=g.NMS_DECAY_LINEAR, keep_cap=9), g.NMS_ERR_CAPACITY),
                      (dict(decay=g.NMS_DECAY_LINEAR, decay_thr=math.nan), g.NMS_ERR_INVALID_ARG)):
        assert g.nms_matrix_run(**dict(a, **bad)) == code, bad
    with pytest.raises(g.NmsError):
        g.nms_matrix_workspace_size(-1)


def test_front_end_entry_validation(lib):
    ws = g.nms_decode_workspace_size(2, 100)
    a = dict(preds=FAKE, batch=2, anchors=100, num_classes=80, conf_thr=0.25, max_objects=10, buffers=FAKE,
             dev_status=0, workspace=FAKE, workspace_bytes=ws, stream=0)
    for bad, code in ((dict(batch=0), g.NMS_ERR_INVALID_ARG), (dict(anchors=-1), g.NMS_ERR_INVALID_ARG),
                      (dict(num_classes=0), g.NMS_ERR_INVALID_ARG), (dict(max_objects=-1), g.NMS_ERR_INVALID_ARG),
                      (dict(conf_thr=math.nan), g.NMS_ERR_INVALID_ARG), (dict(buffers=0), g.NMS_ERR_INVALID_ARG),
                      (dict(preds=FAKE + 2), g.NMS_ERR_INVALID_ARG),
                      (dict(anchors=g.NMS_DECODE_MAX_ANCHORS + 1), g.NMS_ERR_CAPACITY),
                      (dict(num_classes=g.NMS_DECODE_MAX_CLASSES + 1), g.NMS_ERR_CAPACITY),
                      (dict(batch=g.NMS_DECODE_MAX_BATCH + 1), g.NMS_ERR_CAPACITY),
                      (dict(workspace_bytes=ws - 1), g.NMS_ERR_WORKSPACE), (dict(workspace=FAKE + 8), g.NMS_ERR_WORKSPACE)):
        assert g.nms_decode_boxes7(**dict(a, **bad)) == code, bad
    wb = g.nms_boxes7_workspace_size(2, 10, 80)
    b = dict(buffers=FAKE, batch=2, max_objects=10, num_classes=80, iou_thr=0.5, fast=0, dev_status=0,
             workspace=FAKE, workspace_bytes=wb, stream=0)
    for bad, code in ((dict(batch=0), g.NMS_ERR_INVALID_ARG), (dict(num_classes=0), g.NMS_ERR_INVALID_ARG),
                      (dict(fast=2), g.NMS_ERR_INVALID_ARG), (dict(iou_thr=math.nan), g.NMS_ERR_INVALID_ARG),
                      (dict(buffers=0), g.NMS_ERR_INVALID_ARG), (dict(max_objects=-1), g.NMS_ERR_INVALID_ARG),
                      (dict(batch=1 << 20, max_objects=1 << 12), g.NMS_ERR_INVALID_ARG),
                      (dict(batch=g.NMS_DECODE_MAX_BATCH + 1), g.NMS_ERR_CAPACITY),
                      (dict(workspace_bytes=wb - 1), g.NMS_ERR_WORKSPACE)):
        assert g.nms_boxes7_run(**dict(b, **bad)) == code, bad
    with pytest.raises(g.NmsError):
        g.nms_decode_workspace_size(0, 10)
