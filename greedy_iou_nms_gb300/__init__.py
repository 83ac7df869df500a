"""Greedy IoU NMS for GB300: thin Python binding of the libgbnms C ABI.

Every step of the computation runs in the library's CUDA kernels; this module
only marshals arguments.  PyTorch provides device memory and the stream.  The
raw entry points carry the same names as the C functions in include/gbnms.h
(`nms_run`, `nms_workspace_size`, `nms_status_string`, `nms_iou_mask`,
`nms_mask_row_words`) and take device pointers as integers.  `nms()` and
`iou_mask()` are the tensor-level conveniences.

There is no CPU fallback: if the shared library is missing or cannot load,
every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libgbnms.so")

NMS_OK = 0
NMS_ERR_INVALID_ARG = 1
NMS_ERR_WORKSPACE = 2
NMS_ERR_CAPACITY = 3
NMS_ERR_CUDA = 4
NMS_ERR_TIMEOUT = 5
NMS_DECAY_GAUSSIAN = 0  # nms_matrix_run decay kernels
NMS_DECAY_LINEAR = 1
NMS_MAX_SINGLE_N = 1 << 18

EXPORTED = ("nms_status_string", "nms_workspace_size", "nms_run", "nms_fast_run", "nms_run_timed",
            "nms_matrix_workspace_size", "nms_matrix_run", "nms_mask_row_words", "nms_iou_mask",
            "nms_resolve_mask", "nms_resolve_mask_noalloc", "nms_decode_workspace_size", "nms_decode_boxes7",
            "nms_boxes7_workspace_size", "nms_boxes7_run", "nms_mapped_pointer", "nms_copy", "nms_lane_workspace_size",
            "nms_lane_run")
NMS_NOALLOC_MAX_N = 16384
NMS_LANE_VALUES = 77  # values of one lane candidate (nms_lane_run)
NMS_LANE_ROWS = 72
NMS_LANE_MAX_N = 16384
NMS_DECODE_MAX_ANCHORS = 1 << 20
NMS_DECODE_MAX_CLASSES = 384
NMS_DECODE_MAX_BATCH = 65535

_lib = None


class NmsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {nms_status_string(code)} ({code})")


def build(force: bool = False) -> str:
    """Compile libgbnms.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def load():
    """Load libgbnms.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libgbnms.so not built at {LIB_PATH}: call greedy_iou_nms_gb300.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.nms_status_string.argtypes = [ctypes.c_int]
    lib.nms_status_string.restype = ctypes.c_char_p
    lib.nms_workspace_size.argtypes = [i64, i32, i32, ctypes.POINTER(sz)]
    lib.nms_workspace_size.restype = ctypes.c_int
    lib.nms_run.argtypes = [vp, vp, i64, vp, i32, vp, i32, f32, f32, i32, vp, i64, vp, vp, vp, sz, vp]
    lib.nms_run.restype = ctypes.c_int
    lib.nms_matrix_workspace_size.argtypes = [i64, ctypes.POINTER(sz)]
    lib.nms_matrix_workspace_size.restype = ctypes.c_int
    lib.nms_matrix_run.argtypes = [vp, vp, i64, i32, f32, f32, f32, i32, vp, vp, i64, vp, vp, vp, sz, vp]
    lib.nms_matrix_run.restype = ctypes.c_int
    lib.nms_fast_run.argtypes = lib.nms_run.argtypes
    lib.nms_fast_run.restype = ctypes.c_int
    lib.nms_run_timed.argtypes = [vp, vp, i64, vp, i32, vp, i32, f32, f32, i32, vp, i64, vp, vp, vp,
                                  sz, vp, ctypes.POINTER(vp), i32]
    lib.nms_run_timed.restype = ctypes.c_int
    lib.nms_mask_row_words.argtypes = [i64]
    lib.nms_mask_row_words.restype = i64
    lib.nms_iou_mask.argtypes = [vp, i64, f32, vp, i64, vp]
    lib.nms_iou_mask.restype = ctypes.c_int
    lib.nms_resolve_mask.argtypes = [vp, i64, vp, i32, vp, vp, vp, sz, vp]
    lib.nms_resolve_mask.restype = ctypes.c_int
    lib.nms_resolve_mask_noalloc.argtypes = [vp, i64, vp, i32, vp, vp, vp]
    lib.nms_resolve_mask_noalloc.restype = ctypes.c_int
    lib.nms_decode_workspace_size.argtypes = [i32, i32, ctypes.POINTER(sz)]
    lib.nms_decode_workspace_size.restype = ctypes.c_int
    lib.nms_decode_boxes7.argtypes = [vp, i32, i32, i32, f32, i32, vp, vp, vp, sz, vp]
    lib.nms_decode_boxes7.restype = ctypes.c_int
    lib.nms_boxes7_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
    lib.nms_boxes7_workspace_size.restype = ctypes.c_int
    lib.nms_boxes7_run.argtypes = [vp, i32, i32, i32, f32, i32, vp, vp, sz, vp]
    lib.nms_boxes7_run.restype = ctypes.c_int
    lib.nms_mapped_pointer.argtypes = [vp, ctypes.POINTER(vp)]
    lib.nms_mapped_pointer.restype = ctypes.c_int
    lib.nms_copy.argtypes = [vp, vp, sz, vp]
    lib.nms_copy.restype = ctypes.c_int
    lib.nms_lane_workspace_size.argtypes = [i64, ctypes.POINTER(sz)]
    lib.nms_lane_workspace_size.restype = ctypes.c_int
    lib.nms_lane_run.argtypes = [vp, vp, i64, f32, i32, vp, i64, vp, vp, vp, sz, vp]
    lib.nms_lane_run.restype = ctypes.c_int
    _lib = lib
    return lib


# ------------------------------------------------------------- raw C entries

def nms_status_string(code: int) -> str:
    return load().nms_status_string(int(code)).decode()


def nms_mapped_pointer(host_ptr: int) -> Optional[int]:
    """Device address of mapped page-locked host memory, or None when host_ptr
    is not such memory."""
    out = ctypes.c_void_p()
    st = load().nms_mapped_pointer(ctypes.c_void_p(host_ptr), ctypes.byref(out))
    return out.value if st == NMS_OK and out.value else None


def nms_copy(dst: int, src: int, nbytes: int, stream: int) -> int:
    return load().nms_copy(dst or None, src or None, int(nbytes), stream or None)


def nms_workspace_size(n: int, batch: int = 0, num_classes: int = 0) -> int:
    out = ctypes.c_size_t(0)
    st = load().nms_workspace_size(int(n), int(batch), int(num_classes), ctypes.byref(out))
    if st != NMS_OK:
        raise NmsError(st, "nms_workspace_size")
    return int(out.value)


def nms_mask_row_words(n: int) -> int:
    return int(load().nms_mask_row_words(int(n)))


def nms_run(boxes: int, scores: int, n: int, class_ids: int, num_classes: int,
            batch_offsets: int, batch: int, iou_thr: float, score_thr: float, max_out: int,
            keep: int, keep_cap: int, counts: int, dev_status: int, workspace: int,
            workspace_bytes: int, stream: int) -> int:
    """The C entry point with device addresses as ints (0 = NULL).  Returns the status code."""
    return load().nms_run(boxes or None, scores or None, int(n), class_ids or None,
                          int(num_classes), batch_offsets or None, int(batch), float(iou_thr),
                          float(score_thr), int(max_out), keep or None, int(keep_cap),
                          counts or None, dev_status or None, workspace or None,
                          int(workspace_bytes), stream or None)


def nms_fast_run(boxes: int, scores: int, n: int, class_ids: int, num_classes: int,
                 batch_offsets: int, batch: int, iou_thr: float, score_thr: float, max_out: int,
                 keep: int, keep_cap: int, counts: int, dev_status: int, workspace: int,
                 workspace_bytes: int, stream: int) -> int:
    """Fast NMS through the C entry point (arguments as nms_run)."""
    return load().nms_fast_run(boxes or None, scores or None, int(n), class_ids or None,
                               int(num_classes), batch_offsets or None, int(batch), float(iou_thr),
                               float(score_thr), int(max_out), keep or None, int(keep_cap),
                               counts or None, dev_status or None, workspace or None,
                               int(workspace_bytes), stream or None)


def nms_matrix_workspace_size(n: int) -> int:
    out = ctypes.c_size_t(0)
    st = load().nms_matrix_workspace_size(int(n), ctypes.byref(out))
    if st != NMS_OK:
        raise NmsError(st, "nms_matrix_workspace_size")
    return out.value


def nms_matrix_run(boxes: int, scores: int, n: int, decay: int, sigma: float, score_thr: float,
                   decay_thr: float, max_out: int, keep: int, keep_scores: int, keep_cap: int, count: int,
                   dev_status: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """Matrix NMS through the C entry point (device addresses as ints; decay is
    NMS_DECAY_GAUSSIAN or NMS_DECAY_LINEAR)."""
    return load().nms_matrix_run(boxes or None, scores or None, int(n), int(decay), float(sigma), float(score_thr),
                                 float(decay_thr), int(max_out), keep or None, keep_scores or None,
                                 int(keep_cap), count or None, dev_status or None, workspace or None,
                                 int(workspace_bytes), stream or None)


def nms_lane_workspace_size(n: int) -> int:
    b = ctypes.c_size_t(0)
    st = load().nms_lane_workspace_size(int(n), ctypes.byref(b))
    if st != NMS_OK:
        raise NmsError(st, "nms_lane_workspace_size")
    return int(b.value)


def nms_lane_run(props: int, scores: int, n: int, dist_thr: float, max_out: int, keep: int, keep_cap: int,
                 count: int, dev_status: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().nms_lane_run(props or None, scores or None, int(n), float(dist_thr), int(max_out), keep or None,
                               int(keep_cap), count or None, dev_status or None, workspace or None,
                               int(workspace_bytes), stream or None)


def lane_nms(props, scores, dist_thr: float, *, max_out: int = 0):
    """Greedy NMS of lane candidates (CUDA tensors props [n, 77], scores [n]):
    int64 kept indices in score order.  Synchronises the current stream once."""
    torch = _torch()
    if not (props.is_cuda and scores.is_cuda):
        raise ValueError("lane_nms: props and scores must be CUDA tensors")
    props = props.contiguous()
    scores = scores.contiguous()
    n = scores.shape[0]
    cap = max(keep_capacity(n, None, max_out), 1)
    keep = torch.empty(cap, dtype=torch.int64, device=props.device)
    count = torch.empty(1, dtype=torch.int64, device=props.device)
    wsb = nms_lane_workspace_size(n)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=props.device)
    st = nms_lane_run(props.data_ptr() if n else 0, scores.data_ptr() if n else 0, n, dist_thr, max_out,
                      keep.data_ptr(), cap, count.data_ptr(), 0, ws.data_ptr(), wsb,
                      torch.cuda.current_stream(props.device).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_lane_run")
    return keep[: int(count.item())]


def matrix_nms(boxes, scores, decay_thr: float, *, sigma: float = 0.5, decay: str = "gaussian",
               score_thr: Optional[float] = None, max_out: int = 0):
    """Matrix NMS on CUDA tensors with the Gaussian or the linear decay: (kept
    int64 indices in score order, their float32 final scores).  Synchronises
    the current stream once."""
    if decay not in ("gaussian", "linear"):
        raise ValueError("matrix_nms: decay must be 'gaussian' or 'linear'")
    torch = _torch()
    if not (boxes.is_cuda and scores.is_cuda):
        raise ValueError("matrix_nms: boxes and scores must be CUDA tensors")
    boxes = boxes.contiguous()
    scores = scores.contiguous()
    n = scores.shape[0]
    dev = boxes.device
    cap = keep_capacity(n, None, max_out)
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
    ks = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    count = torch.empty(1, dtype=torch.int64, device=dev)
    ws_bytes = nms_matrix_workspace_size(n)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    st = nms_matrix_run(boxes.data_ptr() if n else 0, scores.data_ptr() if n else 0, n,
                        NMS_DECAY_LINEAR if decay == "linear" else NMS_DECAY_GAUSSIAN, sigma,
                        -math.inf if score_thr is None else score_thr, decay_thr, max_out, keep.data_ptr(),
                        ks.data_ptr(), cap, count.data_ptr(), 0, ws.data_ptr(), ws_bytes,
                        torch.cuda.current_stream(dev).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_matrix_run")
    k = int(count.item())
    return keep[:k], ks[:k]


def nms_run_timed(boxes: int, scores: int, n: int, class_ids: int, num_classes: int,
                  batch_offsets: int, batch: int, iou_thr: float, score_thr: float, max_out: int,
                  keep: int, keep_cap: int, counts: int, dev_status: int, workspace: int,
                  workspace_bytes: int, stream: int, events) -> int:
    """nms_run that also records the given CUDA events (handles as ints, or
    objects with a ``cuda_event`` handle such as torch.cuda.Event) between its
    stages: before the first kernel, then after each stage.  The events must
    exist already (a torch.cuda.Event creates its handle at its first record)."""
    handles = [e if isinstance(e, int) else int(e.cuda_event) for e in events]
    if not all(handles):
        raise ValueError("nms_run_timed: every event must already be created")
    arr = (ctypes.c_void_p * max(len(handles), 1))(*[h or None for h in handles])
    return load().nms_run_timed(boxes or None, scores or None, int(n), class_ids or None,
                                int(num_classes), batch_offsets or None, int(batch), float(iou_thr),
                                float(score_thr), int(max_out), keep or None, int(keep_cap),
                                counts or None, dev_status or None, workspace or None,
                                int(workspace_bytes), stream or None, arr, len(handles))


def nms_iou_mask(boxes_sorted: int, n: int, iou_thr: float, mask: int, mask_words: int,
                 stream: int) -> int:
    return load().nms_iou_mask(boxes_sorted or None, int(n), float(iou_thr), mask or None,
                               int(mask_words), stream or None)


def nms_resolve_mask(mask: int, n: int, perm: int, max_out: int, keep: int, count: int,
                     workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().nms_resolve_mask(mask or None, int(n), perm or None, int(max_out), keep or None,
                                   count or None, workspace or None, int(workspace_bytes),
                                   stream or None)


def nms_resolve_mask_noalloc(mask: int, n: int, perm: int, max_out: int, keep: int, count: int,
                             stream: int) -> int:
    """nms_resolve_mask without a workspace: the resolve keeps all its state
    in the shared memory of its one thread block, so the call allocates
    nothing and holds nothing between calls; n <= NMS_NOALLOC_MAX_N."""
    return load().nms_resolve_mask_noalloc(mask or None, int(n), perm or None, int(max_out),
                                           keep or None, count or None, stream or None)


# ----------------------------------------------------------- tensor helpers

def _torch():
    import torch
    return torch


def keep_capacity(n: int, batch: Optional[int], max_out: int) -> int:
    b = 1 if batch is None else batch
    if max_out > 0:
        return min(n, max_out) if batch is None else b * max_out
    return n


class Workspace:
    """A reusable device workspace (a torch uint8 tensor) sized for nms_run."""

    def __init__(self, n: int, batch: int = 0, num_classes: int = 0, device="cuda"):
        torch = _torch()
        self.bytes = nms_workspace_size(n, batch, num_classes)
        self.tensor = torch.empty(max(self.bytes, 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()


def nms(boxes, scores, iou_thr: float, *, class_ids=None, num_classes: Optional[int] = None,
        batch_offsets=None, score_thr: Optional[float] = None, max_out: int = 0,
        workspace: Optional[Workspace] = None, return_counts: bool = False, fast: bool = False):
    """Greedy IoU NMS on CUDA tensors.

    boxes [n,4] fp32 xyxy and scores [n] fp32 on one CUDA device; class_ids
    int32 [n] (optional, with num_classes), batch_offsets int64 [B+1]
    (optional).  Returns the int64 kept indices: for one image a 1-D tensor in
    score order; with batch_offsets a list of per-image tensors.  With
    return_counts=True also returns the device counts tensor; fast=True runs
    Fast NMS (nms_fast_run) instead of greedy NMS.  Runs on the current stream
    and synchronises it once to read the counts.
    """
    torch = _torch()
    if not (boxes.is_cuda and scores.is_cuda):
        raise ValueError("nms: boxes and scores must be CUDA tensors")
    boxes = boxes.contiguous()
    scores = scores.contiguous()
    if boxes.dtype != torch.float32 or scores.dtype != torch.float32:
        raise ValueError("nms: boxes and scores must be float32")
    n = scores.shape[0]
    if boxes.shape != (n, 4):
        raise ValueError("nms: boxes must be [n, 4]")
    dev = boxes.device
    cls_ptr, C = 0, 0
    if class_ids is not None:
        class_ids = class_ids.to(device=dev, dtype=torch.int32).contiguous()
        C = int(num_classes) if num_classes is not None else int(class_ids.max().item()) + 1 if n else 1
        cls_ptr = class_ids.data_ptr()
    off_ptr, B = 0, 0
    if batch_offsets is not None:
        batch_offsets = batch_offsets.to(device=dev, dtype=torch.int64).contiguous()
        B = batch_offsets.shape[0] - 1
        off_ptr = batch_offsets.data_ptr()
    cap = keep_capacity(n, B if batch_offsets is not None else None, max_out)
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
    counts = torch.empty(max(B, 1), dtype=torch.int64, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else Workspace(n, B, C, device=dev)
    st = (nms_fast_run if fast else nms_run)(boxes.data_ptr() if n else 0, scores.data_ptr() if n else 0, n, cls_ptr, C,
                 off_ptr, B, iou_thr, -math.inf if score_thr is None else score_thr, max_out,
                 keep.data_ptr(), cap, counts.data_ptr(), status.data_ptr(), ws.ptr, ws.bytes,
                 torch.cuda.current_stream(dev).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_run")
    cnt = counts.cpu()
    dst = int(status.item())
    if dst != NMS_OK:
        raise NmsError(dst, "nms_run (device)")
    if batch_offsets is None:
        out = keep[: int(cnt[0])]
    else:
        offs = batch_offsets.cpu()
        out = []
        for b in range(B):
            base = b * max_out if max_out > 0 else int(offs[b])
            out.append(keep[base: base + int(cnt[b])])
    return (out, counts) if return_counts else out


class HostPipeline:
    """Greedy NMS of one image held in host memory, replayed as one CUDA graph
    per call.

    The input is one pinned buffer: n boxes (xyxy fp32) followed by n scores;
    write them through ``boxes`` / ``scores`` (numpy views of the first n
    entries, see ``set_n``) or ``load``.  ``run`` replays the graph captured
    for (n, iou_thr, score_thr, max_out) (capturing it on first use, after one
    plain call that also warms the library up), waits for it and returns the
    kept indices: a numpy view of the pinned output buffer (the count, then
    the indices), valid until the next call.

    With ``zero_copy`` (the default, when the pinned buffers are mapped into
    the device address space) the kernels move the data across the host link
    themselves: a copy kernel (nms_copy) stages the input into device memory in
    one pass, and the resolve writes the count and the kept indices into the
    pinned output.  Otherwise the graph is a host->device copy of the input,
    the kernels and a device->host copy of the count and the output capacity.
    """

    def __init__(self, n_max: int, device="cuda", zero_copy: bool = True):
        torch = _torch()
        self.n_max = int(n_max)
        self.device = torch.device(device)
        # 16 spare bytes: the staging copy moves whole 16-byte words
        self._h_in = torch.empty(5 * self.n_max + 4, dtype=torch.float32).pin_memory()
        self._h_out = torch.empty(self.n_max + 1, dtype=torch.int64).pin_memory()
        self._status = torch.empty(1, dtype=torch.int32, device=self.device)
        self._out_np = self._h_out.numpy()
        self.workspace = Workspace(self.n_max, device=self.device)
        self._graphs = {}
        self._d_in = torch.empty(5 * self.n_max + 4, dtype=torch.float32, device=self.device)
        self._in_addr = self._d_in.data_ptr()
        self.zero_copy = False
        if zero_copy:
            din, dout = nms_mapped_pointer(self._h_in.data_ptr()), nms_mapped_pointer(self._h_out.data_ptr())
            if din is not None and dout is not None:
                self.zero_copy = True
                self._h_in_dev, self._out_addr = din, dout
        if not self.zero_copy:
            self._d_out = torch.empty(self.n_max + 1, dtype=torch.int64, device=self.device)
            self._out_addr = self._d_out.data_ptr()
        self.set_n(self.n_max)

    def set_n(self, n: int) -> None:
        """Use the first n boxes: boxes is [n,4] at the start of the input
        buffer, scores [n] right after them (16n bytes in: 16-byte aligned)."""
        if not 0 <= n <= self.n_max:
            raise ValueError("HostPipeline: n out of range")
        self.n = int(n)
        flat = self._h_in.numpy()
        self.boxes = flat[: 4 * self.n].reshape(self.n, 4)
        self.scores = flat[4 * self.n: 5 * self.n]

    def load(self, boxes, scores) -> None:
        import numpy as np
        n = len(scores)
        self.set_n(n)
        self.boxes[...] = np.asarray(boxes, dtype=np.float32).reshape(n, 4)
        self.scores[...] = np.asarray(scores, dtype=np.float32)

    @property
    def in_bytes(self) -> int:
        """Input bytes that cross to the device per call."""
        return 20 * self.n

    def out_bytes(self, max_out: int = 0, kept: Optional[int] = None) -> int:
        """Output bytes that cross to the host per call: the count and the
        kept indices written in place (zero-copy; `kept` from the last run),
        else the count and the whole output capacity copied."""
        if self.zero_copy:
            return 8 * (1 + (int(self._out_np[0]) if kept is None else int(kept)))
        return 8 * (1 + keep_capacity(self.n, None, max_out))

    def _enqueue(self, n, iou_thr, score_thr, max_out, stream):
        cap = keep_capacity(n, None, max_out)
        if self.zero_copy:
            st = nms_copy(self._d_in.data_ptr(), self._h_in_dev, (20 * n + 15) // 16 * 16, stream.cuda_stream)
            if st != NMS_OK:
                raise NmsError(st, "nms_copy")
        else:
            self._d_in[: 5 * n].copy_(self._h_in[: 5 * n], non_blocking=True)
        base_in, base_out = self._in_addr, self._out_addr
        st = nms_run(base_in if n else 0, base_in + 16 * n if n else 0, n, 0, 0, 0, 0, iou_thr,
                     -math.inf if score_thr is None else score_thr, max_out, base_out + 8,
                     max(cap, 1), base_out, self._status.data_ptr(), self.workspace.ptr,
                     self.workspace.bytes, stream.cuda_stream)
        if st != NMS_OK:
            raise NmsError(st, "nms_run")
        if not self.zero_copy:
            self._h_out[: cap + 1].copy_(self._d_out[: cap + 1], non_blocking=True)

    def launch(self, iou_thr: float, score_thr: Optional[float] = None, max_out: int = 0) -> None:
        """Enqueue one call on the current stream (the captured graph) without
        waiting; ``result`` waits and returns the kept indices."""
        torch = _torch()
        key = (self.n, float(iou_thr), score_thr, int(max_out))
        graph = self._graphs.get(key)
        if graph is None:
            stream = torch.cuda.current_stream(self.device)
            self._enqueue(self.n, iou_thr, score_thr, max_out, stream)  # checks and warms up
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                self._enqueue(self.n, iou_thr, score_thr, max_out,
                              torch.cuda.current_stream(self.device))
            self._graphs[key] = graph
        graph.replay()

    def result(self):
        torch = _torch()
        torch.cuda.current_stream(self.device).synchronize()
        out = self._out_np
        return out[1: 1 + int(out[0])]

    def run(self, iou_thr: float, score_thr: Optional[float] = None, max_out: int = 0):
        self.launch(iou_thr, score_thr, max_out)
        return self.result()


def iou_mask(boxes_sorted, iou_thr: float):
    """Suppression bitmask of score-sorted boxes: int64 tensor [n, nms_mask_row_words(n)]
    holding the uint64 words (bit j%64 of word j//64 of row i: j > i and IoU > thr).
    Words left of each row's diagonal tile are zero here."""
    torch = _torch()
    boxes_sorted = boxes_sorted.contiguous()
    n = boxes_sorted.shape[0]
    ldw = nms_mask_row_words(n)
    mask = torch.zeros((n, max(ldw, 1)), dtype=torch.int64, device=boxes_sorted.device)
    st = nms_iou_mask(boxes_sorted.data_ptr() if n else 0, n, iou_thr, mask.data_ptr(),
                      mask.numel(), torch.cuda.current_stream(boxes_sorted.device).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_iou_mask")
    return mask[:, :ldw]


def resolve_mask(mask, max_out: int = 0, perm=None, workspace: Optional[Workspace] = None):
    """Kept sorted positions (or perm entries) of a mask in the iou_mask layout."""
    torch = _torch()
    n = mask.shape[0]
    cap = min(n, max_out) if max_out > 0 else n
    keep = torch.empty(max(cap, 1), dtype=torch.int64, device=mask.device)
    count = torch.empty(1, dtype=torch.int64, device=mask.device)
    if perm is not None:
        perm = perm.to(device=mask.device, dtype=torch.int32).contiguous()
    ws = workspace if workspace is not None else Workspace(n, device=mask.device)
    st = nms_resolve_mask(mask.data_ptr() if n else 0, n, perm.data_ptr() if perm is not None else 0,
                          max_out, keep.data_ptr(), count.data_ptr(), ws.ptr, ws.bytes,
                          torch.cuda.current_stream(mask.device).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_resolve_mask")
    return keep[: int(count.item())]


# ------------------------------------------- front end for YOLO-shaped outputs

def nms_decode_workspace_size(batch: int, anchors: int) -> int:
    out = ctypes.c_size_t(0)
    st = load().nms_decode_workspace_size(int(batch), int(anchors), ctypes.byref(out))
    if st != NMS_OK:
        raise NmsError(st, "nms_decode_workspace_size")
    return int(out.value)


def nms_decode_boxes7(preds: int, batch: int, anchors: int, num_classes: int, conf_thr: float, max_objects: int,
                      buffers: int, dev_status: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """The C entry point (device addresses as ints)."""
    return load().nms_decode_boxes7(preds or None, int(batch), int(anchors), int(num_classes), float(conf_thr),
                                    int(max_objects), buffers or None, dev_status or None, workspace or None,
                                    int(workspace_bytes), stream or None)


def nms_boxes7_workspace_size(batch: int, max_objects: int, num_classes: int) -> int:
    out = ctypes.c_size_t(0)
    st = load().nms_boxes7_workspace_size(int(batch), int(max_objects), int(num_classes), ctypes.byref(out))
    if st != NMS_OK:
        raise NmsError(st, "nms_boxes7_workspace_size")
    return int(out.value)


def nms_boxes7_run(buffers: int, batch: int, max_objects: int, num_classes: int, iou_thr: float, fast: int,
                   dev_status: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """The C entry point (device addresses as ints)."""
    return load().nms_boxes7_run(buffers or None, int(batch), int(max_objects), int(num_classes), float(iou_thr),
                                 int(fast), dev_status or None, workspace or None, int(workspace_bytes),
                                 stream or None)


def decode_boxes7(preds, conf_thr: float, max_objects: int):
    """Count-header buffers [batch, 1 + 7 * max_objects] (float32, CUDA) from
    YOLO-shaped predictions [batch, anchors, 5 + classes] (float32, CUDA).
    Rows past the candidates are zero."""
    torch = _torch()
    if not preds.is_cuda or preds.dtype != torch.float32 or preds.dim() != 3 or preds.shape[2] < 6:
        raise ValueError("decode_boxes7: preds must be a float32 CUDA tensor [batch, anchors, 5 + classes]")
    preds = preds.contiguous()
    batch, anchors, width = preds.shape
    dev = preds.device
    out = torch.zeros((batch, 1 + 7 * max_objects), dtype=torch.float32, device=dev)
    wsb = nms_decode_workspace_size(batch, anchors)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = nms_decode_boxes7(preds.data_ptr(), batch, anchors, width - 5, conf_thr, max_objects, out.data_ptr(),
                           status.data_ptr(), ws.data_ptr(), wsb, torch.cuda.current_stream(dev).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_decode_boxes7")
    dst = int(status.item())
    if dst != NMS_OK:
        raise NmsError(dst, "nms_decode_boxes7 (device)")
    return out


def boxes7_nms(buffers, num_classes: int, iou_thr: float, *, fast: bool = False):
    """NMS in place over count-header buffers [batch, 1 + 7 * max_objects]
    (float32, CUDA): keep_flag of the taking-part rows becomes 1 or 0.
    Synchronises the current stream once to read the device status."""
    torch = _torch()
    if not buffers.is_cuda or buffers.dtype != torch.float32 or buffers.dim() != 2 or not buffers.is_contiguous():
        raise ValueError("boxes7_nms: buffers must be a contiguous float32 CUDA tensor [batch, 1 + 7 * max_objects]")
    batch, width = buffers.shape
    if (width - 1) % 7:
        raise ValueError("boxes7_nms: the row length must be 1 + 7 * max_objects")
    max_objects = (width - 1) // 7
    dev = buffers.device
    wsb = nms_boxes7_workspace_size(batch, max_objects, num_classes)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = nms_boxes7_run(buffers.data_ptr(), batch, max_objects, num_classes, iou_thr, 1 if fast else 0,
                        status.data_ptr(), ws.data_ptr(), wsb, torch.cuda.current_stream(dev).cuda_stream)
    if st != NMS_OK:
        raise NmsError(st, "nms_boxes7_run")
    dst = int(status.item())
    if dst != NMS_OK:
        raise NmsError(dst, "nms_boxes7_run (device)")
    return buffers
