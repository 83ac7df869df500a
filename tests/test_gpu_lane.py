"""GPU parity of lane-candidate NMS (nms_lane_run) with the oracle: kept
indices and their order bit-exact, on the seeded lane workloads, hand-worked
distances (constant offsets at the threshold, partial row overlaps), spans
that are fractional, negative or past the last row, non-finite x values in
covered rows, NaN scores, identical lanes, max_out, and sizes over several
64-lane tiles with a ragged tail."""
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


def _check(props, scores, thr, max_out=0):
    p = torch.from_numpy(np.ascontiguousarray(props, np.float32)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    got = g.lane_nms(p, s, thr, max_out=max_out).cpu().numpy()
    exp = oracle.lane_nms(props, scores, thr, max_out=max_out)
    assert got.tolist() == exp.tolist()
    return got


def _lane(x, start=0, length=72):
    p = np.zeros(77, np.float32)
    p[2], p[4] = start, length
    p[5:] = np.broadcast_to(np.asarray(x, np.float32), (72,))
    return p


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("n", [1, 63, 64, 65, 1000, 3000])
@pytest.mark.parametrize("thr", [5.0, 15.0, 40.0])
def test_workloads(seed, n, thr):
    props, scores = W.lanes(seed, n=n)
    _check(props, scores, thr)


@pytest.mark.parametrize("max_out", [1, 5, 50])
def test_max_out(max_out):
    props, scores = W.lanes(4, n=2000)
    k = _check(props, scores, 15.0, max_out=max_out)
    full = oracle.lane_nms(props, scores, 15.0)
    assert k.tolist() == full[:max_out].tolist()


def test_exact_distances_at_the_threshold():
    """Constant offsets 0, 1.5, 3, ..., so distances equal the threshold
    exactly (kept) or lie one ulp around it; partial overlaps whose far rows
    would otherwise decide."""
    r = np.arange(72, dtype=np.float32)
    props = np.stack([_lane(100 + r + 1.5 * i, start=(i * 7) % 30, length=72) for i in range(40)])
    s = np.linspace(0.9, 0.1, 40).astype(np.float32)
    for thr in (1.5, float(np.nextafter(np.float32(1.5), np.float32(2))), float(np.nextafter(np.float32(1.5),
                                                                                                np.float32(0))), 3.0):
        _check(props, s, thr)
    xb = (100 + r + 3).astype(np.float32)
    xb[:20] = 1e6
    props = np.stack([_lane(100 + r, 0, 40), _lane(xb, 20, 52), _lane(100 + r + 2.9, 10, 5)])
    _check(props, np.array([0.9, 0.8, 0.7], np.float32), 3.0)
    _check(props, np.array([0.9, 0.8, 0.7], np.float32), 3.1)


def test_spans_and_special_values():
    """Fractional, negative and overlong spans; NaN and infinite starts and
    lengths; NaN and infinite x in covered rows (the exact per-pair path) and
    in uncovered ones (ignored); NaN and -0 scores; identical lanes."""
    rng = np.random.default_rng(9)
    props, scores = W.lanes(9, n=600)
    props[::7, 2] += 0.6
    props[::11, 4] += 0.9
    props[3::13, 2] = -5
    props[5::17, 4] = 200
    props[7, 2] = np.nan
    props[8, 4] = np.inf
    props[9, 2] = -np.inf
    props[20, 5 + int(props[20, 2]) + 1] = np.nan  # covered row
    props[21, 5 + int(props[21, 2])] = np.inf
    props[22, 5:] = props[23, 5:] = props[24, 5:]
    props[22, 2:5] = props[23, 2:5] = props[24, 2:5]
    props[25, 5 + int(props[25, 2])] = -np.inf
    props[26, 5 + int(props[26, 2])] = -np.inf  # with 25: -inf - -inf is NaN in a common row
    props[26, 2:5] = props[25, 2:5]
    if props[30, 2] >= 1:
        props[30, 5] = np.nan  # uncovered row
    scores[40] = np.nan
    scores[41] = -0.0
    scores[42] = 0.0
    for thr in (5.0, 15.0, 1e30):
        _check(props, scores, thr)


def test_largest_and_empty():
    props, scores = W.lanes(2, n=g.NMS_LANE_MAX_N)
    _check(props, scores, 15.0)
    k = g.lane_nms(torch.zeros((0, 77), device="cuda"), torch.zeros(0, device="cuda"), 15.0)
    assert len(k) == 0


def test_repeat_calls_are_identical():
    props, scores = W.lanes(1, n=3000)
    a = _check(props, scores, 10.0)
    b = _check(props, scores, 10.0)
    assert a.tolist() == b.tolist()


def test_one_workspace_across_calls():
    """One workspace for calls of several sizes and densities in turn (lists
    that one CTA holds, lists that the all-SM passes 0 and 1 shrink into one
    CTA or leave longer, and lists longer than the workspace holds): every
    call zeroes the passes' byte planes and pair count again, so a byte left
    by an earlier call never removes a lane."""
    n_max = 3000
    wsb = g.nms_lane_workspace_size(n_max)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for seed, n, thr in [(0, 3000, 40.0), (1, 1000, 15.0), (2, 3000, 15.0), (3, 500, 5.0), (0, 3000, 40.0),
                         (1, 1000, 15.0)]:
        assert g.nms_lane_workspace_size(n) <= wsb
        props, scores = W.lanes(seed, n=n)
        p = torch.from_numpy(props).cuda()
        s = torch.from_numpy(scores).cuda()
        keep = torch.empty(n, dtype=torch.int64, device="cuda")
        count = torch.empty(1, dtype=torch.int64, device="cuda")
        st = g.nms_lane_run(p.data_ptr(), s.data_ptr(), n, thr, 0, keep.data_ptr(), n, count.data_ptr(), 0,
                            ws.data_ptr(), wsb, stream.cuda_stream)
        assert st == g.NMS_OK
        got = keep[: int(count.item())].cpu().numpy()
        assert got.tolist() == oracle.lane_nms(props, scores, thr).tolist(), (seed, n, thr)
