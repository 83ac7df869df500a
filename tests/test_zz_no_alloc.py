"""The allocation-free resolve entry point against the workspace one.

nms_resolve_mask_noalloc serves callers that cannot allocate device memory
where they run NMS (a plugin whose host framework owns all allocations, a
real-time loop with memory planned at start-up, a deployment that bans
allocation after initialisation).  It keeps all its state in the shared
memory of its one thread block and holds nothing between calls.  Two calls in
a row through the C ABI, on different masks, must each give exactly the keep
list and count of nms_resolve_mask (the workspace entry point, which today
runs the same resolve and leaves its workspace untouched) and, the check that
counts, of the oracle: calls in a row must be independent.  Keep indices are
integers, so the comparisons are exact, as in the other parity tests.  This
file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import greedy_iou_nms_gb300 as g
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _sorted_boxes(n, seed, span):
    rng = np.random.default_rng(seed)
    c = rng.uniform(0, span, (n, 2))
    wh = rng.uniform(2, 40, (n, 2))
    return np.concatenate([c - wh / 2, c + wh / 2], 1).astype(np.float32)


def _noalloc(mask, n, max_out):
    cap = min(n, max_out) if max_out > 0 else n
    keep = torch.full((max(cap, 1),), -1, dtype=torch.int64, device="cuda")
    count = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    st = g.nms_resolve_mask_noalloc(mask.data_ptr(), n, 0, max_out, keep.data_ptr(),
                                    count.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == g.NMS_OK, g.nms_status_string(st)
    return keep[: int(count.item())].cpu().numpy()


@pytest.mark.parametrize("n,span,max_out", [(5000, 300.0, 0), (16384, 1200.0, 777)])
def test_noalloc_matches_workspace_entry_point_twice(n, span, max_out):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    g.load()
    for call in range(2):  # two calls in a row, on different masks, are independent
        b = _sorted_boxes(n, 10 * n + call, span)
        m = g.iou_mask(torch.from_numpy(b).cuda(), 0.5)
        ref = g.resolve_mask(m, max_out=max_out).cpu().numpy()
        got = _noalloc(m, n, max_out)
        assert got.tolist() == ref.tolist()
        s = np.linspace(1.0, 0.0, n, dtype=np.float32)
        assert got.tolist() == oracle.nms_single(b, s, 0.5, max_out=max_out).tolist()


def test_noalloc_rejects_sizes_beyond_its_limit():
    g.build()
    g.load()
    n = g.NMS_NOALLOC_MAX_N + 1
    st = g.nms_resolve_mask_noalloc(1 << 20, n, 0, 0, 1 << 20, 1 << 20, 0)
    assert st == g.NMS_ERR_CAPACITY
