"""CPU model of the graph resolve's pass scheme, checked against the oracle.

The GPU resolve decides greedy NMS in rounds over the pair graph: one byte
per box holds the last pass that blocked it (plus 2, mod 256), one byte says
"removed"; in pass r a pair (s -> j) drops out when s is removed, removes j
when s is kept (s not removed, byte == r), and otherwise blocks j (byte =
r + 2) and stays.  Pass 0 starts from the bytes 2 (a box with a source) and 0;
passes 0 and 1 may also run in bulk first (pass 0 removes the targets of the
sources without a source, pass 1 keeps nothing: it drops the pairs whose
source pass 0 removed and blocks the targets of the rest), as the all-SM
prepass of lane NMS and the cluster prologue of the box path do.

This models that algorithm, not the kernels: within a pass the pairs are
visited in a random order, and each store of the pass becomes visible to the
later readers of that pass at once or only after the pass, at random, as
stores racing in the same pass may.  The kept boxes must equal the oracle's
greedy result on random small inputs, and on a dependency chain long enough
to wrap the pass byte."""
import numpy as np
import pytest

import oracle


def _pairs(boxes_sorted, thr):
    m = oracle.mask(boxes_sorted, thr)
    n = len(boxes_sorted)
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(n, -1)[:, :n]
    i, j = np.nonzero(bits)
    return list(zip(i.tolist(), j.tolist()))


def _resolve_model(n, pairs, rng, bulk01):
    has = [False] * n
    for _, j in pairs:
        has[j] = True
    fl = [2 if h else 0 for h in has]
    rm = [False] * n
    live = list(pairs)
    r = 0
    if bulk01:
        for i, j in pairs:
            if not has[i]:
                rm[j] = True
        live = [(i, j) for i, j in pairs if has[i] and not rm[i]]
        for _, j in live:
            fl[j] = 3
        r = 2
    while live:
        rng.shuffle(live)
        late = []  # stores of this pass that its later readers do not see
        out = []
        kept_f = r % 256
        for i, j in live:
            if rm[i]:
                continue
            if fl[i] == kept_f:
                store = ("rm", j, True)
            else:
                store = ("fl", j, (r + 2) % 256)
                out.append((i, j))
            if rng.random() < 0.5:
                late.append(store)
            else:
                (rm if store[0] == "rm" else fl)[store[1]] = store[2]
        for plane, j, v in late:
            (rm if plane == "rm" else fl)[j] = v
        live = out
        r += 1
    return [j for j in range(n) if not rm[j]]


def _check(boxes, scores, thr, rng, bulk01):
    order = oracle.score_order(scores)
    kept = _resolve_model(len(boxes), _pairs(boxes[order], thr), rng, bulk01)
    got = [int(order[j]) for j in kept]
    assert got == oracle.nms_single(boxes, scores, thr).tolist()


@pytest.mark.parametrize("bulk01", [False, True])
def test_random_inputs(bulk01):
    rng = np.random.default_rng(7)
    for case in range(300):
        n = int(rng.integers(1, 48))
        span = float(rng.choice([10.0, 40.0, 150.0]))
        xy = rng.uniform(0, span, (n, 2))
        wh = rng.uniform(5, 40, (n, 2))
        boxes = np.concatenate([xy, xy + wh], 1).astype(np.float32)
        scores = rng.choice(np.linspace(0, 1, 9), n).astype(np.float32)  # ties too
        thr = float(rng.choice([0.1, 0.3, 0.5, 0.7]))
        _check(boxes, scores, thr, rng, bulk01)


@pytest.mark.parametrize("bulk01", [False, True])
def test_chain_past_the_byte_wrap(bulk01):
    """600 unit boxes sliding by 0.3: one pair per link, about 300 passes."""
    rng = np.random.default_rng(3)
    x = (np.arange(600) * 0.3).astype(np.float32)
    boxes = np.stack([x, np.zeros_like(x), x + 1.0, np.ones_like(x)], 1).astype(np.float32)
    scores = np.linspace(1.0, 0.0, 600, endpoint=False).astype(np.float32)
    perm = rng.permutation(600)
    _check(boxes[perm], scores[perm], 0.5, rng, bulk01)
