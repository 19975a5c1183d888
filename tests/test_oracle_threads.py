"""The oracle on several host threads at once gives the results it gives on
one: the CPU baseline runs one tree per thread."""
import concurrent.futures

import numpy as np

import oracle


def _case(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((12, 2000)) * 2.0).astype(np.float32)
    _, _, ids, lps = oracle.candidates(x, 32)
    U = (rng.standard_normal((2000, 8)) * 0.3).astype(np.float32)
    Vt = (rng.standard_normal((2000, 8)) * 0.3).astype(np.float32)
    return lps, ids, oracle.markov_table(ids, U, Vt, 3)


def _heap(args):
    lps, ids, E = args
    t = oracle.heap_select(lps, ids, 400, E=E).trimmed()
    return t.tok.tobytes() + t.parent.tobytes() + t.score.tobytes()


def test_heap_is_thread_safe():
    cases = [_case(s) for s in range(16)]
    serial = [_heap(c) for c in cases]
    with concurrent.futures.ThreadPoolExecutor(max_workers=8) as ex:
        for _ in range(3):
            assert list(ex.map(_heap, cases)) == serial
