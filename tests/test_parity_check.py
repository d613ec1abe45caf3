"""The sampled-id checker used by the GPU parity tests, exercised on the CPU:
ids taken from the oracle itself agree on every row, and an id outside the
keep-set (or a wrong greedy id) is rejected."""
import numpy as np
import pytest

import oracle
from grammar_constrained_logit_gb300 import synthetic as syn
from parity_check import Pool, check_ids, check_workload, relaxed


def _ids(w, off):
    pr = {k: w.per_row(k) for k in ("temperature", "top_k", "top_p", "min_p")}
    return oracle.mask_and_sample(w.logits, dtype={"f32": 0, "f16": 1, "bf16": 2}[w.dtype],
                                  bitmask=w.bitmask, vocab_size=w.vocab_size, indices=w.indices,
                                  cols=w.cols, seed=w.seed, offset=off, **pr)


def test_oracle_ids_agree_everywhere():
    w = syn.speculative_verify(slots=6, rows_per_slot=4, V=3000, constrained_slots=3)
    pool = Pool("oracle against itself")
    for off in range(3):
        pool.add(check_workload(w, off, _ids(w, off)))
    assert pool.agree == pool.n == 3 * w.B
    pool.done(min_draws=1)


def test_rejects_ids_outside_the_keep_set_and_wrong_greedy():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((4, 500)) * 3).astype(np.float32)
    prm = {"temperature": np.array([0.9, 0.9, 0.0, 0.9], np.float32),
           "top_k": np.array([5, 5, 0, 5], np.int32),
           "top_p": np.ones(4, np.float32), "min_p": np.zeros(4, np.float32)}
    ids = oracle.mask_and_sample(x, dtype=oracle.F32, seed=1, **prm)
    a, n, mism = check_ids(x, "f32", ids, params=prm, seed=1, offset=0)
    assert (a, n, mism) == (4, 4, [])
    bad = ids.copy()
    bad[1] = int(np.argmin(x[1]))            # far below the top-5 threshold
    with pytest.raises(AssertionError):
        check_ids(x, "f32", bad, params=prm, seed=1, offset=0)
    bad = ids.copy()
    bad[2] = (ids[2] + 1) % 500              # greedy must be exact
    with pytest.raises(AssertionError):
        check_ids(x, "f32", bad, params=prm, seed=1, offset=0)


def test_relaxed_parameters():
    tp, mp = relaxed(np.array([0.9, 1.0], np.float32), np.array([0.05, 0.0], np.float32))
    assert tp[0] > np.float32(0.9) and tp[1] == 1.0
    assert mp[0] < np.float32(0.05) and mp[1] == 0.0
