"""Sampled-id parity of the GPU sampler against the CPU oracle, pooled per path.

The bar (Kernel Hub "logits-processor", Correctness: agreement with an
independent reference sampler; the tolerance rule of the design notes):

  * every GPU id is accepted: it lies in the oracle keep-set K, or its
    probability is within 1e-6 (relative) of the threshold, or it lies in K',
    the keep-set recomputed with top_p raised and min_p lowered by 1e-6
    (relative); greedy and unsatisfiable rows must match exactly;
  * over each path, GPU ids equal the oracle's (same Philox stream) on at least
    99.9% of at least 5000 draws.

The oracle runs in threads over chunks of rows (its C calls release the
interpreter lock), so full-size batches are checked row by row in seconds.
Agreement rates are printed (``[parity]`` lines; ``pytest -rP`` shows them).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle

REL = 1e-6
FLOOR = 0.999
MIN_DRAWS = 5000
DT = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16}
WORKERS = max(1, min(16, os.cpu_count() or 1))
NAMES = ("temperature", "top_k", "top_p", "min_p")


def relaxed(tp: np.ndarray, mp: np.ndarray):
    """top_p raised and min_p lowered by 1e-6 relative (the K' of the rule)."""
    tp = np.asarray(tp, np.float32)
    mp = np.asarray(mp, np.float32)
    tp2 = np.where(tp < 1, np.minimum(tp * (1 + REL), np.float32(0.99999994)), tp)
    return tp2.astype(np.float32), (mp * (1 - REL)).astype(np.float32)


def _oracle_rows(logits, dtype, rows, prm, seed, offset, bitmask, vocab_size, indices, cols,
                 seeds, want_all):
    kw = dict(dtype=dtype, bitmask=bitmask, vocab_size=vocab_size, indices=indices, cols=cols,
              temperature=prm["temperature"], top_k=prm["top_k"], top_p=prm["top_p"],
              min_p=prm["min_p"], seed=seed, offset=offset, row_ids=rows,
              seeds=None if seeds is None else seeds[rows])
    if want_all:
        kw.update(want_keep=True, want_p=True, want_thr=True)
    return oracle.mask_and_sample(np.ascontiguousarray(logits[rows]), **kw)


def check_ids(logits: np.ndarray, dtype: str, gpu_ids: np.ndarray, *, params: dict, seed: int,
              offset: int, rows=None, bitmask=None, vocab_size=None, indices=None, cols=None,
              seeds=None, chunk: int = 32):
    """Checks the GPU ids of ``rows`` (default: all) against the oracle.

    ``params`` holds per-row arrays (length = logits rows) of the four sampling
    parameters; ``seeds`` optional per-row Philox seeds.  Raises on any id the
    rule does not accept; returns (rows whose id equals the oracle's, rows
    checked, [(row, gpu id, oracle id)] of the others)."""
    B = logits.shape[0]
    rows = np.arange(B) if rows is None else np.asarray(rows)
    dt = DT[dtype]
    prm_all = {k: np.asarray(params[k]) for k in NAMES}

    def work(rs):
        prm = {k: v[rs] for k, v in prm_all.items()}
        ids, keep, p, thr = _oracle_rows(logits, dt, rs, prm, seed, offset, bitmask, vocab_size,
                                         indices, cols, seeds, True)
        g = gpu_ids[rs]
        out, need = [], []
        for i, r in enumerate(rs):
            v = int(g[i])
            if ids[i] < 0 or thr[i] < 0:          # unsatisfiable or greedy: exact
                ok = v == ids[i]
            else:
                ok = 0 <= v < keep.shape[1] and bool(keep[i, v] or p[i, v] >= thr[i] * (1 - REL))
                if not ok and 0 <= v < keep.shape[1]:
                    need.append(i)
                    ok = None                      # decided by K' below
            out.append([int(r), v, int(ids[i]), ok,
                        float(p[i, v]) if 0 <= v < p.shape[1] else None, float(thr[i])])
        if need:
            sub = rs[need]
            tp2, mp2 = relaxed(prm["top_p"][need], prm["min_p"][need])
            prm2 = {k: prm[k][need] for k in NAMES}
            prm2["top_p"], prm2["min_p"] = tp2, mp2
            _, keep2, _, _ = _oracle_rows(logits, dt, sub, prm2, seed, offset, bitmask,
                                          vocab_size, indices, cols, seeds, True)
            for j, i in enumerate(need):
                out[i][3] = bool(keep2[j, out[i][1]])
        return out

    parts = [rows[i:i + chunk] for i in range(0, rows.size, chunk)]
    with ThreadPoolExecutor(WORKERS) as ex:
        res = [x for part in ex.map(work, parts) for x in part]
    bad = [tuple(x) for x in res if not x[3]]
    assert not bad, bad[:10]
    mism = [(x[0], x[1], x[2]) for x in res if x[1] != x[2]]
    return len(res) - len(mism), len(res), mism


class Pool:
    """Id agreement of one path, pooled over calls."""

    def __init__(self, name: str):
        self.name, self.agree, self.n, self.mism = name, 0, 0, []

    def add(self, result):
        a, n, mism = result
        self.agree += a
        self.n += n
        self.mism += mism

    def done(self, floor: float = FLOOR, min_draws: int = MIN_DRAWS):
        rate = self.agree / max(self.n, 1)
        print(f"[parity] {self.name}: {self.agree}/{self.n} ids identical to the oracle "
              f"({rate:.5f}); {self.n - self.agree} mismatches {self.mism[:5]}")
        assert self.n >= min_draws, (self.name, self.n)
        assert rate >= floor, (self.name, rate, self.mism[:10])
        return rate


def workload_params(w, rows=None) -> dict:
    return {k: (w.per_row(k) if rows is None else w.per_row(k)[rows]) for k in NAMES}


def check_workload(w, offset: int, gpu_ids: np.ndarray, rows=None, use_mask: bool = True):
    """check_ids on a synthetic workload (its mask, indices and parameters)."""
    return check_ids(w.logits, w.dtype, gpu_ids, params=workload_params(w), seed=w.seed,
                     offset=offset, rows=rows,
                     bitmask=w.bitmask if use_mask else None, vocab_size=w.vocab_size,
                     indices=w.indices if use_mask else None, cols=w.cols)
