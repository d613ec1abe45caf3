"""Fused mask + sample on the GPU against the CPU oracle.

The bar (greedy and masking exact; sampling by the stated tolerance):
  * greedy ids (temperature <= 0, top_k == 1) identical to the oracle, lowest
    index on ties; unsatisfiable rows -1;
  * the device Philox4x32-10 identical to the oracle's, word for word;
  * every sampled id accepted: in the oracle keep-set K, or with probability
    within 1e-6 (relative) of the threshold, or in K' (the keep-set with top_p
    raised and min_p lowered by 1e-6 relative);
  * ids identical to the oracle's on >= 99.9% of rows (same noise stream),
    pooled per path over >= 5000 draws (offsets and filter settings), every
    rate printed;
  * draw histograms within total variation 0.002 of the oracle's on the same
    streams, and a goodness-of-fit to the exact filtered softmax;
  * deterministic in (seed, offset), different when either changes;
  * heterogeneous per-row parameters equal to broadcasting each row's own.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from grammar_constrained_logit_gb300 import ops  # noqa: E402
from grammar_constrained_logit_gb300 import synthetic as syn  # noqa: E402
from parity_check import REL, Pool, check_ids, check_workload  # noqa: E402

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DT = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grammar_constrained_logit_gb300 import _lib

    _lib.load()


def to_dev(storage: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(storage.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(storage).cuda()


def params_of(w: syn.Workload, rows=None):
    out = {}
    for name in ("temperature", "top_k", "top_p", "min_p"):
        a = w.per_row(name)
        out[name] = a if rows is None else a[rows]
    return out


def run_gpu(w: syn.Workload, offset: int, use_mask=True):
    lg = to_dev(w.logits, w.dtype)[:, :w.cols]
    p = {k: torch.from_numpy(v).cuda() for k, v in params_of(w).items()}
    bm = torch.from_numpy(w.bitmask).cuda() if (use_mask and w.bitmask is not None) else None
    idx = None if w.indices is None else torch.from_numpy(w.indices).cuda()
    ids = ops.mask_and_sample(lg, bm, p["temperature"], p["top_k"], p["top_p"], p["min_p"],
                              seed=w.seed, offset=offset, indices=idx,
                              vocab_size=w.vocab_size if bm is not None else None)
    return ids.cpu().numpy()


def check_rows(w, offset, gpu_ids, rows=None, use_mask=True):
    """Acceptance of every row (raises otherwise); the agreement counts for a Pool."""
    return check_workload(w, offset, gpu_ids, rows=rows, use_mask=use_mask)


# ------------------------------------------------------------------- Philox

def test_philox_words_identical():
    rng = np.random.default_rng(3)
    n = 20000
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    key[0] = 0
    got = ops.philox4x32_10(torch.from_numpy(ctr.view(np.int32)).cuda(),
                            torch.from_numpy(key.view(np.int32)).cuda()).cpu().numpy().view(np.uint32)
    for i in range(0, n, 7):
        assert got[i].tolist() == oracle.philox4x32_10(ctr[i], key[i]).tolist(), i


# ------------------------------------------------------------------- golden

def test_golden_keep_sets_and_greedy():
    g = json.load(open(os.path.join(GOLDEN, "keep_set_small.json")))
    for case in g["cases"]:
        l = (np.log(np.array(case["probs"], dtype=np.float64)).astype(np.float32)
             if "probs" in case else np.array([float(x) for x in case["logits"]], np.float32))
        x = torch.from_numpy(np.tile(l, (64, 1))).cuda()
        bm = None
        if case.get("mask_bits") is not None:
            bm = torch.from_numpy(np.tile(syn.pack_bits(np.array([case["mask_bits"]], bool)),
                                          (64, 1))).cuda()
        for off in range(4):
            ids = ops.mask_and_sample(x, bm, case["T"], case["top_k"], case["top_p"],
                                      case["min_p"], seed=11, offset=off).cpu().numpy()
            assert set(ids.tolist()) <= set(case["kept"]), case["name"]
    for case in g["greedy_cases"]:
        l = np.array([float(x) for x in case["logits"]], np.float32)
        x = torch.from_numpy(l[None, :]).cuda()
        bm = None
        if case.get("mask_bits") is not None:
            bm = torch.from_numpy(syn.pack_bits(np.array([case["mask_bits"]], bool))).cuda()
        ids = ops.mask_and_sample(x, bm, case["T"], case["top_k"]).cpu().numpy()
        assert ids[0] == case["id"], case["name"]


# ------------------------------------------------------------------- greedy

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [1, 31, 1003, 32000, 131072, 202048])
def test_greedy_exact(dtype, V):
    rng = np.random.default_rng(V + DT[dtype])
    B = 16
    x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    x[: B // 2] = np.round(x[: B // 2])          # exact ties everywhere
    x[1, :] = 5.0                                # a row of all-equal values
    x[2, :] = -np.inf                            # no finite candidate
    allowed = rng.random((B, V)) < 0.3
    allowed[3] = False                           # unsatisfiable
    st = syn.to_storage(x, dtype)
    bm = syn.pack_bits(allowed)
    lg = to_dev(st, dtype)
    bmd = torch.from_numpy(bm).cuda()
    for temp, k in ((0.0, 0), (-1.0, 7), (0.8, 1)):
        got = ops.mask_and_sample(lg, bmd, temp, k).cpu().numpy()
        want = oracle.mask_and_sample(st, dtype=DT[dtype], bitmask=bm, temperature=temp, top_k=k)
        assert np.array_equal(got, want), (temp, k, np.flatnonzero(got != want)[:5])
        got = ops.sample(lg, temp, k).cpu().numpy()
        want = oracle.mask_and_sample(st, dtype=DT[dtype], temperature=temp, top_k=k)
        assert np.array_equal(got, want), (temp, k)


def test_top_k_one_equals_greedy_equals_argmax():
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((64, 50000)).astype(np.float32)).cuda()
    a = ops.sample(x, 0.0).cpu().numpy()
    b = ops.sample(x, 0.9, top_k=1, top_p=0.5, seed=3).cpu().numpy()
    c = torch.argmax(x, dim=1).cpu().numpy()
    assert np.array_equal(a, b) and np.array_equal(a, c)


# ------------------------------------------------------- sampled parity

def _small_workloads():
    yield syn.tiny_greedy()
    yield syn.apply_only(B=24, V=5000, padded_cols=5120, n_indexed=10, density=0.05)
    yield syn.fused_sample(B=48, V=20000, steps=3)
    for tp in (0.5, 0.9, 0.99):
        yield syn.zipf_top_p(B=64, V=32000, top_p=tp)
    yield syn.speculative_verify(slots=12, rows_per_slot=8, V=20000, constrained_slots=6)


def test_small_workloads_parity():
    pool = Pool("reduced-size workloads (the five configurations' shapes), 14 offsets")
    for w in _small_workloads():
        if w.name == "apply_only":   # no sampling parameters: sample it plainly
            w.temperature, w.top_k, w.top_p, w.min_p = 0.9, 40, 0.95, 0.01
        for off in range(14):
            pool.add(check_rows(w, off, run_gpu(w, off)))
    pool.done()


def test_min_p_below_a_narrower_window():
    """min-p admits tokens below the narrower top-k window that the tiles
    compact: the keep-set must still include them (here 2000 tied tokens just
    below the window carry ~38% of the kept mass)."""
    V, B = 12000, 64
    row = np.full(V, -5.0, np.float32)
    row[0] = 10.0                 # the maximum
    row[1:1000] = 5.0             # inside the 6-logit top-k window
    row[1000:3000] = 3.95         # below the window, above the min-p bound 3.8
    x = np.tile(row, (B, 1))
    args = dict(temperature=1.0, top_k=2500, min_p=float(np.exp(-6.2)))
    w = syn.Workload("minp_gap", "f32", x, V, V, seed=4)
    w.temperature, w.top_k, w.min_p = 1.0, 2500, args["min_p"]
    pool = Pool("min-p below the top-k window")
    xd = torch.from_numpy(x).cuda()
    for off in range(80):
        g = ops.sample(xd, seed=4, offset=off, **args).cpu().numpy()
        pool.add(check_rows(w, off, g))
    pool.done()


def test_workspace_reuse_across_shapes():
    """One workspace serves calls of any shape in any order: every call leaves
    the state the next one needs (the counters at its front zero)."""
    rng = np.random.default_rng(8)
    ws = torch.zeros(ops.sample_workspace_bytes(torch.float32, 300, 70000), dtype=torch.uint8,
                     device="cuda")
    shapes = [(300, 1000), (2, 70000), (300, 70000), (17, 5000), (1, 64), (300, 33),
              (150, 40000), (3, 1003)]
    pool = Pool("one workspace reused across shapes")
    for rnd in range(5):
        for i, (B, V) in enumerate(shapes):
            x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
            args = dict(temperature=0.8, top_k=30, top_p=0.9, min_p=0.02)
            own = (i + rnd) % 2 == 0
            g = ops.sample(torch.from_numpy(x).cuda(), seed=rnd, offset=B, **args,
                           workspace=ws if own else None).cpu().numpy()
            w = syn.Workload("ws", "f32", x, V, V, seed=rnd)
            w.temperature, w.top_k, w.top_p, w.min_p = 0.8, 30, 0.9, 0.02
            pool.add(check_rows(w, B, g))
    torch.cuda.synchronize()
    assert int(ws[:256 + 4 * 16384].count_nonzero()) == 0
    pool.done()


def test_stale_workspace_front_is_still_correct():
    """A workspace whose front counters are not zero (as a call that failed
    part-way could leave them, or one never zero-filled) still gives correct ids:
    a stale row key above the row's maximum sends the row to the re-read path,
    and a stale pool counter only flags tiles as overflowed.  The call resets
    the counters of its rows, and the next call runs at full speed again."""
    rng = np.random.default_rng(31)
    B, V = 64, 30000
    x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    w = syn.Workload("stale", "f32", x, V, V, seed=3)
    # top-k/top-p rows, and min-p-only rows (whose cut rests on the compacted
    # buffers alone)
    w.temperature = np.float32(0.9)
    w.top_k = np.where(np.arange(B) % 2 == 0, 40, 0).astype(np.int32)
    w.top_p = np.where(np.arange(B) % 2 == 0, 0.9, 1.0).astype(np.float32)
    w.min_p = np.where(np.arange(B) % 2 == 0, 0.0, 0.05).astype(np.float32)
    front = 256 + 4 * 16384
    ws = torch.zeros(ops.sample_workspace_bytes(torch.float32, B, V), dtype=torch.uint8,
                     device="cuda")
    xd = torch.from_numpy(x).cuda()
    p = {k: torch.from_numpy(w.per_row(k)).cuda() for k in ("temperature", "top_k", "top_p",
                                                            "min_p")}
    pool = Pool("stale workspace front (0xff bytes, then a 0x7f pattern)")
    for off, junk in enumerate([0xFF, 0x7F] * 40):
        ws[:front].fill_(junk)
        g = ops.sample(xd, p["temperature"], p["top_k"], p["top_p"], p["min_p"], seed=3,
                       offset=off, workspace=ws).cpu().numpy()
        pool.add(check_rows(w, off, g))
        # the pool counter and the rows' keys are back to zero
        assert int(ws[:4].count_nonzero()) == 0
        assert int(ws[256:256 + 4 * B].count_nonzero()) == 0
    pool.done()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_filter_grid_parity(dtype):
    """Every combination of filters, on rows narrow and flat, masked and not,
    including flat rows whose keep-set overflows the compaction buffers."""
    rng = np.random.default_rng(77 + DT[dtype])
    B, V = 96, 60000
    x = rng.standard_normal((B, V)).astype(np.float32) * np.float32(2.0)
    x[::3] *= np.float32(0.05)                   # flat rows
    st = syn.to_storage(x, dtype)
    allowed = rng.random((B, V)) < 0.5
    allowed[::4] = True
    w = syn.Workload("grid", dtype, st, V, V, bitmask=syn.pack_bits(allowed), seed=5)
    grid = [(k, tp, mp) for k in (0, 2, 50, 1000, 5000) for tp in (1.0, 0.3, 0.9, 0.999)
            for mp in (0.0, 0.05)]
    w.temperature = rng.uniform(0.4, 1.6, B).astype(np.float32)
    sel = [grid[i % len(grid)] for i in range(B)]
    w.top_k = np.array([s[0] for s in sel], np.int32)
    w.top_p = np.array([s[1] for s in sel], np.float32)
    w.min_p = np.array([s[2] for s in sel], np.float32)
    pool = Pool(f"filter grid {dtype} (top-k x top-p x min-p, flat and narrow rows)")
    for off in range(53):
        pool.add(check_rows(w, off, run_gpu(w, off)))
    pool.done()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_small_top_k_rows_parity(dtype):
    """Top-k rows with k <= 32 and around it: Gaussian rows, rows of a few
    repeated values (ties at the k-th logit), rows with fewer candidates than k,
    and rows whose candidates sit in one short run of the vocabulary."""
    rng = np.random.default_rng(91 + DT[dtype])
    B, V = 96, 40000
    x = rng.standard_normal((B, V)).astype(np.float32) * np.float32(2.0)
    x[1::4] = np.round(x[1::4])                      # ties
    st = syn.to_storage(x, dtype)
    allowed = rng.random((B, V)) < 0.6
    allowed[2::4] = False                            # a handful of candidates
    for r in range(2, B, 4):
        allowed[r, rng.choice(V, size=int(rng.integers(1, 40)), replace=False)] = True
    allowed[3::4] = False                            # one short run
    for r in range(3, B, 4):
        s0 = int(rng.integers(0, V - 3000))
        allowed[r, s0:s0 + 3000] = True
    w = syn.Workload("topk", dtype, st, V, V, bitmask=syn.pack_bits(allowed), seed=6)
    ks = np.array([1, 2, 7, 20, 31, 32, 33, 50], np.int32)
    w.temperature = rng.uniform(0.4, 1.6, B).astype(np.float32)
    w.top_k = ks[np.arange(B) % len(ks)]
    w.top_p = np.where(np.arange(B) % 3 == 0, 0.9, 1.0).astype(np.float32)
    w.min_p = np.where(np.arange(B) % 5 == 0, 0.05, 0.0).astype(np.float32)
    pool = Pool(f"top-k rows with k near 32, {dtype} (ties, few candidates, one run)")
    for off in range(53):
        pool.add(check_rows(w, off, run_gpu(w, off)))
    pool.done()


def test_masked_token_never_drawn_and_indices():
    rng = np.random.default_rng(8)
    B, V = 64, 4099
    x = torch.from_numpy(rng.standard_normal((B, V)).astype(np.float32) * 3).cuda()
    allowed = rng.random((B, V)) < 0.02
    bm = torch.from_numpy(syn.pack_bits(allowed)).cuda()
    idx = np.array([3, 5, 7, 63, -4, 200, 5], dtype=np.int32)  # invalid and duplicate entries
    masked_rows = {3, 5, 7, 63}
    hit_unmasked = 0
    for off in range(20):
        ids = ops.mask_and_sample(x, bm, 1.0, seed=1, offset=off,
                                  indices=torch.from_numpy(idx)).cpu().numpy()
        full = ops.mask_and_sample(x, bm, 1.0, 0, 0.95, 0.0, seed=2, offset=off).cpu().numpy()
        for r in range(B):
            if r in masked_rows:
                assert allowed[r, ids[r]]
            else:
                hit_unmasked += int(not allowed[r, ids[r]])
            assert allowed[r, full[r]]
    assert hit_unmasked > 0  # rows outside indices really are unmasked


def test_unsatisfiable_rows_return_minus_one():
    x = torch.randn(6, 3000, device="cuda")
    bm = torch.full((6, 94), -1, dtype=torch.int32, device="cuda")
    bm[1] = 0
    bm[4] = 0
    for args in ((0.0, 0), (1.0, 0), (0.7, 5, 0.9, 0.1), (1.3, 0, 1.0, 0.0)):
        ids = ops.mask_and_sample(x, bm, *args).cpu().numpy()
        assert ids[1] == -1 and ids[4] == -1 and (ids[[0, 2, 3, 5]] >= 0).all()


def test_edge_shapes():
    for B, V in ((1, 1), (3, 2), (2, 33), (5, 7)):
        x = np.random.default_rng(V).standard_normal((B, V)).astype(np.float32)
        for args in (dict(temperature=0.0), dict(temperature=1.0),
                     dict(temperature=1.0, top_k=2, top_p=0.5, min_p=0.1)):
            g = ops.sample(torch.from_numpy(x).cuda(), **args, seed=1).cpu().numpy()
            w = oracle.mask_and_sample(x, dtype=oracle.F32, seed=1, **args)
            assert np.array_equal(g, w), (B, V, args)
    # zero-width vocabulary: every row has no candidate
    ids = ops.sample(torch.randn(4, 8, device="cuda"), 1.0, vocab_size=0).cpu().numpy()
    assert (ids == -1).all()
    # empty batch: nothing launched
    assert ops.sample(torch.randn(0, 8, device="cuda"), 1.0).numel() == 0


def test_misaligned_rows_and_strides():
    rng = np.random.default_rng(12)
    for dtype in ("f32", "f16", "bf16"):
        B, V, stride = 9, 3001, 3011
        x = (rng.standard_normal((B, stride)) * 2).astype(np.float32)
        st = syn.to_storage(x, dtype)
        base = to_dev(np.concatenate([st.reshape(-1), st.reshape(-1)[:1]]), dtype)
        lg = base[1:1 + B * stride].view(B, stride)[:, :V]     # base pointer off by one element
        allowed = rng.random((B, V)) < 0.4
        bm = syn.pack_bits(allowed)
        for args in (dict(temperature=0.0), dict(temperature=0.9, top_k=30, top_p=0.9)):
            got = ops.mask_and_sample(lg, torch.from_numpy(bm).cuda(), seed=4, **args).cpu().numpy()
            shifted = np.concatenate([st.reshape(-1), st.reshape(-1)[:1]])[1:1 + B * stride]
            want = oracle.mask_and_sample(shifted.reshape(B, stride), dtype=DT[dtype], bitmask=bm,
                                          cols=V, seed=4, **args)
            assert np.array_equal(got, want), (dtype, args)


def test_long_rows():
    """Rows of 1.5 M bf16 tokens (split over a cluster of CTAs) and a single row of
    4 M float32 tokens, all three paths, against the oracle."""
    rng = np.random.default_rng(13)
    for B, V, dtype in ((3, 1_500_000, "bf16"), (1, 4_000_000, "f32")):
        x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
        st = syn.to_storage(x, dtype)
        lg = to_dev(st, dtype)
        for args in (dict(temperature=0.0), dict(temperature=1.0, top_k=100),
                     dict(temperature=1.0, top_p=0.5), dict(temperature=0.2)):
            got = ops.sample(lg, seed=9, **args).cpu().numpy()
            want = oracle.mask_and_sample(st, dtype=DT[dtype], seed=9, **args)
            assert np.array_equal(got, want), (B, V, args)


def test_small_rows_after_large_rows():
    """Rows with fewer vectors than threads, sampled right after a launch that
    leaves large logits in the staging shared memory: lanes without a vector
    must contribute nothing (a cut of -inf once admitted them)."""
    rng = np.random.default_rng(14)
    big = to_dev(syn.to_storage((rng.standard_normal((3, 1_500_000)) * 8).astype(np.float32),
                                "bf16"), "bf16")
    V = 64
    x = np.tile((rng.standard_normal(V) * 1.5).astype(np.float32), (20_000, 1))
    xt = torch.from_numpy(x).cuda()
    for args in (dict(temperature=0.7, top_k=10), dict(temperature=1.2, top_p=0.8),
                 dict(temperature=1.0, min_p=0.1), dict(temperature=1.0)):
        ops.sample(big, seed=1, temperature=1.0, top_k=100)
        g = ops.sample(xt, seed=99, offset=5, **args).cpu().numpy()
        want = oracle.mask_and_sample(x, dtype=oracle.F32, seed=99, offset=5, **args)
        assert ((g >= 0) & (g < V)).all(), args
        assert (g == want).mean() >= 0.999, args


# ---------------------------------------------------- distribution, determinism

def test_distribution_same_streams_and_exact():
    from scipy import stats

    V = 64
    rng = np.random.default_rng(21)
    l = (rng.standard_normal(V) * 1.5).astype(np.float32)
    N = 100_000
    x = np.tile(l, (N, 1))
    for args in (dict(temperature=1.0), dict(temperature=0.7, top_k=10),
                 dict(temperature=1.2, top_p=0.8), dict(temperature=1.0, min_p=0.1)):
        g = ops.sample(torch.from_numpy(x).cuda(), seed=99, offset=5, **args).cpu().numpy()
        o, keep, p, _ = oracle.mask_and_sample(x[:1], dtype=oracle.F32, seed=99, offset=5,
                                               want_keep=True, want_p=True, **args)
        o = oracle.mask_and_sample(x, dtype=oracle.F32, seed=99, offset=5, **args)
        hg = np.bincount(g, minlength=V) / N
        ho = np.bincount(o, minlength=V) / N
        assert 0.5 * np.abs(hg - ho).sum() <= 0.002, args
        q = np.where(keep[0], p[0], 0.0)
        q /= q.sum()
        assert hg[~keep[0]].sum() == 0
        sel = keep[0]
        cnt = hg[sel] * N
        chi2 = ((cnt - N * q[sel]) ** 2 / (N * q[sel])).sum()
        pval = stats.chi2.sf(chi2, df=max(int(sel.sum()) - 1, 1)) if sel.sum() > 1 else 1.0
        assert pval > 1e-4, (args, chi2, pval)


def test_determinism_and_offset():
    w = syn.fused_sample(B=64, V=40000, steps=1)
    a = run_gpu(w, 0)
    b = run_gpu(w, 0)
    c = run_gpu(w, 1)
    w2 = syn.fused_sample(B=64, V=40000, steps=1)
    w2.seed = 8
    d = run_gpu(w2, 0)
    assert np.array_equal(a, b)
    assert (a != c).mean() > 0.3 and (a != d).mean() > 0.3


def test_heterogeneous_rows_equal_broadcast():
    w = syn.speculative_verify(slots=8, rows_per_slot=8, V=30000, constrained_slots=4)
    het = run_gpu(w, 3)
    pr = params_of(w)
    lg = to_dev(w.logits, w.dtype)
    bm = torch.from_numpy(w.bitmask).cuda()
    idx = torch.from_numpy(w.indices).cuda()
    for r in range(0, w.B, 5):
        one = ops.mask_and_sample(lg, bm, float(pr["temperature"][r]), int(pr["top_k"][r]),
                                  float(pr["top_p"][r]), float(pr["min_p"][r]), seed=w.seed,
                                  offset=3, indices=idx).cpu().numpy()
        assert one[r] == het[r], r


# ------------------------------------------------------ full-size workloads

def test_slots_per_slot_params_and_row_seeds():
    """The [slots, rows_per_slot, V] entry point: one parameter per slot shared by
    its rows, and a Philox seed per row, against the oracle run with the slot
    values repeated over the rows and the same seeds."""
    R = 8
    w = syn.speculative_verify(slots=12, rows_per_slot=R, V=20000, constrained_slots=6)
    names = ("temperature", "top_k", "top_p", "min_p")
    slot = {k: np.ascontiguousarray(w.per_row(k)[::R]) for k in names}
    rowp = {k: np.repeat(v, R) for k, v in slot.items()}
    seeds = np.random.default_rng(5).integers(0, 2**63, size=w.B, dtype=np.int64)
    lg = to_dev(w.logits, w.dtype)[:, :w.cols]
    bm = torch.from_numpy(w.bitmask).cuda()
    idx = torch.from_numpy(w.indices).cuda()
    p = {k: torch.from_numpy(v).cuda() for k, v in slot.items()}
    sd = torch.from_numpy(seeds).cuda()
    pool = Pool("slot layout with per-slot parameters and per-row seeds")
    for off in range(53):
        g = ops.mask_and_sample_slots(lg, bm, R, p["temperature"], p["top_k"], p["top_p"],
                                      p["min_p"], offset=off, seeds=sd, indices=idx,
                                      vocab_size=w.vocab_size).cpu().numpy()
        pool.add(check_ids(w.logits, w.dtype, g, params=rowp, seed=0, offset=off,
                           bitmask=w.bitmask, vocab_size=w.vocab_size, indices=w.indices,
                           cols=w.cols, seeds=seeds.view(np.uint64)))
    pool.done()
    # one row per slot and no seeds: the plain entry point's ids
    w1 = syn.speculative_verify(slots=6, rows_per_slot=4, V=5000, constrained_slots=3)
    pp = {k: torch.from_numpy(w1.per_row(k)).cuda() for k in names}
    l1 = to_dev(w1.logits, w1.dtype)[:, :w1.cols]
    b1, i1 = torch.from_numpy(w1.bitmask).cuda(), torch.from_numpy(w1.indices).cuda()
    a = ops.mask_and_sample(l1, b1, pp["temperature"], pp["top_k"], pp["top_p"], pp["min_p"],
                            seed=11, offset=2, indices=i1, vocab_size=w1.vocab_size)
    b = ops.mask_and_sample_slots(l1, b1, 1, pp["temperature"], pp["top_k"], pp["top_p"],
                                  pp["min_p"], seed=11, offset=2, indices=i1,
                                  vocab_size=w1.vocab_size)
    assert torch.equal(a, b)


def test_fused_sample_full_size():
    """B=256, V=131072 bf16, 10% mask, per-row T, top_k 50, top_p 0.9, min_p 0.05;
    every row of 20 steps (offsets 0, 5, .., 95) against the oracle."""
    w = syn.fused_sample()
    pool = Pool("fused_sample full size (B=256, V=131072 bf16)")
    for off in range(0, 100, 5):
        pool.add(check_rows(w, off, run_gpu(w, off)))
    pool.done()


@pytest.mark.parametrize("tp", [0.5, 0.9, 0.99, "greedy"])
def test_zipf_top_p_full_size(tp):
    """B=1024, V=32000 fp32 Zipf-ranked logits, T=0.7, top_p sweep and greedy;
    every row of five steps against the oracle."""
    w = syn.zipf_top_p(top_p=0.9 if tp == "greedy" else tp)
    if tp == "greedy":
        w.temperature = 0.0
    pool = Pool(f"zipf_top_p full size, top_p {tp}")
    for off in range(5):
        pool.add(check_rows(w, off, run_gpu(w, off)))
    pool.done()


def test_speculative_verify_full_size():
    """1024 rows x 202048 fp16, 512 masked rows, heterogeneous parameters; every
    row of five steps against the oracle."""
    w = syn.speculative_verify()
    pool = Pool("speculative_verify full size (1024 x 202048 fp16)")
    for off in range(5):
        g = run_gpu(w, off)
        assert (g >= -1).all() and (g < w.vocab_size).all()
        pool.add(check_rows(w, off, g))
    pool.done()
