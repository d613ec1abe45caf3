"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against something fixed by the pages or
by mathematics: hand-worked golden cases (tests/golden), numpy's bit unpacking
and argmax, numpy's and PyTorch's float conversions, a brute-force pointwise
definition of the keep-set on tiny vocabularies, PyTorch's own Philox engine
header, the exponential-race identity of the Gumbel-max draw, and a
goodness-of-fit test of the draws against the exact filtered softmax.
"""
import json
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from grammar_constrained_logit_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DT = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16}


def _fill_storage(fill: float, dtype: str):
    """Storage value of ``fill`` in ``dtype`` by numpy / PyTorch conversion."""
    import torch

    x = np.float32(fill)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return np.float16(x)
    return np.uint16(torch.tensor(float(x), dtype=torch.float32).to(torch.bfloat16)
                     .view(torch.int16).item() & 0xFFFF)


def _np_apply(logits, dtype, bitmask, vocab_size, indices, fill):
    """Independent restatement of the apply loop: every word unpacked by numpy."""
    B = logits.shape[0]
    words = bitmask.shape[1]
    by = np.ascontiguousarray(bitmask).view(np.uint8).reshape(bitmask.shape[0], words * 4)
    bits = np.unpackbits(by, axis=1, bitorder="little")
    out = logits.copy()
    rows = range(B) if indices is None else [
        int(i) for i in indices if 0 <= int(i) < min(B, bitmask.shape[0])]
    fv = _fill_storage(fill, dtype)
    for b in rows:
        sel = bits[b, :vocab_size] == 0
        out[b, :vocab_size][sel] = fv
    return out


# ------------------------------------------------------------------ goldens

def _golden_logits(case, cases):
    v = case["logits"]
    if isinstance(v, str):
        v = cases[0]["logits"]
    return np.array(v, dtype=np.float32)


def test_golden_apply():
    g = json.load(open(os.path.join(GOLDEN, "apply_small.json")))
    for case in g["cases"]:
        logits = _golden_logits(case, g["cases"])
        bm = np.array([[int(h, 16) for h in row] for row in case["bitmask_hex"]],
                      dtype=np.uint32).view(np.int32)
        fill = float("-inf") if case["fill"] == "-inf" else float(case["fill"])
        out = oracle.apply(logits, bm, dtype=oracle.F32, fill=fill,
                           vocab_size=case["vocab_size"], indices=case["indices"])
        for b, kept in enumerate(case["expected_kept"]):
            kept = set(kept)
            for j in range(logits.shape[1]):
                if j in kept:
                    assert out[b, j] == logits[b, j], (case["name"], b, j)
                else:
                    assert out[b, j] == np.float32(fill), (case["name"], b, j)


def _case_logits(case):
    if "probs" in case:
        return np.log(np.array(case["probs"], dtype=np.float64)).astype(np.float32)
    return np.array([float(x) for x in case["logits"]], dtype=np.float32)


def _case_mask(case, V):
    bits = case.get("mask_bits")
    if bits is None:
        return None
    return syn.pack_bits(np.array([bits], dtype=bool))


def test_golden_keep_sets():
    g = json.load(open(os.path.join(GOLDEN, "keep_set_small.json")))
    for case in g["cases"]:
        l = _case_logits(case)[None, :]
        ids, keep, _, _ = oracle.mask_and_sample(
            l, dtype=oracle.F32, bitmask=_case_mask(case, l.shape[1]),
            temperature=case["T"], top_k=case["top_k"], top_p=case["top_p"],
            min_p=case["min_p"], seed=5, want_keep=True)
        assert sorted(np.flatnonzero(keep[0]).tolist()) == case["kept"], case["name"]
        assert ids[0] in case["kept"], case["name"]


def test_golden_greedy():
    g = json.load(open(os.path.join(GOLDEN, "keep_set_small.json")))
    for case in g["greedy_cases"]:
        l = _case_logits(case)[None, :]
        ids = oracle.mask_and_sample(l, dtype=oracle.F32, bitmask=_case_mask(case, l.shape[1]),
                                     temperature=case["T"], top_k=case["top_k"])
        assert ids[0] == case["id"], case["name"]


# -------------------------------------------------------------------- apply

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_apply_matches_numpy_unpack(dtype):
    rng = np.random.default_rng(100 + DT[dtype])
    for trial in range(60):
        B = int(rng.integers(1, 7))
        cols = int(rng.choice([1, 7, 31, 32, 33, 64, 100, 257, 1003]))
        pad = int(rng.choice([0, 0, 3, 8]))
        vocab = [None, cols, max(0, cols - int(rng.integers(0, 9))), 0][int(rng.integers(0, 4))]
        need = ((cols if vocab is None else vocab) + 31) // 32
        words = max(need, 1) + int(rng.integers(0, 3))
        bm_rows = B + int(rng.integers(0, 3))
        bm = rng.integers(0, 2**32, size=(bm_rows, words), dtype=np.uint64).astype(np.uint32).view(np.int32)
        x = (rng.standard_normal((B, cols + pad)) * 4).astype(np.float32)
        logits = syn.to_storage(x, dtype)
        idx = None
        if trial % 3 == 1:
            idx = rng.choice(B, size=int(rng.integers(0, B + 1)), replace=False).astype(np.int32)
        elif trial % 3 == 2:
            idx = np.array([B - 1, -1, B + 5, 0], dtype=np.int32)
        fill = float("-inf") if trial % 2 == 0 else float(rng.standard_normal() * 1e3)
        vs = oracle.resolve_vocab(vocab, cols, words)
        got = oracle.apply(logits, bm, dtype=DT[dtype], fill=fill, vocab_size=vocab,
                           indices=idx, cols=cols)
        want = _np_apply(logits, dtype, bm, vs, idx, fill)
        # columns >= cols of the padded buffer are never touched by either
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (trial, dtype)


def test_apply_special_cases():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 70)).astype(np.float32)
    ones = np.full((3, 3), -1, dtype=np.int32)
    zeros = np.zeros((3, 3), dtype=np.int32)
    assert np.array_equal(oracle.apply(x, ones, dtype=oracle.F32), x)          # identity
    z = oracle.apply(x, zeros, dtype=oracle.F32, vocab_size=70)
    assert np.all(np.isneginf(z))                                             # fill everywhere
    z0 = oracle.apply(x, zeros, dtype=oracle.F32, vocab_size=0)
    assert np.array_equal(z0, x)                                              # empty vocab
    zp = oracle.apply(x, zeros, dtype=oracle.F32, vocab_size=40)
    assert np.all(np.isneginf(zp[:, :40])) and np.array_equal(zp[:, 40:], x[:, 40:])
    # bits past vocab_size are never read: garbage there changes nothing
    g = zeros.copy()
    g[:, 1] = np.int32(-256)  # bits 8..31 of word 1 = tokens 40..63
    assert np.array_equal(oracle.apply(x, g, dtype=oracle.F32, vocab_size=40), zp)


def test_inconsistent_geometry_is_rejected():
    x = np.zeros((2, 40), dtype=np.float32)
    bm = np.zeros((2, 1), dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.apply(x, bm, dtype=oracle.F32, vocab_size=40)   # 40 > 1 word * 32
    with pytest.raises(ValueError):
        oracle.apply(x, np.zeros((2, 2), np.int32), dtype=oracle.F32, vocab_size=41)


# ------------------------------------------------------ dtype conversions

def test_decode_all_half_patterns():
    import torch

    pats = np.arange(65536, dtype=np.uint32)
    f16 = pats.astype(np.uint16).view(np.float16).astype(np.float64)
    bf = torch.from_numpy(pats.astype(np.uint16).view(np.int16)).view(torch.bfloat16).float().double().numpy()
    got16 = np.array([oracle.decode(int(p), oracle.F16) for p in pats[::7]])
    gotbf = np.array([oracle.decode(int(p), oracle.BF16) for p in pats[::7]])
    np.testing.assert_array_equal(got16, f16[::7])
    np.testing.assert_array_equal(gotbf, bf[::7])


def test_encode_round_to_nearest_even():
    import torch

    rng = np.random.default_rng(9)
    xs = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 6, 3000),
        rng.standard_normal(500) * 1e-6,          # fp16 subnormal range
        np.array([65504.0, 65519.0, 65520.0, 1e5, -1e5, 3.4e38, -3.4e38, 0.0, -0.0,
                  float("inf"), float("-inf"), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                  1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 6.0e-8, 2.9e-8, 3.0e-8]),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want16 = xs.astype(np.float16).view(np.uint16)
    wantbf = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, w16, wbf in zip(xs, want16, wantbf):
        assert oracle.encode(float(x), oracle.F16) == int(w16), float(x)
        assert oracle.encode(float(x), oracle.BF16) == int(wbf), float(x)
        assert oracle.encode(float(x), oracle.F32) == int(np.float32(x).view(np.uint32))


# ------------------------------------------------------------------- greedy

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_greedy_matches_numpy_argmax(dtype):
    rng = np.random.default_rng(40 + DT[dtype])
    B, V = 64, 300
    x = rng.standard_normal((B, V)).astype(np.float32)
    x[: B // 2] = np.round(x[: B // 2] * 2) / 2          # many exact ties
    x[5, :] = -np.inf                                    # no finite candidate
    x[6, ::3] = -np.inf
    st = syn.to_storage(x, dtype)
    vals = syn.storage_to_f32(st, dtype)
    allowed = rng.random((B, V)) < 0.6
    allowed[7] = False                                   # unsatisfiable row
    bm = syn.pack_bits(allowed)
    for temp, k in ((0.0, 0), (-1.0, 5), (0.9, 1)):
        ids = oracle.mask_and_sample(st, dtype=DT[dtype], bitmask=bm, temperature=temp, top_k=k)
        for b in range(B):
            cand = allowed[b] & (vals[b] > -np.inf)
            want = -1 if not cand.any() else int(np.argmax(np.where(cand, vals[b], -np.inf)))
            assert ids[b] == want, (b, temp, k)


# ---------------------------------------------------------------- keep-set

def _pointwise_keep(vals, cand, T, k, tp, mp):
    """Keep-set from its pointwise definition, no sorting: v is kept iff fewer than
    k candidates have larger p, the mass of strictly larger p is below top_p, and
    p_v >= min_p * p_max; the maximum itself is always kept."""
    z = vals.astype(np.float64) / T
    zc = np.where(cand, z, -np.inf)
    e = np.where(cand, np.exp(zc - zc.max()), 0.0)
    p = e / e.sum()
    pmax = p.max()
    keep = np.zeros(len(vals), dtype=bool)
    for v in np.flatnonzero(cand):
        greater = cand & (p > p[v])
        ok = True
        if k > 0:
            ok &= greater.sum() < k
        if tp < 1.0:
            ok &= p[greater].sum() < tp
        if mp > 0.0:
            ok &= p[v] >= mp * pmax
        keep[v] = ok or p[v] >= pmax
    return keep


def test_keep_set_brute_force_tiny_vocab():
    rng = np.random.default_rng(77)
    grid = [(k, tp, mp, T) for k in (0, 2, 3, 7, 16) for tp in (0.0, 0.1, 0.35, 0.6, 0.9, 1.0)
            for mp in (0.0, 0.05, 0.3, 1.0) for T in (0.5, 1.0, 2.0)]
    rows = []
    for V in (1, 2, 5, 16):
        for r in range(6):
            x = (rng.standard_normal(V) * 2).astype(np.float32)
            if r % 3 == 0:
                x = np.round(x).astype(np.float32)        # forced ties
            allowed = rng.random(V) < 0.7
            if r == 1:
                allowed[:] = True
            rows.append((x, allowed))
    checked = 0
    for x, allowed in rows:
        V = len(x)
        bm = syn.pack_bits(allowed[None, :])
        for (k, tp, mp, T) in grid:
            if k == 1:
                continue
            ids, keep, _, _ = oracle.mask_and_sample(x[None, :], dtype=oracle.F32, bitmask=bm,
                                                     vocab_size=V, temperature=T, top_k=k,
                                                     top_p=tp, min_p=mp, seed=1, want_keep=True)
            if not allowed.any():
                assert ids[0] == -1 and not keep.any()
                continue
            want = _pointwise_keep(x, allowed, T, k, tp, mp)
            assert np.array_equal(keep[0], want), (x, allowed, k, tp, mp, T)
            assert want[ids[0]]
            checked += 1
    assert checked > 1000


# ------------------------------------------------------------------- Philox

_PROBE_SRC = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
#include <cinttypes>
int main() {
  unsigned long long seed, sub, off;
  while (std::scanf("%llu %llu %llu", &seed, &sub, &off) == 3) {
    at::philox_engine e(seed, sub, off);
    for (int i = 0; i < 4; ++i) std::printf("%u ", (unsigned)e(10));
    std::printf("\n");
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    """PyTorch's own Philox4x32-10 engine (header-only, compiled for the host)."""
    import torch

    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    d = tmp_path_factory.mktemp("philox")
    src, exe = d / "probe.cpp", d / "probe"
    src.write_text(_PROBE_SRC)
    try:
        subprocess.check_call(["g++", "-std=c++17", "-O1", f"-I{inc}", str(src), "-o", str(exe)])
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("PyTorch Philox header does not compile here")

    def run(triples):
        text = "\n".join(f"{s} {u} {o}" for s, u, o in triples) + "\n"
        res = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True)
        return [list(map(int, line.split())) for line in res.stdout.strip().splitlines()]

    return run


def test_philox_matches_pytorch_engine(torch_philox):
    """PyTorch's engine takes key = seed and counter = (offset lo, offset hi,
    subsequence lo, subsequence hi); its first four outputs are one Philox4x32-10
    block at that counter."""
    rng = np.random.default_rng(5)
    triples, ctrs, keys = [], [], []
    for i in range(3000):
        c = rng.integers(0, 2**32, size=4, dtype=np.uint64)
        k = rng.integers(0, 2**32, size=2, dtype=np.uint64)
        if i == 0:
            c[:], k[:] = 0, 0
        elif i == 1:
            c[:], k[:] = 0xFFFFFFFF, 0xFFFFFFFF
        seed = int(k[0]) | (int(k[1]) << 32)
        off = int(c[0]) | (int(c[1]) << 32)
        sub = int(c[2]) | (int(c[3]) << 32)
        triples.append((seed, sub, off))
        ctrs.append(c.astype(np.uint32))
        keys.append(k.astype(np.uint32))
    want = torch_philox(triples)
    for c, k, w in zip(ctrs, keys, want):
        assert oracle.philox4x32_10(c, k).tolist() == w


def test_random_word_counter_layout(torch_philox):
    """Token v of row `row` under (seed, offset) uses word v & 3 of the block at
    counter (v >> 2, row, lo32(offset), hi32(offset)), key (lo32(seed), hi32(seed))."""
    rng = np.random.default_rng(6)
    cases = []
    for _ in range(1500):
        seed = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        offset = int(rng.integers(0, 2**63))
        row = int(rng.integers(0, 2**20))
        v = int(rng.integers(0, 2**22))
        cases.append((seed, offset, row, v))
    # torch: counter = (off lo, off hi, sub lo, sub hi) -> off = (row << 32) | (v >> 2), sub = offset
    want = torch_philox([(s, o, (r << 32) | (v >> 2)) for s, o, r, v in cases])
    for (s, o, r, v), w in zip(cases, want):
        assert oracle.random_word(s, o, r, v) == w[v & 3]


def test_uniform_and_gumbel_range():
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(0x1FF) == 2.0 ** -24          # low 9 bits are dropped
    assert oracle.uniform(0x200) == 3 * 2.0 ** -24
    g_lo, g_hi = oracle.gumbel(0), oracle.gumbel(0xFFFFFFFF)
    assert abs(g_lo - (-math.log(-math.log(2.0 ** -24)))) < 1e-12
    assert abs(g_hi - (-math.log(-math.log(1 - 2.0 ** -24)))) < 1e-9
    assert -2.82 < g_lo < -2.81 and 16.63 < g_hi < 16.64
    xs = sorted(np.random.default_rng(1).integers(0, 2**32, 200).tolist())
    gs = [oracle.gumbel(x) for x in xs]
    assert all(a <= b for a, b in zip(gs, gs[1:]))      # monotone in the word


# ---------------------------------------------------------------------- draw

def test_draw_is_exponential_race():
    """argmax_v (z_v + g_v) = argmax_v p_v / E_v with E_v = -log u_v (the
    exponential race); computed here in the ratio domain from the raw words."""
    rng = np.random.default_rng(8)
    B, V = 200, 37
    x = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    allowed = rng.random((B, V)) < 0.8
    bm = syn.pack_bits(allowed)
    seed, offset = 0x1234_5678_9ABC_DEF0, 42
    T = 0.8
    ids = oracle.mask_and_sample(x, dtype=oracle.F32, bitmask=bm, temperature=T, seed=seed,
                                 offset=offset)
    for b in range(B):
        p = np.where(allowed[b], np.exp((x[b].astype(np.float64) - x[b][allowed[b]].max()) / T), 0)
        E = np.array([-math.log(oracle.uniform(oracle.random_word(seed, offset, b, v)))
                      for v in range(V)])
        ratio = np.where(allowed[b], p / E, -1.0)
        assert ids[b] == int(np.argmax(ratio))


@pytest.mark.parametrize("T,k,tp,mp", [(1.0, 0, 1.0, 0.0), (0.7, 3, 1.0, 0.0),
                                       (1.3, 0, 0.8, 0.0), (1.0, 0, 1.0, 0.2)])
def test_draw_distribution_goodness_of_fit(T, k, tp, mp):
    """20000 independent draws (one per row, same logits) against the exact
    renormalised filtered softmax: chi-square p-value and total variation."""
    from scipy import stats

    l = np.array([2.0, 1.5, 1.0, 0.0, -1.0, 0.5, -3.0, 1.2], dtype=np.float32)
    allowed = np.array([1, 1, 0, 1, 1, 1, 1, 1], dtype=bool)
    N = 20000
    x = np.tile(l, (N, 1))
    bm = np.tile(syn.pack_bits(allowed[None, :]), (N, 1))
    ids, keep, p, _ = oracle.mask_and_sample(x[:1], dtype=oracle.F32, bitmask=bm[:1],
                                             temperature=T, top_k=k, top_p=tp, min_p=mp,
                                             want_keep=True, want_p=True)
    want_keep = _pointwise_keep(l, allowed, T, k, tp, mp)
    assert np.array_equal(keep[0], want_keep)
    q = np.where(want_keep, p[0], 0.0)
    q /= q.sum()
    ids = oracle.mask_and_sample(x, dtype=oracle.F32, bitmask=bm, temperature=T, top_k=k,
                                 top_p=tp, min_p=mp, seed=2024, offset=3)
    counts = np.bincount(ids, minlength=len(l)).astype(np.float64)
    assert counts[~want_keep].sum() == 0
    sel = want_keep
    chi2 = (((counts[sel] - N * q[sel]) ** 2) / (N * q[sel])).sum()
    pval = stats.chi2.sf(chi2, df=int(sel.sum()) - 1) if sel.sum() > 1 else 1.0
    assert pval > 1e-4, (chi2, pval)
    assert 0.5 * np.abs(counts / N - q).sum() < 0.02


def test_draw_deterministic_and_offset_sensitive():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((300, 500)).astype(np.float32)
    a = oracle.mask_and_sample(x, dtype=oracle.F32, temperature=1.0, seed=9, offset=0)
    b = oracle.mask_and_sample(x, dtype=oracle.F32, temperature=1.0, seed=9, offset=0)
    c = oracle.mask_and_sample(x, dtype=oracle.F32, temperature=1.0, seed=9, offset=1)
    d = oracle.mask_and_sample(x, dtype=oracle.F32, temperature=1.0, seed=10, offset=0)
    assert np.array_equal(a, b)
    assert (a != c).mean() > 0.5 and (a != d).mean() > 0.5


def test_single_kept_token_ignores_noise():
    x = np.array([[0.0, 5.0, 1.0, 4.9]], dtype=np.float32)
    for off in range(50):
        ids = oracle.mask_and_sample(x, dtype=oracle.F32, temperature=1.0, top_k=0,
                                     top_p=1.0, min_p=0.99, seed=off, offset=off)
        assert ids[0] == 1


# ------------------------------------------------- per-row flags and report
# TensorRT-Edge-LLM "Guided Decoder", struct Impl (deviceRowNeedsMask,
# rowHasAnyToken) and fillMasks (unsatisfiableSlots).

def test_apply_rows_hand_worked():
    """Three rows of four tokens, vocab_size 3: row 0 flagged with bits 0 and 2
    set, row 1 flagged with no bit set (unsatisfiable), row 2 not flagged with
    no bit set (left alone, keeps everything); token 3 is past vocab_size in
    every row and never changes."""
    x = np.arange(12, dtype=np.float32).reshape(3, 4)
    bm = np.array([[0b0101], [0], [0]], dtype=np.int32)
    out, has = oracle.apply_rows(x, bm, dtype=oracle.F32, flags=[1, 1, 0], vocab_size=3)
    ninf = -np.inf
    want = np.array([[0, ninf, 2, 3], [ninf, ninf, ninf, 7], [8, 9, 10, 11]], dtype=np.float32)
    assert np.array_equal(out, want)
    assert has.tolist() == [1, 0, 1]


def test_apply_rows_report_edges():
    """A kept bit only at vocab_size (outside the vocabulary) does not count;
    one at vocab_size - 1 does; vocab_size 0 keeps nothing anywhere; with no
    flags every row is masked."""
    x = np.zeros((2, 64), dtype=np.float32)
    bm = np.zeros((2, 2), dtype=np.int32)
    bm[0, 1] = 1 << 8          # token 40
    bm[1, 1] = 1 << 7          # token 39
    _, has = oracle.apply_rows(x, bm, dtype=oracle.F32, vocab_size=40)
    assert has.tolist() == [0, 1]
    _, has = oracle.apply_rows(x, bm, dtype=oracle.F32, flags=[0, 0], vocab_size=0)
    assert has.tolist() == [0, 0]


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.F16])
def test_apply_rows_against_numpy_and_indices(dtype):
    """The masked rows equal numpy's own bit unpacking applied to the flagged
    rows, the report equals numpy's any() over the unpacked bits, and the result
    equals the indexed apply on the list of flagged rows."""
    rng = np.random.default_rng(77)
    npdt = np.float32 if dtype == oracle.F32 else np.float16
    for _ in range(20):
        B = int(rng.integers(1, 7))
        cols = int(rng.integers(1, 200))
        vocab = int(rng.integers(0, cols + 1))
        words = (cols + 31) // 32
        bm = rng.integers(0, 2**32, size=(B, words), dtype=np.uint64).astype(np.uint32)
        if B > 1:
            bm[1] = 0
        bm = bm.view(np.int32)
        flags = rng.integers(0, 2, size=B).astype(np.uint8)
        x = rng.standard_normal((B, cols)).astype(npdt)
        out, has = oracle.apply_rows(x, bm, dtype=dtype, flags=flags, vocab_size=vocab)
        bits = np.unpackbits(bm.view(np.uint8), axis=1, bitorder="little")[:, :cols].astype(bool)
        drop = (flags[:, None] != 0) & ~bits & (np.arange(cols)[None, :] < vocab)
        want = np.where(drop, npdt(-np.inf), x)
        assert np.array_equal(out.view(np.uint8), want.view(np.uint8))
        keeps = ~drop & (np.arange(cols)[None, :] < vocab)
        assert has.tolist() == keeps.any(axis=1).astype(int).tolist()
        via_idx = oracle.apply(x, bm, dtype=dtype, vocab_size=vocab,
                               indices=np.flatnonzero(flags).astype(np.int32))
        assert np.array_equal(out.view(np.uint8), via_idx.view(np.uint8))


# ------------------------------------------- per-row seeds and slot parameters
# Kernel Hub "logits-processor", Ops, sample: the draw is keyed by (seed, row,
# offset); TensorRT-Edge-LLM "Guided Decoder": rows grouped rowsPerSlot to a slot.

def test_per_row_seeds_key_only_their_row():
    """With every row's seed equal to the call's seed the draw is the scalar
    seed's; a row's id depends on its own seed and not on the other rows'; and a
    row keyed by seed s is the row the scalar seed s draws."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((6, 500)) * 2).astype(np.float32)
    kw = dict(dtype=oracle.F32, temperature=1.1, top_p=0.95)
    base = oracle.mask_and_sample(x, seed=21, **kw)
    assert np.array_equal(oracle.mask_and_sample(x, seeds=[21] * 6, **kw), base)
    s1 = np.array([3, 4, 5, 6, 7, 8], dtype=np.uint64)
    s2 = s1.copy()
    s2[[0, 2, 5]] += 1000
    a, b = oracle.mask_and_sample(x, seeds=s1, **kw), oracle.mask_and_sample(x, seeds=s2, **kw)
    assert np.array_equal(a[[1, 3, 4]], b[[1, 3, 4]])
    for r in range(6):
        assert a[r] == oracle.mask_and_sample(x, seed=int(s1[r]), **kw)[r]
