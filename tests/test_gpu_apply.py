"""Bitmask apply on the GPU, bit-exact against the CPU oracle.

Covers float32 / float16 / bfloat16, vocabularies that are not multiples of 32,
padded logits and bitmask widths, explicit vocab_size, row strides that break
16-byte alignment, misaligned base pointers, index lists (with out-of-range and
duplicate entries), in place and out of place, canary columns past cols and
guard regions around every buffer, the empty cases, and the two apply
workloads at full size.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from grammar_constrained_logit_gb300 import ops  # noqa: E402
from grammar_constrained_logit_gb300 import synthetic as syn  # noqa: E402

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DT = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16}
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
CANARY = {"f32": np.float32(1234.5).view(np.uint32), "f16": np.uint16(0x7BFF),
          "bf16": np.uint16(0x4242)}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grammar_constrained_logit_gb300 import _lib

    _lib.load()


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32 if a.itemsize == 4 else np.uint16)


def _dev_view(storage: np.ndarray, dtype: str, guard: int, shift: int):
    """Place a [B, stride] storage array inside a larger device buffer, `guard`
    elements of canary on both sides and `shift` extra elements before it (to
    misalign the base pointer).  Returns (base tensor, 2-D view)."""
    B, stride = storage.shape
    n = B * stride
    flat = np.full(n + 2 * guard + shift, CANARY[dtype], dtype=_bits(storage).dtype)
    flat[guard + shift: guard + shift + n] = _bits(storage).reshape(-1)
    tdt = TDT[dtype]
    if dtype == "f32":
        base = torch.from_numpy(flat.view(np.float32)).cuda()
    elif dtype == "f16":
        base = torch.from_numpy(flat.view(np.float16)).cuda()
    else:
        base = torch.from_numpy(flat.view(np.int16)).cuda().view(torch.bfloat16)
    assert base.dtype == tdt
    view = base[guard + shift: guard + shift + n].view(B, stride)
    return base, view


def _host(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _check_guard(base, dtype, guard, shift, n):
    h = _bits(_host(base, dtype))
    assert np.all(h[:guard + shift] == CANARY[dtype])
    assert np.all(h[guard + shift + n:] == CANARY[dtype])


def test_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "apply_small.json")))
    first = np.array(g["cases"][0]["logits"], dtype=np.float32)
    for case in g["cases"]:
        logits = first if isinstance(case["logits"], str) else np.array(case["logits"], np.float32)
        bm = np.array([[int(h, 16) for h in row] for row in case["bitmask_hex"]],
                      dtype=np.uint32).view(np.int32)
        fill = float("-inf") if case["fill"] == "-inf" else float(case["fill"])
        x = torch.from_numpy(logits).cuda()
        b = torch.from_numpy(bm).cuda()
        if case["fill"] == "-inf":
            ops.apply_token_bitmask_inplace(x, b, vocab_size=case["vocab_size"],
                                            indices=case["indices"])
            out = x.cpu().numpy()
        else:
            out = ops.apply_packed_bitmask(x, b, fill, vocab_size=case["vocab_size"],
                                           indices=case["indices"]).cpu().numpy()
        for r, kept in enumerate(case["expected_kept"]):
            kept = set(kept)
            for j in range(logits.shape[1]):
                want = logits[r, j] if j in kept else np.float32(fill)
                assert out[r, j] == want, (case["name"], r, j)


def _random_case(rng, dtype):
    B = int(rng.integers(1, 9))
    cols = int(rng.choice([1, 5, 31, 32, 33, 100, 1003, 4099, 40000]))
    pad = int(rng.choice([0, 0, 1, 3, 8, 64]))
    vocab = [None, cols, max(0, cols - int(rng.integers(0, 40))), 0][int(rng.integers(0, 4))]
    need = ((cols if vocab is None else vocab) + 31) // 32
    words = max(need, 1) + int(rng.integers(0, 3))
    bm_pad = int(rng.integers(0, 3))
    bm_rows = B + int(rng.integers(0, 3))
    full = rng.integers(0, 2**32, size=(bm_rows, words + bm_pad), dtype=np.uint64).astype(np.uint32)
    style = int(rng.integers(0, 4))
    if style == 1:    # mostly masked, few runs: exercises the store-only path
        full &= rng.integers(0, 2**32, size=full.shape, dtype=np.uint64).astype(np.uint32)
        full &= rng.integers(0, 2**32, size=full.shape, dtype=np.uint64).astype(np.uint32)
    elif style == 2:  # whole words all-ones / all-zero
        full = np.where(rng.random(full.shape) < 0.5, np.uint32(0xFFFFFFFF), np.uint32(0))
        full = full.astype(np.uint32)
    bm = np.ascontiguousarray(full.view(np.int32))
    x = (rng.standard_normal((B, cols + pad)) * 3).astype(np.float32)
    logits = syn.to_storage(x, dtype)
    idx = None
    r = int(rng.integers(0, 3))
    if r == 1:
        idx = rng.choice(B, size=int(rng.integers(0, B + 1)), replace=False).astype(np.int32)
    elif r == 2:
        idx = np.array([B - 1, -1, B + 7, 0, 0], dtype=np.int32)  # invalid + duplicate
    return B, cols, vocab, words, bm, logits, idx


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("inplace", [True, False])
def test_random_parity(dtype, inplace):
    rng = np.random.default_rng(1000 + 10 * DT[dtype] + int(inplace))
    for trial in range(40):
        B, cols, vocab, words, bm, logits, idx = _random_case(rng, dtype)
        stride = logits.shape[1]
        guard, shift = 64, int(rng.integers(0, 3))
        base, view = _dev_view(logits, dtype, guard, shift)
        lv = view[:, :cols]
        bm_words_view = torch.from_numpy(bm).cuda()[:, :words]
        fill = float("-inf") if inplace or trial % 2 == 0 else float(rng.standard_normal() * 50)
        want = oracle.apply(logits, bm[:, :words], dtype=DT[dtype], fill=fill, vocab_size=vocab,
                            indices=idx, cols=cols)
        if inplace:
            ops.apply_token_bitmask_inplace(lv, bm_words_view, vocab_size=vocab, indices=idx)
            got = _host(view, dtype)
            assert np.array_equal(_bits(got), _bits(want)), (trial, dtype, B, cols, vocab, idx)
            _check_guard(base, dtype, guard, shift, B * stride)
        else:
            canary = np.full(logits.shape, CANARY[dtype], dtype=_bits(logits).dtype)
            obase, oview = _dev_view(canary.view(logits.dtype), dtype, guard,
                                     int(rng.integers(0, 3)))
            ops.apply_packed_bitmask(lv, bm_words_view, fill, out=oview[:, :cols],
                                     vocab_size=vocab, indices=idx)
            got = _bits(_host(oview, dtype))
            assert np.array_equal(got[:, :cols], _bits(want)[:, :cols]), (trial, dtype, B, cols)
            assert np.all(got[:, cols:] == CANARY[dtype])     # padding never written
            assert np.array_equal(_bits(_host(view, dtype)), _bits(logits))  # input untouched


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_rows_parity(dtype):
    """Per-row flags and the keeps-a-token report, bit-exact against the oracle;
    some flagged rows have an all-zero mask (report 0), and the report buffer is
    zeroed by the call whatever it held."""
    rng = np.random.default_rng(2000 + DT[dtype])
    for trial in range(30):
        B, cols, vocab, words, bm, logits, _ = _random_case(rng, dtype)
        bm = bm.copy()
        bm_rows = bm.shape[0]
        if B > 1:
            bm[int(rng.integers(0, B))] = 0
        flags = rng.integers(0, 2, size=B).astype(np.uint8) if trial % 3 else None
        stride = logits.shape[1]
        guard, shift = 64, int(rng.integers(0, 3))
        base, view = _dev_view(logits, dtype, guard, shift)
        want, want_has = oracle.apply_rows(logits, bm[:, :words], dtype=DT[dtype], flags=flags,
                                           vocab_size=vocab, cols=cols)
        fl = None if flags is None else torch.from_numpy(flags).cuda()
        has = ops.apply_token_bitmask_rows(view[:, :cols], torch.from_numpy(bm).cuda()[:, :words],
                                           fl, vocab_size=vocab, report=True)
        got = _host(view, dtype)
        assert np.array_equal(_bits(got), _bits(want)), (trial, dtype, B, cols, vocab)
        assert has.cpu().numpy().tolist() == want_has.tolist(), (trial, dtype, B, cols, vocab)
        _check_guard(base, dtype, guard, shift, B * stride)
        assert bm_rows >= B


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_report_single_token_anywhere(dtype):
    """Flagged rows that keep exactly one token: in the ragged head before the
    first 16-byte boundary, past the first block's tokens, in the last partial
    word below vocab_size, just above vocab_size (not kept), or none at all; the
    report and the logits match the oracle bit for bit."""
    rng = np.random.default_rng(4100 + DT[dtype])
    B, V = 48, 40007
    words = (V + 31) // 32
    vocab = V - 5
    logits = syn.to_storage(rng.standard_normal((B, V)).astype(np.float32), dtype)
    allowed = np.zeros((B, words * 32), dtype=bool)
    spots = [0, 1, 2, 3, 7, 9000, 20000, 33000, vocab - 1, vocab - 2, vocab, V - 1]
    for r in range(B):
        if r % 8 == 7:
            continue  # no token at all
        allowed[r, spots[r % len(spots)] if r < 24 else int(rng.integers(0, V))] = True
    bm = syn.pack_bits(allowed)
    flags = np.ones(B, dtype=np.uint8)
    flags[5] = 0
    guard, shift = 64, 1
    base, view = _dev_view(logits, dtype, guard, shift)
    want, want_has = oracle.apply_rows(logits, bm, dtype=DT[dtype], flags=flags,
                                       vocab_size=vocab, cols=V)
    has = ops.apply_token_bitmask_rows(view[:, :V], torch.from_numpy(bm).cuda(),
                                       torch.from_numpy(flags).cuda(), vocab_size=vocab,
                                       report=True)
    assert np.array_equal(_bits(_host(view, dtype)), _bits(want))
    assert has.cpu().numpy().tolist() == want_has.tolist()
    _check_guard(base, dtype, guard, shift, B * logits.shape[1])


def test_rows_report_overwrites_and_without_report():
    x = torch.zeros(3, 100, device="cuda")
    bm = torch.zeros(3, 4, dtype=torch.int32, device="cuda")
    bm[2, 0] = 1
    has = ops.apply_token_bitmask_rows(x, bm, torch.tensor([1, 0, 1], dtype=torch.uint8,
                                                           device="cuda"), report=True)
    assert has.cpu().tolist() == [0, 1, 1]
    assert torch.isinf(x[0]).all() and not torch.isinf(x[1]).any()
    assert x[2, 0] == 0 and torch.isinf(x[2, 1:]).all()
    # no flags: every row is masked; no report
    assert ops.apply_token_bitmask_rows(x, bm, None) is None
    assert torch.isinf(x[1]).all() and x[2, 0] == 0


def test_apply_only_workload_as_row_flags():
    """The 32 indexed rows of the bf16 apply workload given as per-row flags: the
    same logits as the indexed apply, and a report of every row."""
    w = syn.apply_only()
    flags = np.zeros(w.B, dtype=np.uint8)
    flags[w.indices] = 1
    want, want_has = oracle.apply_rows(w.logits, w.bitmask, dtype=oracle.BF16, flags=flags,
                                       vocab_size=w.vocab_size, cols=w.cols)
    x = torch.from_numpy(w.logits.view(np.int16)).cuda().view(torch.bfloat16)
    has = ops.apply_token_bitmask_rows(x[:, :w.cols], torch.from_numpy(w.bitmask).cuda(),
                                       torch.from_numpy(flags).cuda(), vocab_size=w.vocab_size,
                                       report=True)
    assert np.array_equal(_host(x, "bf16"), want)
    assert has.cpu().numpy().tolist() == want_has.tolist()


def test_upload_then_apply_on_another_stream():
    """A host-filled mask and row flags, copied on a side stream and signalled by
    an event: the apply on the current stream, after waiting on the event, masks
    exactly as the oracle does with the host mask."""
    rng = np.random.default_rng(31)
    B, cols = 16, 5000
    words = (cols + 31) // 32
    x = (rng.standard_normal((B, cols)) * 2).astype(np.float32)
    hm = torch.from_numpy(rng.integers(0, 2**32, size=(B, words), dtype=np.uint64)
                          .astype(np.uint32).view(np.int32)).pin_memory()
    hf = torch.from_numpy((rng.random(B) < 0.5).astype(np.uint8)).pin_memory()
    dm = torch.zeros(B, words + 3, dtype=torch.int32, device="cuda")[:, :words]
    dfl = torch.zeros(B, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    ev = ops.upload_bitmask(dm, hm, device_flags=dfl, host_flags=hf, copy_stream=side)
    torch.cuda.current_stream().wait_event(ev)
    xd = torch.from_numpy(x).cuda()
    has = ops.apply_token_bitmask_rows(xd, dm, dfl, report=True)
    want, want_has = oracle.apply_rows(x, hm.numpy(), dtype=oracle.F32, flags=hf.numpy())
    assert np.array_equal(xd.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert has.cpu().numpy().tolist() == want_has.tolist()


def test_bitmask_stager_steps():
    """Five steps through the double-buffered stager, each with a new mask and new
    flags filled on the host: every apply sees its own step's mask."""
    rng = np.random.default_rng(32)
    B, cols = 8, 3000
    words = (cols + 31) // 32
    st = ops.BitmaskStager(B, words)
    for step in range(5):
        hm, hf = st.host()
        m = rng.integers(0, 2**32, size=(B, words), dtype=np.uint64).astype(np.uint32)
        f = (rng.random(B) < 0.6).astype(np.uint8)
        hm.copy_(torch.from_numpy(m.view(np.int32)))
        hf.copy_(torch.from_numpy(f))
        dm, dfl = st.upload()
        x = (rng.standard_normal((B, cols))).astype(np.float32)
        xd = torch.from_numpy(x).cuda()
        ops.apply_token_bitmask_rows(xd, dm, dfl)
        st.consumed()
        want, _ = oracle.apply_rows(x, m.view(np.int32), dtype=oracle.F32, flags=f)
        assert np.array_equal(xd.cpu().numpy().view(np.uint32), want.view(np.uint32)), step


def test_empty_cases():
    x = torch.randn(3, 40, device="cuda")
    ref = x.clone()
    bm = torch.zeros(3, 2, dtype=torch.int32, device="cuda")
    ops.apply_token_bitmask_inplace(x, bm, vocab_size=0)
    ops.apply_token_bitmask_inplace(x, bm, indices=[])
    ops.apply_token_bitmask_inplace(x[:0], bm[:0])
    assert torch.equal(x, ref)
    out = ops.apply_packed_bitmask(x, bm, 0.0, vocab_size=0)
    assert torch.equal(out, ref)


def test_all_ones_is_identity_and_all_zero_fills():
    for tdt in (torch.float32, torch.float16, torch.bfloat16):
        x = torch.randn(5, 777, device="cuda").to(tdt)
        ref = x.clone()
        ops.apply_token_bitmask_inplace(x, torch.full((5, 25), -1, dtype=torch.int32, device="cuda"))
        assert torch.equal(x, ref)
        ops.apply_token_bitmask_inplace(x, torch.zeros(5, 25, dtype=torch.int32, device="cuda"))
        assert torch.all(torch.isneginf(x))


def test_in_place_through_out_of_place_entry():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 1000)).astype(np.float32)
    bm = rng.integers(0, 2**32, size=(6, 32), dtype=np.uint64).astype(np.uint32).view(np.int32)
    t = torch.from_numpy(x).cuda()
    ops.apply_packed_bitmask(t, torch.from_numpy(bm).cuda(), -7.0, out=t, indices=[4, 1])
    want = oracle.apply(x, bm, dtype=oracle.F32, fill=-7.0, indices=[4, 1])
    assert np.array_equal(t.cpu().numpy(), want)


def test_large_bitmap_out_of_place_path():
    """More rows than the per-block selection bitmap holds: copy, then mask."""
    B, V = 400_000, 32
    rng = np.random.default_rng(6)
    x = rng.standard_normal((B, V)).astype(np.float32)
    bm = rng.integers(0, 2**32, size=(B, 1), dtype=np.uint64).astype(np.uint32).view(np.int32)
    idx = rng.choice(B, size=1000, replace=False).astype(np.int32)
    out = ops.apply_packed_bitmask(torch.from_numpy(x).cuda(), torch.from_numpy(bm).cuda(),
                                   -1.0, indices=torch.from_numpy(idx))
    want = oracle.apply(x, bm, dtype=oracle.F32, fill=-1.0, indices=idx)
    assert np.array_equal(out.cpu().numpy(), want)


def test_bad_arguments_raise():
    from grammar_constrained_logit_gb300._lib import LPError

    x = torch.randn(2, 64, device="cuda")
    with pytest.raises(LPError):
        ops.apply_token_bitmask_inplace(x, torch.zeros(2, 1, dtype=torch.int32, device="cuda"),
                                        vocab_size=64)
    with pytest.raises(LPError):
        ops.apply_token_bitmask_inplace(x, torch.zeros(1, 2, dtype=torch.int32, device="cuda"))


def _run_workload_apply(w, inplace: bool):
    dtype = w.dtype
    logits = w.logits
    base, view = _dev_view(logits, dtype, 128, 0)
    lv = view[:, :w.cols]
    bm = torch.from_numpy(w.bitmask).cuda()
    idx = None if w.indices is None else torch.from_numpy(w.indices).cuda()
    want = oracle.apply(logits, w.bitmask, dtype=DT[dtype], vocab_size=w.vocab_size,
                        indices=w.indices, cols=w.cols)
    if inplace:
        ops.apply_token_bitmask_inplace(lv, bm, vocab_size=w.vocab_size, indices=idx)
        got = _bits(_host(view, dtype))
    else:
        out = torch.empty_like(view)
        ops.apply_packed_bitmask(lv, bm, out=out[:, :w.cols], vocab_size=w.vocab_size, indices=idx)
        got = _bits(_host(out, dtype))[:, :w.cols]
        want = want[:, :w.cols]
    assert np.array_equal(got, _bits(want)[:, :got.shape[1]])
    _check_guard(base, dtype, 128, 0, logits.size)


def test_tiny_greedy_workload_apply():
    _run_workload_apply(syn.tiny_greedy(), True)


@pytest.mark.parametrize("inplace", [True, False])
def test_apply_only_workload_full_size(inplace):
    """B=64 bf16 rows padded to 128512 columns, vocab 128256, 1% grammar-like
    mask, 32 indexed rows: every element bit-exact."""
    _run_workload_apply(syn.apply_only(), inplace)


def test_speculative_verify_workload_apply_full_size():
    """1024 fp16 rows x 202048, 512 indexed rows with grammar-like masks."""
    _run_workload_apply(syn.speculative_verify(), True)
