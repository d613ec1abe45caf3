"""CPU oracle for grammar-constrained logit masking and fused sampling.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check
(``__graft_entry__.smoke``) and the CPU-baseline leg of ``bench.py`` may import
this package.  The product path (the CUDA library and its binding) never does,
and this package imports nothing from the product: the two share no code.

The arithmetic lives in ``lp_oracle.c`` (plain C, double precision); this module
only compiles it with the system C compiler and marshals numpy arrays.  Every
function cites, in ``lp_oracle.c``, the page section it restates:

* XGrammar "Bitmask Operations" -- ``apply_token_bitmask_inplace`` (the row/token
  double loop, the Padding and Indices notes);
* Modular MAX "apply_packed_bitmask" -- out-of-place apply with a fill value;
* Kernel Hub "logits-processor" -- "Ops", "Correctness" and "How it works" for
  greedy, temperature, top-k / top-p / min-p and the Gumbel-max draw;
* TensorRT-Edge-LLM "Guided Decoder" -- an all-zero mask row is unsatisfiable;
* Salmon et al., SC'11 -- Philox4x32-10.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against values that do not come from this code:
numpy bit unpacking, numpy argmax, a brute-force pointwise keep-set on tiny
vocabularies, PyTorch's own Philox engine header, hand-worked golden cases under
``tests/golden/``, and goodness-of-fit of the draws to the exact distribution.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lp_oracle.c")
_LIB = os.path.join(_HERE, "liblp_oracle.so")

F32, F16, BF16 = 0, 1, 2
_DT = {np.dtype(np.float32): F32, np.dtype(np.float16): F16}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``lp_oracle.c`` into ``liblp_oracle.so`` (gcc -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, i32, u64, u32 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32
    vp = ctypes.c_void_p
    lib.lpo_apply.restype = i32
    lib.lpo_apply.argtypes = [vp, i64, vp, i32, i64, i64, i64, vp, i64, i64, i64,
                              ctypes.c_float, i64, vp, i64]
    lib.lpo_apply_rows.restype = i32
    lib.lpo_apply_rows.argtypes = [vp, i32, i64, i64, i64, vp, i64, i64, i64, i64, vp, vp]
    lib.lpo_mask_and_sample.restype = i32
    lib.lpo_mask_and_sample.argtypes = [vp, i32, i64, i64, i64, vp, i64, i64, i64, i64,
                                        vp, i64, vp, vp, vp, vp, u64, u64, vp, vp, vp, vp, vp]
    lib.lpo_philox4x32_10.restype = None
    lib.lpo_philox4x32_10.argtypes = [vp, vp, vp]
    lib.lpo_random_word.restype = u32
    lib.lpo_random_word.argtypes = [u64, u64, u64, u64]
    lib.lpo_uniform.restype = ctypes.c_double
    lib.lpo_uniform.argtypes = [u32]
    lib.lpo_gumbel.restype = ctypes.c_double
    lib.lpo_gumbel.argtypes = [u32]
    lib.lpo_encode.restype = u32
    lib.lpo_encode.argtypes = [ctypes.c_float, i32]
    lib.lpo_decode.restype = ctypes.c_double
    lib.lpo_decode.argtypes = [u32, i32]
    lib.lpo_resolve_vocab.restype = i64
    lib.lpo_resolve_vocab.argtypes = [i64, i64, i64]
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def dtype_code(a: np.ndarray, bf16: bool = False) -> int:
    """Dtype code of a logits array.  bfloat16 arrays are carried as uint16 bit
    patterns, so the caller states ``bf16=True`` for them."""
    if bf16:
        assert a.dtype == np.uint16
        return BF16
    return _DT[a.dtype]


def resolve_vocab(vocab_size, cols, bitmask_words) -> int:
    return int(_load().lpo_resolve_vocab(-1 if vocab_size is None else vocab_size,
                                         cols, bitmask_words))


def apply(logits: np.ndarray, bitmask: np.ndarray, *, dtype: int, fill: float = float("-inf"),
          vocab_size=None, indices=None, cols=None, out: np.ndarray | None = None) -> np.ndarray:
    """Masked copy of ``logits`` (a 2-D array of the dtype's storage type).

    ``cols`` is the logical width of each row (default: the array width; a wider
    array models a padded row stride).  Returns ``out`` (a fresh copy when None).
    """
    lib = _load()
    logits = np.ascontiguousarray(logits)
    bitmask = np.ascontiguousarray(bitmask, dtype=np.int32)
    B, stride = logits.shape
    cols = stride if cols is None else cols
    if out is None:
        out = logits.copy()
    idx = None if indices is None else np.ascontiguousarray(indices, dtype=np.int32)
    rc = lib.lpo_apply(_ptr(out), out.shape[1], _ptr(logits), dtype, B, cols, stride,
                       _ptr(bitmask), bitmask.shape[0], bitmask.shape[1], bitmask.shape[1],
                       float(fill), -1 if vocab_size is None else int(vocab_size),
                       _ptr(idx), 0 if idx is None else idx.size)
    if rc != 0:
        raise ValueError("inconsistent geometry")
    return out


def apply_rows(logits: np.ndarray, bitmask: np.ndarray, *, dtype: int, flags=None,
               vocab_size=None, cols=None):
    """In-place apply on the rows whose flag is nonzero (all rows for None), on a
    copy of ``logits``; returns (masked copy, int32 per-row "keeps a token")."""
    lib = _load()
    out = np.ascontiguousarray(logits).copy()
    bitmask = np.ascontiguousarray(bitmask, dtype=np.int32)
    B, stride = out.shape
    cols = stride if cols is None else cols
    fl = None if flags is None else np.ascontiguousarray(flags, dtype=np.uint8)
    has = np.zeros(B, dtype=np.int32)
    rc = lib.lpo_apply_rows(_ptr(out), dtype, B, cols, stride, _ptr(bitmask), bitmask.shape[0],
                            bitmask.shape[1], bitmask.shape[1],
                            -1 if vocab_size is None else int(vocab_size), _ptr(fl), _ptr(has))
    if rc != 0:
        raise ValueError("inconsistent geometry")
    return out, has


def _per_row(x, B, dt):
    a = np.asarray(x, dtype=dt)
    if a.ndim == 0:
        a = np.full(B, a, dtype=dt)
    assert a.shape == (B,)
    return np.ascontiguousarray(a)


def mask_and_sample(logits: np.ndarray, *, dtype: int, bitmask=None, vocab_size=None,
                    indices=None, cols=None, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0,
                    seed: int = 0, offset: int = 0, row_ids=None, want_keep: bool = False,
                    want_p: bool = False, want_thr: bool = False, seeds=None):
    """Per-row greedy / filtered Gumbel-max sampling (double precision).

    ``row_ids`` (optional, one per array row) gives each row's logical index,
    which keys the noise and addresses the bitmask (default 0..B-1), so a subset
    of a batch can be checked on its own.  Returns ids (int64 [B]) and, when
    asked, keep flags [B, V] (bool), probabilities [B, V] and thresholds [B] as a
    tuple (ids, keep, p, thr).  ``seeds`` (optional, one per row) keys each row's
    noise with its own seed: rows are independent, so each row is then sampled
    on its own with its seed and its logical row index."""
    if seeds is not None:
        n = np.ascontiguousarray(logits).shape[0]
        sd = [int(x) & (2**64 - 1) for x in np.asarray(seeds).astype(np.uint64).reshape(-1)]
        assert len(sd) == n
        rid = np.arange(n) if row_ids is None else np.asarray(row_ids)
        parts = []
        for b in range(n):
            one = lambda x: x if np.ndim(x) == 0 else np.asarray(x)[b:b + 1]  # noqa: E731
            parts.append(mask_and_sample(
                np.ascontiguousarray(logits)[b:b + 1], dtype=dtype, bitmask=bitmask,
                vocab_size=vocab_size, indices=indices, cols=cols,
                temperature=one(temperature), top_k=one(top_k), top_p=one(top_p),
                min_p=one(min_p), seed=sd[b], offset=offset, row_ids=rid[b:b + 1],
                want_keep=want_keep, want_p=want_p, want_thr=want_thr))
        if not (want_keep or want_p or want_thr):
            return np.concatenate(parts)
        cat = lambda k: None if parts[0][k] is None else np.concatenate([q[k] for q in parts])  # noqa: E731
        return cat(0), cat(1), cat(2), cat(3)
    lib = _load()
    logits = np.ascontiguousarray(logits)
    B, stride = logits.shape
    cols = stride if cols is None else cols
    bm = None if bitmask is None else np.ascontiguousarray(bitmask, dtype=np.int32)
    words = 0 if bm is None else bm.shape[1]
    if bm is not None:
        V = resolve_vocab(vocab_size, cols, words)
    else:
        V = cols if vocab_size is None else int(vocab_size)
    idx = None if indices is None else np.ascontiguousarray(indices, dtype=np.int32)
    T = _per_row(temperature, B, np.float32)
    K = _per_row(top_k, B, np.int32)
    P = _per_row(top_p, B, np.float32)
    M = _per_row(min_p, B, np.float32)
    rid = None if row_ids is None else np.ascontiguousarray(row_ids, dtype=np.int64)
    assert rid is None or rid.shape == (B,)
    ids = np.empty(B, dtype=np.int64)
    keep = np.empty((B, V), dtype=np.uint8) if want_keep else None
    p = np.empty((B, V), dtype=np.float64) if want_p else None
    thr = np.empty(B, dtype=np.float64) if want_thr else None
    rc = lib.lpo_mask_and_sample(
        _ptr(logits), dtype, B, cols, stride, _ptr(bm), 0 if bm is None else bm.shape[0],
        words, words, -1 if vocab_size is None else int(vocab_size), _ptr(idx),
        0 if idx is None else idx.size, _ptr(T), _ptr(K), _ptr(P), _ptr(M),
        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(rid), _ptr(ids), _ptr(keep),
        _ptr(p), _ptr(thr))
    if rc != 0:
        raise ValueError("inconsistent geometry")
    if not (want_keep or want_p or want_thr):
        return ids
    return ids, (None if keep is None else keep.astype(bool)), p, thr


def philox4x32_10(ctr, key) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib.lpo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def random_word(seed: int, offset: int, row: int, v: int) -> int:
    return int(_load().lpo_random_word(seed, offset, row, v))


def uniform(x: int) -> float:
    return float(_load().lpo_uniform(x))


def gumbel(x: int) -> float:
    return float(_load().lpo_gumbel(x))


def encode(x: float, dtype: int) -> int:
    return int(_load().lpo_encode(float(x), dtype))


def decode(bits: int, dtype: int) -> float:
    return float(_load().lpo_decode(int(bits), dtype))
