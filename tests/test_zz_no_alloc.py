"""lp_mask_and_sample_noalloc: the sampler with the library's own device scratch
instead of a caller workspace.  It must give exactly the ids of
lp_mask_and_sample, leave its scratch valid for the next call (any shape), and
refuse sizes whose scratch exceeds what the library holds."""
import ctypes

import numpy as np
import pytest

from grammar_constrained_logit_gb300 import _lib

FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first


def _params(T=0.8, k=30, tp=0.9, mp=0.02, seed=5, offset=0):
    p = _lib.SamplingParams()
    p.temperature_scalar, p.top_k_scalar, p.top_p_scalar, p.min_p_scalar = T, k, tp, mp
    p.seed, p.offset = seed, offset
    return p


def test_noalloc_refuses_oversized_calls():
    lib = _lib.load()
    p = _params()
    # 2^20 rows of 2^17 tokens need far more than the library's 128 MiB
    st = lib.lp_mask_and_sample_noalloc(FAKE, 2, 1 << 20, 1 << 17, 1 << 17, None, 0, 0, 0, -1,
                                        None, 0, ctypes.byref(p), FAKE, None)
    assert st == _lib.LP_ERR_TOO_LARGE
    assert lib.lp_mask_and_sample_noalloc(None, 2, 0, 8, 8, None, 0, 0, 0, -1, None, 0,
                                          ctypes.byref(p), None, None) == _lib.LP_OK


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point():
    """Two rounds of calls of several shapes (an explicit vocab_size below the row
    width, an index list of masked rows, three dtypes): every id equals the one
    lp_mask_and_sample gives with a caller workspace, and is accepted by the
    oracle's tolerance rule.  The shared array's counters are left zero by each
    call (the same kernels keep a caller workspace's front zero, which the
    workspace-reuse parity test reads back)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grammar_constrained_logit_gb300 import ops
    from grammar_constrained_logit_gb300 import synthetic as syn
    from parity_check import check_ids

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rng = np.random.default_rng(12)
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    name = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    # (B, cols, dtype, masked, vocab_size or None, number of indexed rows or None)
    shapes = [(64, 20000, torch.bfloat16, True, None, None),
              (300, 5000, torch.float32, False, None, None),
              (7, 70000, torch.float16, True, None, None),
              (40, 9000, torch.float32, True, 8700, None),
              (48, 12000, torch.bfloat16, True, None, 20)]
    for rnd in range(2):
        for it, (B, V, dt, masked, vocab, nidx) in enumerate(shapes):
            off = 10 * rnd + it
            x32 = (rng.standard_normal((B, V)) * 2).astype(np.float32)
            x = torch.from_numpy(x32).cuda().to(dt)
            bm = idx = None
            bm_np = idx_np = None
            if masked:
                bm_np = syn.pack_bits(rng.random((B, V)) < 0.3)
                bm = torch.from_numpy(bm_np).cuda()
            if nidx is not None:
                idx_np = np.sort(rng.choice(B, size=nidx, replace=False)).astype(np.int32)
                idx = torch.from_numpy(idx_np).cuda()
            want = ops.mask_and_sample(x, bm, 0.8, 30, 0.9, 0.02, seed=5, offset=off,
                                       indices=idx, vocab_size=vocab)
            got = torch.empty(B, dtype=torch.int64, device="cuda")
            p = _params(offset=off)
            st = lib.lp_mask_and_sample_noalloc(
                ctypes.c_void_p(x.data_ptr()), code[dt], B, V, V,
                ctypes.c_void_p(0 if bm is None else bm.data_ptr()),
                0 if bm is None else bm.size(0), 0 if bm is None else bm.size(1),
                0 if bm is None else bm.size(1), -1 if vocab is None else vocab,
                ctypes.c_void_p(0 if idx is None else idx.data_ptr()),
                0 if idx is None else idx.numel(), ctypes.byref(p),
                ctypes.c_void_p(got.data_ptr()), stream)
            assert st == _lib.LP_OK
            assert torch.equal(got, want), (rnd, it)
            # the oracle's rule on the same inputs (bf16 compared on its bit patterns)
            st_np = syn.to_storage(x32, name[dt]) if dt != torch.float32 else x32
            prm = {"temperature": np.full(B, 0.8, np.float32), "top_k": np.full(B, 30, np.int32),
                   "top_p": np.full(B, 0.9, np.float32), "min_p": np.full(B, 0.02, np.float32)}
            check_ids(st_np, name[dt], got.cpu().numpy(), params=prm, seed=5, offset=off,
                      bitmask=bm_np, vocab_size=vocab, indices=idx_np, cols=V)
