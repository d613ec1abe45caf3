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
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grammar_constrained_logit_gb300 import ops
    from grammar_constrained_logit_gb300 import synthetic as syn

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rng = np.random.default_rng(12)
    shapes = [(64, 20000, torch.bfloat16, True), (300, 5000, torch.float32, False),
              (7, 70000, torch.float16, True), (64, 20000, torch.bfloat16, True)]
    for it, (B, V, dt, masked) in enumerate(shapes):
        x = torch.from_numpy((rng.standard_normal((B, V)) * 2).astype(np.float32)).cuda().to(dt)
        bm = None
        if masked:
            allowed = rng.random((B, V)) < 0.3
            bm = torch.from_numpy(syn.pack_bits(allowed)).cuda()
        want = ops.mask_and_sample(x, bm, 0.8, 30, 0.9, 0.02, seed=5, offset=it)
        got = torch.empty(B, dtype=torch.int64, device="cuda")
        p = _params(offset=it)
        st = lib.lp_mask_and_sample_noalloc(
            ctypes.c_void_p(x.data_ptr()), {torch.float32: 0, torch.float16: 1,
                                            torch.bfloat16: 2}[dt], B, V, V,
            ctypes.c_void_p(0 if bm is None else bm.data_ptr()),
            0 if bm is None else bm.size(0), 0 if bm is None else bm.size(1),
            0 if bm is None else bm.size(1), -1, None, 0, ctypes.byref(p),
            ctypes.c_void_p(got.data_ptr()), stream)
        assert st == _lib.LP_OK
        assert torch.equal(got, want), it
