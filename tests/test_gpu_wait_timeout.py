"""A bounded wait inside the streaming kernel made to run out, on the GPU.

The product build cannot reach this path on demand, so the test compiles its
own copy of the library with LP_TEST_FRESH_TIMEOUT set: one wait of CTA 0 (the
hand-over of a tile's shared state, a pure shared-memory poll with no copy in
flight) polls for a hand-over that never comes, 1000 times, and gives up.  The
CTA then marks its tiles from there on as failed, waits once more (bounded) for
the real hand-over, and carries on.  The call must return normally, the rows
of the failed tiles must report -2, every other row must equal the product
library's id, and the workspace must be left valid (its counters zero).
"""
import ctypes

import numpy as np
import pytest

from grammar_constrained_logit_gb300 import _lib
from grammar_constrained_logit_gb300 import build

pytestmark = pytest.mark.gpu


def test_tile_handover_wait_runs_out_and_rows_report_minus_two():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grammar_constrained_logit_gb300 import ops

    path = build.build_variant("fresh_timeout_test", {"LP_TEST_FRESH_TIMEOUT": 1000},
                               sources=("apply.cu", "sample.cu", "upload.cu"))
    lib = ctypes.CDLL(path)
    _lib.declare(lib)

    rng = np.random.default_rng(41)
    B, V = 64, 131072
    x = torch.from_numpy((rng.standard_normal((B, V)) * 2).astype(np.float32)).cuda()
    x = x.to(torch.bfloat16)
    args = dict(temperature=0.9, top_k=50, top_p=0.9, min_p=0.0, seed=7, offset=3)
    want = ops.sample(x, **args).cpu().numpy()

    nbytes = lib.lp_sample_workspace_bytes(_lib.LP_BF16, B, V)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(B, dtype=torch.int64, device="cuda")
    p = _lib.SamplingParams()
    p.temperature_scalar, p.top_k_scalar = args["temperature"], args["top_k"]
    p.top_p_scalar, p.min_p_scalar = args["top_p"], args["min_p"]
    p.seed, p.offset = args["seed"], args["offset"]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        st = lib.lp_sample(ctypes.c_void_p(x.data_ptr()), _lib.LP_BF16, B, V, V, ctypes.byref(p),
                           ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), nbytes,
                           stream)
        assert st == _lib.LP_OK
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        failed = got == -2
        assert failed.any(), "the forced timeout left no row reporting -2"
        assert not failed.all()
        assert np.array_equal(got[~failed], want[~failed])
        # the counters at the workspace's front are zero again
        assert int(ws[:4].count_nonzero()) == 0
        assert int(ws[256:256 + 4 * B].count_nonzero()) == 0
    # the product library still gives its ids on the same workspace
    again = ops.sample(x, **args, workspace=ws).cpu().numpy()
    assert np.array_equal(again, want)
