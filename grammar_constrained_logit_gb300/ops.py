"""PyTorch-facing binding of liblp.so.

Argument marshalling only: every op passes device pointers, sizes, strides and
the current CUDA stream to the C entry point of the same name (include/lp.h),
which does all of the work in its own kernels.  PyTorch supplies device memory
and streams.  The names follow the pages: ``apply_token_bitmask_inplace``
(XGrammar "Bitmask Operations"), ``apply_packed_bitmask`` (Modular MAX), and
``sample`` (Kernel Hub "logits-processor"); ``lp_*`` aliases carry the C names.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import torch

from . import _lib
from ._lib import SamplingParams, check

_DT = {torch.float32: _lib.LP_F32, torch.float16: _lib.LP_F16, torch.bfloat16: _lib.LP_BF16}


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"logits must be float32, float16 or bfloat16, not {t.dtype}") from None


def _matrix(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() == 1:
        t = t.unsqueeze(0)
    if t.dim() != 2:
        raise ValueError(f"{name} must be 1-D or 2-D, got {tuple(t.shape)}")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")
    return t


def _matrix_host(t: torch.Tensor) -> torch.Tensor:
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError("host bitmask must be 2-D with contiguous rows")
    return t


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _bitmask(bitmask: torch.Tensor, device) -> torch.Tensor:
    bm = _matrix(bitmask, "bitmask")
    if bm.dtype != torch.int32:
        raise TypeError("bitmask must be int32")
    if bm.device != device:
        raise ValueError("bitmask must be on the same device as logits")
    return bm


class _Indices:
    """Row list marshalled for the C ABI.  An empty list still needs a non-NULL
    pointer (NULL means "every row"), so it points at a one-element buffer."""

    def __init__(self, t: torch.Tensor):
        self.n = t.numel()
        self.t = t if self.n else torch.empty(1, dtype=torch.int32, device=t.device)

    def data_ptr(self):
        return self.t.data_ptr()

    def numel(self):
        return self.n


def _indices(indices, device):
    if indices is None:
        return None
    if isinstance(indices, torch.Tensor):
        idx = indices.to(device=device, dtype=torch.int32).contiguous().view(-1)
    else:
        idx = torch.tensor(list(indices), dtype=torch.int32, device=device)
    return _Indices(idx)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stride(t: torch.Tensor) -> int:
    return t.stride(0) if t.size(0) > 1 or t.size(1) <= 1 else max(t.stride(0), t.size(1))


def apply_token_bitmask_inplace(logits: torch.Tensor, bitmask: torch.Tensor, *,
                                vocab_size: int | None = None,
                                indices: Sequence[int] | torch.Tensor | None = None) -> None:
    """Set masked logits to -inf in place (bit 0 = masked, bit 1 = kept)."""
    lg = _matrix(logits, "logits")
    bm = _bitmask(bitmask, lg.device)
    idx = _indices(indices, lg.device)
    lib = _lib.load()
    st = lib.lp_apply_token_bitmask(
        _ptr(lg), _dtype_code(lg), lg.size(0), lg.size(1), _stride(lg), _ptr(bm), bm.size(0),
        bm.size(1), _stride(bm), -1 if vocab_size is None else int(vocab_size), _ptr(idx),
        0 if idx is None else idx.numel(), _stream(lg))
    check("lp_apply_token_bitmask", st)


lp_apply_token_bitmask = apply_token_bitmask_inplace


def apply_token_bitmask_rows(logits: torch.Tensor, bitmask: torch.Tensor,
                             row_needs_mask: torch.Tensor | None = None, *,
                             vocab_size: int | None = None,
                             report: bool = False) -> torch.Tensor | None:
    """Set masked logits to -inf in place in the rows whose ``row_needs_mask``
    flag (uint8 or bool, one per row) is nonzero; every row when it is None.
    With ``report``, returns int32 [B]: 1 where the row keeps a token after the
    call, 0 where its mask admits none (an unsatisfiable row)."""
    lg = _matrix(logits, "logits")
    bm = _bitmask(bitmask, lg.device)
    B = lg.size(0)
    flags = None
    if row_needs_mask is not None:
        if row_needs_mask.device != lg.device:
            raise ValueError("row_needs_mask must be on the same device as logits")
        flags = row_needs_mask.to(torch.uint8).contiguous().view(-1)
        if flags.numel() != B:
            raise ValueError(f"row_needs_mask must have {B} entries")
    has = torch.empty(B, dtype=torch.int32, device=lg.device) if report else None
    lib = _lib.load()
    st = lib.lp_apply_token_bitmask_rows(
        _ptr(lg), _dtype_code(lg), B, lg.size(1), _stride(lg), _ptr(bm), bm.size(0), bm.size(1),
        _stride(bm), -1 if vocab_size is None else int(vocab_size), _ptr(flags), _ptr(has),
        _stream(lg))
    check("lp_apply_token_bitmask_rows", st)
    return has


lp_apply_token_bitmask_rows = apply_token_bitmask_rows


def upload_bitmask(device_bitmask: torch.Tensor, host_bitmask: torch.Tensor, *,
                   device_flags: torch.Tensor | None = None,
                   host_flags: torch.Tensor | None = None,
                   copy_stream: torch.cuda.Stream | None = None,
                   event: torch.cuda.Event | None = None) -> torch.cuda.Event:
    """Copy a host-filled bitmask (int32 [rows, words], best page-locked) and,
    optionally, its uint8 row flags into device buffers on ``copy_stream`` (the
    current stream when None), then record ``event`` (a new one when None) after
    the copies and return it.  A compute stream waits on the event before an
    apply reads the mask; the host must not touch the host buffers until the
    event has completed."""
    if host_bitmask.is_cuda or not device_bitmask.is_cuda:
        raise ValueError("host_bitmask must be on the CPU and device_bitmask on the GPU")
    hb, db = _matrix_host(host_bitmask), _matrix(device_bitmask, "device_bitmask")
    if hb.dtype != torch.int32 or db.dtype != torch.int32:
        raise TypeError("bitmasks must be int32")
    rows, words = hb.size(0), hb.size(1)
    if db.size(0) < rows or db.size(1) < words:
        raise ValueError("device_bitmask is smaller than host_bitmask")
    if (device_flags is None) != (host_flags is None):
        raise ValueError("pass both row-flag buffers or neither")
    if host_flags is not None and (host_flags.numel() < rows or device_flags.numel() < rows or
                                   host_flags.dtype != torch.uint8 or
                                   device_flags.dtype != torch.uint8):
        raise ValueError("row flags must be uint8 with at least one entry per row")
    stream = copy_stream if copy_stream is not None else torch.cuda.current_stream(db.device)
    ev = event if event is not None else torch.cuda.Event()
    lib = _lib.load()
    # PyTorch creates an event's CUDA handle at its first record, so the event is
    # recorded here, on the copy stream right after the enqueued copies
    st = lib.lp_upload_bitmask(_ptr(db), _stride(db), _ptr(hb), _stride(hb), rows, words,
                               _ptr(device_flags), _ptr(host_flags),
                               ctypes.c_void_p(stream.cuda_stream), None)
    check("lp_upload_bitmask", st)
    ev.record(stream)
    return ev


lp_upload_bitmask = upload_bitmask


class BitmaskStager:
    """Double-buffered page-locked staging of the bitmask and its row flags.

    Each step: ``host()`` gives the host buffers to fill (after the upload that
    last used them has completed); ``upload()`` copies them to a device buffer
    on a copy stream and makes the current stream wait for that copy, returning
    the device buffers for the apply; ``consumed()`` marks, on the current
    stream, that the apply enqueued after ``upload`` is done with them, so that
    the copy two steps later may overwrite them."""

    def __init__(self, rows: int, words: int, device=None):
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.rows, self.words = rows, words
        self.host_mask = [torch.zeros(rows, words, dtype=torch.int32).pin_memory()
                          for _ in range(2)]
        self.host_flags = [torch.zeros(rows, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.dev_mask = [torch.zeros(rows, words, dtype=torch.int32, device=dev) for _ in range(2)]
        self.dev_flags = [torch.zeros(rows, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.uploaded = [None, None]
        self.released = [None, None]
        self.i = 0

    def host(self):
        """The host mask and flags of this step, free to fill."""
        if self.uploaded[self.i] is not None:
            self.uploaded[self.i].synchronize()
        return self.host_mask[self.i], self.host_flags[self.i]

    def upload(self):
        """Start this step's copy; the current stream waits for it.  Returns the
        device (mask, flags) the apply should read."""
        i = self.i
        if self.released[i] is not None:
            self.copy_stream.wait_event(self.released[i])
        ev = upload_bitmask(self.dev_mask[i], self.host_mask[i], device_flags=self.dev_flags[i],
                            host_flags=self.host_flags[i], copy_stream=self.copy_stream)
        self.uploaded[i] = ev
        torch.cuda.current_stream(self.dev_mask[i].device).wait_event(ev)
        return self.dev_mask[i], self.dev_flags[i]

    def consumed(self):
        """After enqueueing the apply: its device buffers may be reused later."""
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream(self.dev_mask[self.i].device))
        self.released[self.i] = ev
        self.i ^= 1


def apply_packed_bitmask(logits: torch.Tensor, bitmask: torch.Tensor,
                         fill_value: float = float("-inf"), *, out: torch.Tensor | None = None,
                         vocab_size: int | None = None,
                         indices: Sequence[int] | torch.Tensor | None = None) -> torch.Tensor:
    """Out-of-place apply: masked positions take ``fill_value``; returns ``out``."""
    lg = _matrix(logits, "logits")
    bm = _bitmask(bitmask, lg.device)
    if out is None:
        out = torch.empty_like(lg)
    o = _matrix(out, "out")
    if o.dtype != lg.dtype or o.shape != lg.shape:
        raise ValueError("out must match logits in dtype and shape")
    idx = _indices(indices, lg.device)
    lib = _lib.load()
    st = lib.lp_apply_packed_bitmask(
        _ptr(o), _stride(o), _ptr(lg), _dtype_code(lg), lg.size(0), lg.size(1), _stride(lg),
        _ptr(bm), bm.size(0), bm.size(1), _stride(bm), float(fill_value),
        -1 if vocab_size is None else int(vocab_size), _ptr(idx),
        0 if idx is None else idx.numel(), _stream(lg))
    check("lp_apply_packed_bitmask", st)
    return out


lp_apply_packed_bitmask = apply_packed_bitmask


def _param(v, B, dtype, device, keep):
    """A per-row parameter: (device pointer or None, scalar)."""
    if isinstance(v, torch.Tensor) and v.numel() != 1:
        if v.numel() != B:
            raise ValueError(f"per-row parameter must have {B} values, got {v.numel()}")
        t = v.to(device=device, dtype=dtype).contiguous()
        keep.append(t)
        return ctypes.c_void_p(t.data_ptr()), 0
    s = v.item() if isinstance(v, torch.Tensor) else v
    return None, (int(s) if dtype == torch.int32 else float(s))


def _params(B, device, temperature, top_k, top_p, min_p, seed, offset, keep):
    p = SamplingParams()
    p.temperature, p.temperature_scalar = _param(temperature, B, torch.float32, device, keep)
    p.top_k, p.top_k_scalar = _param(top_k, B, torch.int32, device, keep)
    p.top_p, p.top_p_scalar = _param(top_p, B, torch.float32, device, keep)
    p.min_p, p.min_p_scalar = _param(min_p, B, torch.float32, device, keep)
    p.seed = int(seed) & (2**64 - 1)
    p.offset = int(offset) & (2**64 - 1)
    return p


def _ids_out(out, B, device):
    if out is None:
        return torch.empty(B, dtype=torch.int64, device=device)
    if out.dtype != torch.int64 or out.numel() != B or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 tensor of B elements")
    return out


_workspaces: dict = {}


def sample_workspace_bytes(dtype: torch.dtype, batch_size: int, vocab_size: int) -> int:
    """Bytes of device scratch ``sample`` / ``mask_and_sample`` need."""
    n = _lib.load().lp_sample_workspace_bytes(_DT[dtype], batch_size, vocab_size)
    if n < 0:
        raise ValueError("invalid dtype or size")
    return int(n)


def _workspace(workspace, lg: torch.Tensor, B: int, vocab: int):
    """The caller's workspace (a uint8 CUDA tensor, zero-filled before its first
    use), or one kept per (device, stream), grown on demand; the library keeps its
    counters valid across calls.  When capturing a CUDA graph, pass an explicit
    workspace allocated before the capture: the capture stream would otherwise get
    a workspace of its own allocated (and zero-filled) inside the graph.
    Returns (pointer, bytes)."""
    need = sample_workspace_bytes(lg.dtype, B, max(vocab, 0))
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_contiguous() or \
                workspace.device != lg.device:
            raise ValueError("workspace must be a contiguous uint8 tensor on the logits' device")
        return ctypes.c_void_p(workspace.data_ptr()), workspace.numel()
    key = (lg.device.index, torch.cuda.current_stream(lg.device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=lg.device)
        _workspaces[key] = ws
    return ctypes.c_void_p(ws.data_ptr()), ws.numel()


def sample(logits: torch.Tensor, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0, seed: int = 0,
           offset: int = 0, *, vocab_size: int | None = None,
           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Temperature, top-k ∩ top-p ∩ min-p, Gumbel-max draw keyed by
    (seed, row, offset); greedy for temperature <= 0 or top_k == 1.  Every
    parameter is a scalar or a length-B tensor.  Returns int64 ids [B]."""
    lg = _matrix(logits, "logits")
    B = lg.size(0)
    V = lg.size(1) if vocab_size is None else int(vocab_size)
    keep: list = []
    p = _params(B, lg.device, temperature, top_k, top_p, min_p, seed, offset, keep)
    ids = _ids_out(out, B, lg.device)
    wp, wn = _workspace(workspace, lg, B, V)
    lib = _lib.load()
    st = lib.lp_sample(_ptr(lg), _dtype_code(lg), B, V, _stride(lg),
                       ctypes.byref(p), _ptr(ids), wp, wn, _stream(lg))
    check("lp_sample", st)
    return ids


lp_sample = sample


def mask_and_sample(logits: torch.Tensor, bitmask: torch.Tensor | None, temperature=1.0,
                    top_k=0, top_p=1.0, min_p=0.0, seed: int = 0, offset: int = 0, *,
                    indices: Sequence[int] | torch.Tensor | None = None,
                    vocab_size: int | None = None,
                    out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None) -> torch.Tensor:
    """The bitmask applied on the fly (logits are not written), then ``sample``.
    Rows in ``indices`` (all rows when None) are masked; a masked row whose mask
    admits no token returns -1."""
    lg = _matrix(logits, "logits")
    B = lg.size(0)
    bm = None if bitmask is None else _bitmask(bitmask, lg.device)
    idx = _indices(indices, lg.device)
    keep: list = []
    p = _params(B, lg.device, temperature, top_k, top_p, min_p, seed, offset, keep)
    ids = _ids_out(out, B, lg.device)
    # the workspace is sized by the widest vocabulary the call can use
    wp, wn = _workspace(workspace, lg, B, lg.size(1))
    lib = _lib.load()
    st = lib.lp_mask_and_sample(
        _ptr(lg), _dtype_code(lg), B, lg.size(1), _stride(lg), _ptr(bm),
        0 if bm is None else bm.size(0), 0 if bm is None else bm.size(1),
        0 if bm is None else _stride(bm), -1 if vocab_size is None else int(vocab_size),
        _ptr(idx), 0 if idx is None else idx.numel(), ctypes.byref(p), _ptr(ids), wp, wn,
        _stream(lg))
    check("lp_mask_and_sample", st)
    return ids


lp_mask_and_sample = mask_and_sample


def mask_and_sample_slots(logits: torch.Tensor, bitmask: torch.Tensor | None,
                          rows_per_slot: int, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0,
                          seed: int = 0, offset: int = 0, *,
                          seeds: torch.Tensor | None = None,
                          indices: Sequence[int] | torch.Tensor | None = None,
                          vocab_size: int | None = None,
                          out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None) -> torch.Tensor:
    """``mask_and_sample`` on [slots, rows_per_slot, V] logits (or their
    [slots * rows_per_slot, V] view): every sampling parameter is a scalar or
    one value per slot, shared by the slot's rows; ``seeds`` (optional, one
    uint64 per row, as int64 bit patterns) replaces ``seed`` row by row.
    Returns int64 ids [slots * rows_per_slot]."""
    if logits.dim() == 3:
        if logits.size(1) != rows_per_slot:
            raise ValueError("logits [slots, rows_per_slot, V] must match rows_per_slot")
        logits = logits.reshape(-1, logits.size(2))
    lg = _matrix(logits, "logits")
    B = lg.size(0)
    R = int(rows_per_slot)
    if R < 1 or B % R:
        raise ValueError("rows_per_slot must be >= 1 and divide the number of rows")
    bm = None if bitmask is None else _bitmask(bitmask.reshape(-1, bitmask.size(-1)), lg.device)
    idx = _indices(indices, lg.device)
    keep: list = []
    p = _params(B // R, lg.device, temperature, top_k, top_p, min_p, seed, offset, keep)
    sd = None
    if seeds is not None:
        sd = seeds.to(device=lg.device, dtype=torch.int64).contiguous().view(-1)
        if sd.numel() != B:
            raise ValueError(f"seeds must have {B} entries")
    ids = _ids_out(out, B, lg.device)
    wp, wn = _workspace(workspace, lg, B, lg.size(1))
    lib = _lib.load()
    st = lib.lp_mask_and_sample_slots(
        _ptr(lg), _dtype_code(lg), B, lg.size(1), _stride(lg), _ptr(bm),
        0 if bm is None else bm.size(0), 0 if bm is None else bm.size(1),
        0 if bm is None else _stride(bm), -1 if vocab_size is None else int(vocab_size),
        _ptr(idx), 0 if idx is None else idx.numel(), ctypes.byref(p), R, _ptr(sd), _ptr(ids),
        wp, wn, _stream(lg))
    check("lp_mask_and_sample_slots", st)
    return ids


lp_mask_and_sample_slots = mask_and_sample_slots


def philox4x32_10(counters: torch.Tensor, keys: torch.Tensor) -> torch.Tensor:
    """Device Philox4x32-10 on n blocks: counters [n, 4], keys [n, 2] (int32 bit
    patterns on the GPU) -> [n, 4] words (int32 bit patterns)."""
    c = counters.to(torch.int32).contiguous()
    k = keys.to(torch.int32).contiguous()
    if c.dim() != 2 or c.size(1) != 4 or k.shape != (c.size(0), 2) or not c.is_cuda:
        raise ValueError("counters must be [n, 4] and keys [n, 2], on the GPU")
    out = torch.empty_like(c)
    lib = _lib.load()
    check("lp_philox4x32_10",
          lib.lp_philox4x32_10(_ptr(c), _ptr(k), _ptr(out), c.size(0), _stream(c)))
    return out


lp_philox4x32_10 = philox4x32_10


def get_bitmask_shape(batch_size: int, vocab_size: int) -> tuple[int, int]:
    """(batch_size, ceil(vocab_size / 32)), the packed int32 bitmask shape."""
    return batch_size, (vocab_size + 31) // 32


bitmask_dtype = torch.int32
