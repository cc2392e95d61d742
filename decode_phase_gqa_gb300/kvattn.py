"""Thin ctypes binding of the C ABI in include/kvattn.h (same names).

Only argument marshalling happens here: shapes and dtypes are read off the
torch tensors, raw device pointers and the current CUDA stream are passed to
the library, and a non-zero status is raised as ``KvattnError``.  Every step
of the decode runs in the library's CUDA kernels; there is no Python or CPU
fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvattn.so")

KVATTN_OK = 0
KVATTN_EINVAL = 1
KVATTN_EUNSUPPORTED = 2
KVATTN_ECUDA = 3
KVATTN_EWORKSPACE = 4

KVATTN_KV_BF16 = 0
KVATTN_KV_INT8 = 1

KVATTN_DEV_BAD_LEN = 1
KVATTN_DEV_BAD_PAGE = 2
KVATTN_DEV_TIMEOUT = 4

KVATTN_MAX_SPLITS = 4096
KVATTN_MAX_SEQS = 8192
KVATTN_MAX_LAYERS = 1024
KVATTN_NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None
_lock = threading.Lock()


class KvattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = f"{what}: status {code} ({kvattn_status_string(code)})"
        if code == KVATTN_ECUDA:
            msg += f", cudaError {kvattn_last_cuda_error()}"
        super().__init__(msg)
        self.code = code


def bind(path: str) -> ctypes.CDLL:
    """Open a build of the library at `path` and declare its entry points."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "decode_phase_gqa_gb300.build.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.kvattn_workspace_size.argtypes = [I, I, I, I]
    L.kvattn_workspace_size.restype = S
    L.kvattn_workspace_size_layers.argtypes = [I, I, I, I, I]
    L.kvattn_workspace_size_layers.restype = S
    L.kvattn_workspace_init.argtypes = [P, S, P]
    L.kvattn_workspace_init.restype = I
    dec = [P] * 9 + [I] * 5 + [F, F, I, P, I, I, P, P, P, S]
    L.kvattn_decode.argtypes = dec
    L.kvattn_decode.restype = I
    L.kvattn_decode_splits.argtypes = dec + [I]
    L.kvattn_decode_splits.restype = I
    L.kvattn_decode_layers.argtypes = [I] + dec + [P]
    L.kvattn_decode_layers.restype = I
    L.kvattn_decode_noalloc.argtypes = dec[:-2] + [P]
    L.kvattn_decode_noalloc.restype = I
    L.kvattn_prefill.argtypes = [P] * 9 + [I] * 6 + [F, F, I, P, I, I, P, P, I, P, P, S]
    L.kvattn_prefill.restype = I
    L.kvattn_prefill_workspace_size.argtypes = [I, I, I]
    L.kvattn_prefill_workspace_size.restype = S
    L.kvattn_read_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    L.kvattn_read_device_status.restype = I
    L.kvattn_status_string.argtypes = [I]
    L.kvattn_status_string.restype = ctypes.c_char_p
    L.kvattn_version.argtypes = []
    L.kvattn_version.restype = I
    L.kvattn_last_cuda_error.argtypes = []
    L.kvattn_last_cuda_error.restype = I
    return L


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (fails loudly when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(path)
        return _lib


def kvattn_status_string(code: int) -> str:
    return load().kvattn_status_string(int(code)).decode()


def kvattn_version() -> int:
    return load().kvattn_version()


def kvattn_last_cuda_error() -> int:
    """cudaError_t value behind this thread's last KVATTN_ECUDA return (0: none)."""
    return int(load().kvattn_last_cuda_error())


def kvattn_workspace_size(n_seq: int, n_qh: int, n_kvh: int, head_dim: int) -> int:
    return int(load().kvattn_workspace_size(n_seq, n_qh, n_kvh, head_dim))


def kvattn_workspace_size_layers(n_layers: int, n_seq: int, n_qh: int, n_kvh: int,
                                 head_dim: int) -> int:
    return int(load().kvattn_workspace_size_layers(n_layers, n_seq, n_qh, n_kvh, head_dim))


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def kvattn_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    rc = load().kvattn_workspace_init(workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      _stream_handle(stream, workspace.device))
    if rc:
        raise KvattnError(rc, "kvattn_workspace_init")


def alloc_workspace(n_seq: int, n_qh: int, n_kvh: int, head_dim: int, device="cuda",
                    stream=None, n_layers: int = 1) -> torch.Tensor:
    """Device workspace for this shape (torch allocation, 256-byte aligned), initialised."""
    size = kvattn_workspace_size_layers(n_layers, n_seq, n_qh, n_kvh, head_dim)
    if size == 0:
        raise KvattnError(KVATTN_EINVAL, "kvattn_workspace_size")
    ws = torch.empty(size + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + size]
    kvattn_workspace_init(ws, stream)
    return ws


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtypes, ndim: int, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


_BF = (torch.bfloat16,)
_POOL = (torch.bfloat16, torch.int8)
_I32 = (torch.int32,)
_F32 = (torch.float32,)
_sig_lock = threading.Lock()
_sig_cache = {}  # argument signature -> the marshalled sizes (checks passed)


def _signature(tensors, layered: bool):
    """What the checks of _marshal depend on: shape, dtype, device index and
    contiguity of every tensor argument (None kept as None)."""
    return (layered,) + tuple(
        None if t is None else (t.shape, t.dtype, t.get_device(), t.is_contiguous())
        for t in tensors)


def _marshal(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
             k_scales, v_scales, layered: bool):
    """Shape/dtype checks; returns (n_layers, n_seq, n_qh, n_kvh, d, page, num_pages, int8).

    The checks run once per argument signature; a repeated signature (same
    shapes, dtypes, device and contiguity) reuses their result."""
    tensors = (q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
               k_scales, v_scales)
    try:
        key = _signature(tensors, layered)
    except AttributeError:
        raise TypeError("tensor arguments must be torch.Tensor or None") from None
    hit = _sig_cache.get(key)
    if hit is not None:
        return hit
    res = _marshal_checked(*tensors, layered)
    with _sig_lock:
        if len(_sig_cache) > 256:
            _sig_cache.clear()
        _sig_cache[key] = res
    return res


def _marshal_checked(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
                     k_scales, v_scales, layered: bool):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kvattn_decode runs on CUDA tensors only")
    e = 1 if layered else 0
    _check(q, "q", _BF, 3 + e, dev)
    _check(out, "out", _BF, 3 + e, dev)
    _check(k_new, "k_new", _BF, 3 + e, dev)
    _check(v_new, "v_new", _BF, 3 + e, dev)
    _check(k_pages, "k_pages", _POOL, 4 + e, dev)
    _check(v_pages, "v_pages", (k_pages.dtype,), 4 + e, dev)
    _check(block_table, "block_table", _I32, 2, dev)
    _check(seq_lens, "seq_lens", _I32, 1, dev)
    _check(positions, "positions", _I32, 1, dev)
    n_layers = q.shape[0] if layered else 1
    n_seq, n_qh, d = q.shape[e:]
    num_pages, n_kvh, page, d2 = k_pages.shape[e:]
    lead = (n_layers,) if layered else ()
    if (d2 != d or tuple(out.shape) != tuple(q.shape)
            or tuple(k_new.shape) != lead + (n_seq, n_kvh, d)
            or tuple(v_new.shape) != lead + (n_seq, n_kvh, d)
            or tuple(k_pages.shape) != lead + (num_pages, n_kvh, page, d)
            or tuple(v_pages.shape) != tuple(k_pages.shape)
            or block_table.shape[0] != n_seq or seq_lens.shape[0] != n_seq
            or positions.shape[0] != n_seq):
        raise ValueError("inconsistent shapes")
    int8 = k_pages.dtype == torch.int8
    if int8:
        for name, s in (("k_scales", k_scales), ("v_scales", v_scales)):
            if s is None:
                raise ValueError(f"{name} is required for an int8 cache")
            _check(s, name, _F32, 3 + e, dev)
            if tuple(s.shape) != lead + (num_pages, n_kvh, page):
                raise ValueError(f"{name}: shape {tuple(s.shape)}")
    return n_layers, n_seq, n_qh, n_kvh, d, page, num_pages, int8


def kvattn_decode(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
                  *, rope_theta: float, scale: float, workspace: torch.Tensor,
                  k_scales: Optional[torch.Tensor] = None, v_scales: Optional[torch.Tensor] = None,
                  num_splits: int = 0, stream=None) -> None:
    """One decode step (RoPE, append, attention) queued on ``stream``.

    Shapes: q/out [B, Hq, d] bf16; k_new/v_new [B, Hk, d] bf16; k_pages/v_pages
    [num_pages, Hk, page, d] bf16 or int8; block_table [B, max_pages] int32;
    seq_lens/positions [B] int32; k_scales/v_scales [num_pages, Hk, page] fp32
    (int8 only).  ``num_splits`` 0 = library default.
    """
    _, n_seq, n_qh, n_kvh, d, page, num_pages, int8 = _marshal(
        q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
        k_scales, v_scales, layered=False)
    rc = load().kvattn_decode_splits(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
        block_table.data_ptr(), seq_lens.data_ptr(), positions.data_ptr(), out.data_ptr(),
        n_seq, n_qh, n_kvh, d, page, float(rope_theta), float(scale),
        KVATTN_KV_INT8 if int8 else KVATTN_KV_BF16, _stream_handle(stream, q.device),
        block_table.shape[1], num_pages, _ptr(k_scales) if int8 else None,
        _ptr(v_scales) if int8 else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(num_splits))
    if rc:
        raise KvattnError(rc, "kvattn_decode")


def kvattn_decode_layers(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions,
                         out, *, rope_theta: float, scale: float, workspace: torch.Tensor,
                         k_scales: Optional[torch.Tensor] = None,
                         v_scales: Optional[torch.Tensor] = None, layer_rope=None,
                         stream=None) -> None:
    """One decode step over L layer caches in one launch (kvattn_decode_layers).

    Shapes as for ``kvattn_decode`` with a leading layer dimension L on q, out,
    k_new, v_new, k_pages, v_pages and the scales; block_table, seq_lens and
    positions are shared by all layers.  ``workspace`` from
    ``alloc_workspace(..., n_layers=L)``.  ``layer_rope``: None (every layer
    rotated) or L flags, false for a layer without RoPE.
    """
    n_layers, n_seq, n_qh, n_kvh, d, page, num_pages, int8 = _marshal(
        q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
        k_scales, v_scales, layered=True)
    flags = None
    if layer_rope is not None:
        if len(layer_rope) != n_layers:
            raise ValueError(f"layer_rope: {len(layer_rope)} flags for {n_layers} layers")
        flags = (ctypes.c_uint8 * n_layers)(*[1 if f else 0 for f in layer_rope])
    rc = load().kvattn_decode_layers(
        n_layers, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(),
        v_pages.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), positions.data_ptr(),
        out.data_ptr(), n_seq, n_qh, n_kvh, d, page, float(rope_theta), float(scale),
        KVATTN_KV_INT8 if int8 else KVATTN_KV_BF16, _stream_handle(stream, q.device),
        block_table.shape[1], num_pages, _ptr(k_scales) if int8 else None,
        _ptr(v_scales) if int8 else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(),
        None if flags is None else ctypes.cast(flags, ctypes.c_void_p))
    if rc:
        raise KvattnError(rc, "kvattn_decode_layers")


def kvattn_prefill(q, k_new, v_new, k_pages, v_pages, block_table, seq_starts, ctx_lens, out,
                   *, rope_theta: float, scale: float, max_new_tokens: int,
                   k_scales: Optional[torch.Tensor] = None, v_scales: Optional[torch.Tensor] = None,
                   dev_status: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Paged chunked prefill (kvattn_prefill): append the new tokens, then
    causal attention over the cache and the earlier new tokens.

    Shapes: q/out [T, Hq, d] bf16 (the new tokens of all sequences back to
    back); k_new/v_new [T, Hk, d] bf16; k_pages/v_pages [num_pages, Hk, page, d]
    bf16 or int8 (then k_scales/v_scales [num_pages, Hk, page] fp32); block_table [B, max_pages] int32; seq_starts [B + 1] int32; ctx_lens
    [B] int32; dev_status: None or a 1-element uint32/int32 device tensor that
    receives KVATTN_DEV_* bits; workspace: None or a device tensor of
    ``kvattn_prefill_workspace_size(T, Hq, d)`` bytes (for short chunks).
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kvattn_prefill runs on CUDA tensors only")
    bf = (torch.bfloat16,)
    _check(q, "q", bf, 3, dev)
    _check(out, "out", bf, 3, dev)
    _check(k_new, "k_new", bf, 3, dev)
    _check(v_new, "v_new", bf, 3, dev)
    _check(k_pages, "k_pages", (torch.bfloat16, torch.int8), 4, dev)
    _check(v_pages, "v_pages", (k_pages.dtype,), 4, dev)
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_starts, "seq_starts", (torch.int32,), 1, dev)
    _check(ctx_lens, "ctx_lens", (torch.int32,), 1, dev)
    n_tok, n_qh, d = q.shape
    num_pages, n_kvh, page, d2 = k_pages.shape
    n_seq = ctx_lens.shape[0]
    if (d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(k_new.shape) != (n_tok, n_kvh, d)
            or tuple(v_new.shape) != (n_tok, n_kvh, d) or tuple(v_pages.shape) != tuple(k_pages.shape)
            or block_table.shape[0] != n_seq or seq_starts.shape[0] != n_seq + 1):
        raise ValueError("inconsistent shapes")
    int8 = k_pages.dtype == torch.int8
    if int8:
        for name, s in (("k_scales", k_scales), ("v_scales", v_scales)):
            if s is None:
                raise ValueError(f"{name} is required for an int8 cache")
            _check(s, name, (torch.float32,), 3, dev)
            if tuple(s.shape) != (num_pages, n_kvh, page):
                raise ValueError(f"{name}: shape {tuple(s.shape)}")
    if dev_status is not None:
        _check(dev_status, "dev_status", (torch.int32, torch.uint32), 1, dev)
    rc = load().kvattn_prefill(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
        block_table.data_ptr(), seq_starts.data_ptr(), ctx_lens.data_ptr(), out.data_ptr(),
        n_seq, n_tok, n_qh, n_kvh, d, page, float(rope_theta), float(scale),
        KVATTN_KV_INT8 if int8 else KVATTN_KV_BF16, _stream_handle(stream, dev),
        block_table.shape[1], num_pages, _ptr(k_scales) if int8 else None,
        _ptr(v_scales) if int8 else None, int(max_new_tokens), _ptr(dev_status), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size())
    if rc:
        raise KvattnError(rc, "kvattn_prefill")


def kvattn_prefill_workspace_size(n_tok: int, n_qh: int, head_dim: int) -> int:
    return int(load().kvattn_prefill_workspace_size(n_tok, n_qh, head_dim))


def kvattn_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream, return and clear the sticky device status bits."""
    bits = ctypes.c_uint32(0)
    rc = load().kvattn_read_device_status(workspace.data_ptr(),
                                          _stream_handle(stream, workspace.device),
                                          ctypes.byref(bits))
    if rc:
        raise KvattnError(rc, "kvattn_read_device_status")
    return int(bits.value)
