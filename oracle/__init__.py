"""CPU oracle for one decode step of GQA attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path (the CUDA library and
its Python binding) never imports this package, and this package never imports
the product.  The arithmetic lives in ``oracle.c`` (plain C, IEEE double); this
module builds it with gcc and marshals numpy arrays into it.

bf16 data is passed as ``numpy.uint16`` arrays holding the bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

BAD_LEN = 1
BAD_PAGE = 2

_lib = None
_lock = threading.Lock()


def build(verbose: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (OpenMP when available).

    -ffp-contract=off keeps every product and sum separately rounded, as the
    storage recipe states; no fast-math.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", src, "-o", out + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(out + ".tmp", out)
            if verbose:
                print(" ".join(cmd))
            return out
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def lib() -> ctypes.CDLL:
    """Load the oracle library (building it first when the source is newer).

    ORACLE_LIB_OVERRIDE names another build of oracle.c to load instead; the
    mutation test uses it to check that the pins reject planted mistakes.
    """
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIB_OVERRIDE")
            if not path:
                if _stale():
                    build()
                path = _LIB_PATH
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            F = ctypes.c_float
            D = ctypes.c_double
            L.oracle_rope_f64.argtypes = [P, I, D, D, P]
            L.oracle_rope_f64.restype = None
            L.oracle_rope_store_f32.argtypes = [P, I, I, F, P]
            L.oracle_rope_store_f32.restype = None
            L.oracle_quant_int8.argtypes = [P, I, P, P]
            L.oracle_quant_int8.restype = None
            L.oracle_append.argtypes = [P] * 9 + [I] * 4 + [F] + [I] * 3
            L.oracle_append.restype = ctypes.c_uint
            L.oracle_attend_paged.argtypes = [P] * 9 + [I] * 5 + [F, F] + [I] * 3 + [P, I]
            L.oracle_attend_paged.restype = ctypes.c_uint
            L.oracle_attend_contiguous.argtypes = [P] * 6 + [I] * 4 + [F, F]
            L.oracle_attend_contiguous.restype = None
            L.oracle_decode.argtypes = [P] * 11 + [I] * 5 + [F, F] + [I] * 3 + [P, I]
            L.oracle_decode.restype = ctypes.c_uint
            L.oracle_max_threads.argtypes = []
            L.oracle_max_threads.restype = I
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _req(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError("array must be C-contiguous")
    return a


def max_threads() -> int:
    return lib().oracle_max_threads()


# ------------------------------------------------------------------ pieces --

def rope_f64(x, pos: float, theta: float) -> np.ndarray:
    """Half-split RoPE of one vector, in double."""
    x = _req(np.asarray(x, dtype=np.float64), np.float64)
    y = np.empty_like(x)
    lib().oracle_rope_f64(_p(x), x.shape[-1], float(pos), float(theta), _p(y))
    return y


def rope_store_f32(x_bf16, pos: int, theta: float) -> np.ndarray:
    """Storage recipe of the appended key, before bf16/int8 rounding (fp32)."""
    x = _req(x_bf16, np.uint16)
    y = np.empty(x.shape[-1], dtype=np.float32)
    lib().oracle_rope_store_f32(_p(x), x.shape[-1], int(pos), float(theta), _p(y))
    return y


def quant_int8(x_f32):
    """Symmetric per-row int8 quantisation: (codes int8[d], scale float32)."""
    x = _req(x_f32, np.float32)
    codes = np.empty(x.shape[-1], dtype=np.int8)
    sc = np.zeros(1, dtype=np.float32)
    lib().oracle_quant_int8(_p(x), x.shape[-1], _p(codes), _p(sc))
    return codes, sc[0]


# ------------------------------------------------------------ whole steps --

def append(k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions,
           rope_theta, k_scales=None, v_scales=None) -> int:
    """Write the new k/v of every sequence into its slot (in place)."""
    kv_int8 = int(k_pages.dtype == np.int8)
    k_new = _req(k_new, np.uint16)
    v_new = _req(v_new, np.uint16)
    n_seq, n_kvh, d = k_new.shape
    num_pages, _, page, _ = k_pages.shape
    bt = _req(block_table, np.int32)
    return int(lib().oracle_append(
        _p(k_new), _p(v_new), _p(_req(k_pages, k_pages.dtype)), _p(_req(v_pages, v_pages.dtype)),
        _p(k_scales), _p(v_scales), _p(bt), _p(_req(seq_lens, np.int32)),
        _p(_req(positions, np.int32)), n_seq, n_kvh, d, page, float(rope_theta), kv_int8,
        bt.shape[1], num_pages))


def attend_paged(q, k_pages, v_pages, block_table, seq_lens, positions, rope_theta,
                 scale, k_scales=None, v_scales=None, seq_mask=None, n_threads=0,
                 out=None):
    """fp64 attention over the paged cache as it stands; returns (out, status)."""
    q = _req(q, np.uint16)
    n_seq, n_qh, d = q.shape
    num_pages, n_kvh, page, _ = k_pages.shape
    bt = _req(block_table, np.int32)
    if out is None:
        out = np.full((n_seq, n_qh, d), np.nan, dtype=np.float64)
    mask = None if seq_mask is None else _req(np.asarray(seq_mask, dtype=np.uint8), np.uint8)
    st = lib().oracle_attend_paged(
        _p(q), _p(k_pages), _p(v_pages), _p(k_scales), _p(v_scales), _p(bt),
        _p(_req(seq_lens, np.int32)), _p(_req(positions, np.int32)), _p(out),
        n_seq, n_qh, n_kvh, d, page, float(rope_theta), float(scale),
        int(k_pages.dtype == np.int8), bt.shape[1], num_pages, _p(mask), int(n_threads))
    return out, int(st)


def attend_contiguous(q, k_cache, v_cache, seq_lens, positions, n_kvh, rope_theta, scale):
    """fp64 attention over per-sequence contiguous caches [sum(L+1), n_kvh, d]."""
    q = _req(q, np.uint16)
    n_seq, n_qh, d = q.shape
    kc = _req(k_cache, np.float64)
    vc = _req(v_cache, np.float64)
    out = np.full((n_seq, n_qh, d), np.nan, dtype=np.float64)
    lib().oracle_attend_contiguous(
        _p(q), _p(kc), _p(vc), _p(_req(seq_lens, np.int32)), _p(_req(positions, np.int32)),
        _p(out), n_seq, n_qh, n_kvh, d, float(rope_theta), float(scale))
    return out


def decode(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions,
           rope_theta, scale, k_scales=None, v_scales=None, seq_mask=None, n_threads=0):
    """One decode step on host copies: append (in place), then attend.

    Returns (out float64 [n_seq, n_qh, d] with NaN rows for skipped sequences,
    status bits).
    """
    st = append(k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions,
                rope_theta, k_scales, v_scales)
    out, st2 = attend_paged(q, k_pages, v_pages, block_table, seq_lens, positions,
                            rope_theta, scale, k_scales, v_scales, seq_mask, n_threads)
    return out, st | st2
