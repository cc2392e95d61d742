"""Host-side checks of the C ABI: exports, workspace sizing and fail-closed validation.

Runs without a GPU: every call below is rejected by the host checks (or has
nothing to do) before the library touches the CUDA runtime.
"""
import ctypes
import os
import re
import subprocess

import pytest

from decode_phase_gqa_gb300 import build as B
from decode_phase_gqa_gb300 import kvattn as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvattn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvattn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted([
        "kvattn_decode", "kvattn_decode_layers", "kvattn_decode_noalloc",
        "kvattn_decode_splits", "kvattn_last_cuda_error", "kvattn_prefill",
        "kvattn_prefill_workspace_size",
        "kvattn_read_device_status",
        "kvattn_status_string", "kvattn_version", "kvattn_workspace_init",
        "kvattn_workspace_size", "kvattn_workspace_size_layers"])


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvattn_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c():
    src = f'#include "{HEADER}"\nint main(void){{return KVATTN_OK;}}\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-x", "c", "-", "-fsyntax-only"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    for code in range(5):
        assert K.kvattn_status_string(code)
    assert K.kvattn_status_string(99) == "unknown status"
    assert K.kvattn_version() >= 101
    assert K.kvattn_last_cuda_error() == 0   # no call has failed in CUDA here


def test_workspace_size(lib):
    s = K.kvattn_workspace_size
    assert s(0, 4, 1, 64) > 0
    assert s(1, 4, 1, 64) % 256 == 0
    assert s(64, 32, 8, 128) > s(8, 32, 8, 128) > 0
    # a partial-state record (acc, m, l of a 4-head group) for every stream and
    # split
    assert s(64, 32, 8, 128) >= (64 * 8 + K.KVATTN_MAX_SPLITS) * 4 * 130 * 4
    for bad in ((-1, 4, 1, 64), (1, 0, 1, 64), (1, 4, 3, 64), (1, 4, 1, 96),
                (K.KVATTN_MAX_SEQS + 1, 4, 1, 64)):
        assert s(*bad) == 0, bad


# a plausible argument list with fake (never dereferenced) aligned pointers
FAKE = 0x10000


def args(**kw):
    a = dict(q=FAKE, k_new=FAKE, v_new=FAKE, k_pages=FAKE, v_pages=FAKE, block_table=FAKE,
             seq_lens=FAKE, positions=FAKE, out=FAKE, n_seq=2, n_qh=8, n_kvh=2, head_dim=64,
             page_size=16, rope_theta=1e4, scale=0.125, kv_dtype=0, stream=None,
             max_pages_per_seq=4, num_pages=8, k_scales=None, v_scales=None,
             workspace=FAKE, workspace_bytes=1 << 30, num_splits=0)
    a.update(kw)
    return a


def call(lib, **kw):
    a = args(**kw)
    return lib.kvattn_decode_splits(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(n_qh=6, n_kvh=4), K.KVATTN_EINVAL),
    (dict(n_kvh=0), K.KVATTN_EINVAL),
    (dict(n_seq=-1), K.KVATTN_EINVAL),
    (dict(max_pages_per_seq=0), K.KVATTN_EINVAL),
    (dict(num_pages=0), K.KVATTN_EINVAL),
    (dict(num_splits=-1), K.KVATTN_EINVAL),
    (dict(num_splits=K.KVATTN_MAX_SPLITS + 1), K.KVATTN_EINVAL),
    (dict(scale=float("nan")), K.KVATTN_EINVAL),
    (dict(scale=float("inf")), K.KVATTN_EINVAL),
    (dict(rope_theta=float("nan")), K.KVATTN_EINVAL),
    (dict(head_dim=96), K.KVATTN_EUNSUPPORTED),
    (dict(head_dim=256), K.KVATTN_EUNSUPPORTED),
    (dict(page_size=8), K.KVATTN_EUNSUPPORTED),
    (dict(page_size=48), K.KVATTN_EUNSUPPORTED),
    (dict(page_size=512), K.KVATTN_EUNSUPPORTED),
    (dict(kv_dtype=2), K.KVATTN_EUNSUPPORTED),
    (dict(n_seq=K.KVATTN_MAX_SEQS + 1), K.KVATTN_EUNSUPPORTED),
    (dict(max_pages_per_seq=1 << 27, page_size=64), K.KVATTN_EUNSUPPORTED),
    # 4096 sequences x 64 KV heads x 131072 units: the unit count passes 2^31
    (dict(n_seq=4096, n_qh=64, n_kvh=64, max_pages_per_seq=8192, page_size=256),
     K.KVATTN_EUNSUPPORTED),
    (dict(q=None), K.KVATTN_EINVAL),
    (dict(out=None), K.KVATTN_EINVAL),
    (dict(block_table=None), K.KVATTN_EINVAL),
    (dict(k_pages=FAKE + 8), K.KVATTN_EINVAL),
    (dict(v_pages=FAKE + 4), K.KVATTN_EINVAL),
    (dict(q=FAKE + 1), K.KVATTN_EINVAL),
    (dict(seq_lens=FAKE + 2), K.KVATTN_EINVAL),
    (dict(kv_dtype=1), K.KVATTN_EINVAL),                     # int8 without scales
    (dict(kv_dtype=1, k_scales=FAKE, v_scales=FAKE + 4), K.KVATTN_EINVAL),
    (dict(workspace=None), K.KVATTN_EWORKSPACE),
    (dict(workspace=FAKE + 128), K.KVATTN_EWORKSPACE),
    (dict(workspace_bytes=1024), K.KVATTN_EWORKSPACE),
])
def test_invalid_arguments_fail_closed(lib, kw, code):
    assert call(lib, **kw) == code


def test_empty_batch_is_a_no_op(lib):
    assert call(lib, n_seq=0) == K.KVATTN_OK


def test_plain_decode_entry_has_the_same_checks(lib):
    a = args(head_dim=80)
    del a["num_splits"]
    assert lib.kvattn_decode(*a.values()) == K.KVATTN_EUNSUPPORTED


def test_workspace_init_and_status_checks(lib):
    assert lib.kvattn_workspace_init(None, 1024, None) == K.KVATTN_EWORKSPACE
    assert lib.kvattn_workspace_init(FAKE + 16, 1024, None) == K.KVATTN_EWORKSPACE
    assert lib.kvattn_workspace_init(FAKE, 128, None) == K.KVATTN_EWORKSPACE
    assert lib.kvattn_read_device_status(FAKE, None, None) == K.KVATTN_EINVAL
    bits = ctypes.c_uint32()
    assert lib.kvattn_read_device_status(None, None, ctypes.byref(bits)) == K.KVATTN_EWORKSPACE


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.reload(K)
    try:
        mod._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            mod.load(str(tmp_path / "nope.so"))
    finally:
        importlib.reload(K)


def test_workspace_size_layers(lib):
    s1, sl = K.kvattn_workspace_size, K.kvattn_workspace_size_layers
    assert sl(1, 64, 32, 8, 128) == s1(64, 32, 8, 128)
    # records for every layer's streams: as many as one layer of 36 x 64 sequences
    assert sl(36, 64, 32, 8, 128) == s1(36 * 64, 32, 8, 128) > s1(64, 32, 8, 128)
    for bad in ((0, 8, 4, 1, 64), (-1, 8, 4, 1, 64), (K.KVATTN_MAX_LAYERS + 1, 8, 4, 1, 64),
                (2, 8, 4, 3, 64), (2, K.KVATTN_MAX_SEQS + 1, 4, 1, 64)):
        assert sl(*bad) == 0, bad


def call_layers(lib, n_layers, **kw):
    a = args(**kw)
    del a["num_splits"]
    return lib.kvattn_decode_layers(n_layers, *a.values(), None)


@pytest.mark.parametrize("n_layers,kw,code", [
    (0, {}, K.KVATTN_EINVAL),
    (-3, {}, K.KVATTN_EINVAL),
    (K.KVATTN_MAX_LAYERS + 1, {}, K.KVATTN_EUNSUPPORTED),
    # every layer's pool rows must stay below 2^31: 1024 x 2^17 pages x 16 x 16
    (1024, dict(num_pages=1 << 17, n_kvh=16, n_qh=16), K.KVATTN_EUNSUPPORTED),
    # one layer's workspace is too small for 36 layers' partial states
    (36, dict(workspace_bytes=None), K.KVATTN_EWORKSPACE),
    (2, dict(head_dim=96), K.KVATTN_EUNSUPPORTED),
    (2, dict(q=None), K.KVATTN_EINVAL),
    (2, dict(n_seq=0), K.KVATTN_OK),
])
def test_layers_entry_fails_closed(lib, n_layers, kw, code):
    if kw.get("workspace_bytes", 0) is None:
        a = args()
        kw = dict(workspace_bytes=K.kvattn_workspace_size(a["n_seq"], a["n_qh"], a["n_kvh"],
                                                          a["head_dim"]))
    assert call_layers(lib, n_layers, **kw) == code


def prefill_args(**kw):
    a = dict(q=FAKE, k_new=FAKE, v_new=FAKE, k_pages=FAKE, v_pages=FAKE, block_table=FAKE,
             seq_starts=FAKE, ctx_lens=FAKE, out=FAKE, n_seq=2, n_tok=40, n_qh=8, n_kvh=2,
             head_dim=64, page_size=16, rope_theta=1e4, scale=0.125, kv_dtype=0, stream=None,
             max_pages_per_seq=4, num_pages=8, k_scales=None, v_scales=None, max_new_tokens=32,
             dev_status=None, workspace=None, workspace_bytes=0)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(n_seq=-1), K.KVATTN_EINVAL),
    (dict(n_tok=-1), K.KVATTN_EINVAL),
    (dict(n_qh=6, n_kvh=4), K.KVATTN_EINVAL),
    (dict(n_qh=6, n_kvh=2), K.KVATTN_EUNSUPPORTED),     # groups of 3 heads
    (dict(head_dim=96), K.KVATTN_EUNSUPPORTED),
    (dict(page_size=8), K.KVATTN_EUNSUPPORTED),
    (dict(max_new_tokens=-1), K.KVATTN_EINVAL),
    (dict(scale=float("nan")), K.KVATTN_EINVAL),
    (dict(q=None), K.KVATTN_EINVAL),
    (dict(seq_starts=None), K.KVATTN_EINVAL),
    (dict(k_new=FAKE + 8), K.KVATTN_EINVAL),
    (dict(dev_status=FAKE + 2), K.KVATTN_EINVAL),
    (dict(workspace=FAKE + 8, workspace_bytes=1 << 20), K.KVATTN_EINVAL),
    (dict(kv_dtype=2), K.KVATTN_EUNSUPPORTED),
    (dict(kv_dtype=1), K.KVATTN_EINVAL),                      # int8 without scales
    (dict(kv_dtype=1, k_scales=FAKE, v_scales=FAKE + 4), K.KVATTN_EINVAL),
    (dict(n_tok=0), K.KVATTN_OK),
    (dict(n_seq=0), K.KVATTN_OK),
])
def test_prefill_entry_fails_closed(lib, kw, code):
    assert lib.kvattn_prefill(*prefill_args(**kw).values()) == code
