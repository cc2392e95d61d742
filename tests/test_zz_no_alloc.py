"""kvattn_decode_noalloc: the decode step for callers that cannot allocate.

Some callers of this library cannot hand it a device buffer: an engine that
reserved nearly all of HBM for its KV-page pool up front, or a plugin whose
host framework owns every device allocation and forbids cudaMalloc.  For them
the library keeps the step's scratch in a fixed array of its own.  These tests
call that entry point through the C ABI (ctypes, raw pointers) and compare it
with kvattn_decode given a normal workspace and with the oracle, on two calls
in a row, and check that a call's device status bits reach the caller and do
not leak into the next call.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from decode_phase_gqa_gb300 import build as B
from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests.gpu_helpers import MAX_ABS, MEAN_ABS, assert_close, out_f64, pool_bits, to_dev
from tests.helpers import host_inputs, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.load()


def _common_args(wl, d, out, stream):
    """The arguments kvattn_decode and kvattn_decode_noalloc share, in ABI order."""
    n_seq, n_qh, hd = d["q"].shape
    num_pages, n_kvh, page, _ = d["k_pages"].shape
    ptr = lambda t: None if t is None else t.data_ptr()
    return [d["q"].data_ptr(), d["k_new"].data_ptr(), d["v_new"].data_ptr(),
            d["k_pages"].data_ptr(), d["v_pages"].data_ptr(), d["block_table"].data_ptr(),
            d["seq_lens"].data_ptr(), d["positions"].data_ptr(), out.data_ptr(),
            n_seq, n_qh, n_kvh, hd, page, float(wl.rope_theta), float(wl.scale),
            K.KVATTN_KV_INT8 if wl.kv_dtype == "int8" else K.KVATTN_KV_BF16, stream,
            d["block_table"].shape[1], num_pages, ptr(d["k_scales"]), ptr(d["v_scales"])]


def _case(seed, kv, d):
    # long and short sequences: the long ones are cut across warps, so the
    # partial-state records of the scratch are exercised
    wl = W.make_workload("custom", seed=seed, n_seq=6, n_qh=16, n_kvh=4, head_dim=d,
                         page_size=16, rope_theta=1e6, kv_dtype=kv,
                         lengths=[3000, 17, 900, 0, 4095, 256], spare=0.1)
    return wl, host_inputs(wl)


def _assert_pools_equal(d, kp, vp, ks, vs):
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)
    if ks is not None:
        assert np.array_equal(d["k_scales"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(d["v_scales"].cpu().numpy().view(np.uint32), vs.view(np.uint32))


def test_noalloc_matches_workspace_entry_and_oracle_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream().cuda_stream
    for seed, kv, d in ((21, "bf16", 128), (22, "int8", 64)):
        wl, h = _case(seed, kv, d)
        ref, ost, kp, vp, ks, vs = oracle_decode(wl, h)
        assert ost == 0
        # the existing entry point, with a workspace from the caller
        d_ws = to_dev(h)
        out_ws = torch.empty(d_ws["q"].shape, dtype=torch.bfloat16, device="cuda")
        ws = K.alloc_workspace(wl.n_seq, wl.n_qh, wl.n_kvh, d)
        rc = lib.kvattn_decode(*_common_args(wl, d_ws, out_ws, stream), ws.data_ptr(), ws.numel())
        assert rc == K.KVATTN_OK
        assert K.kvattn_read_device_status(ws) == 0
        # the no-allocation entry point on a fresh copy of the same inputs
        d_na = to_dev(h)
        out_na = torch.full(d_na["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = lib.kvattn_decode_noalloc(*_common_args(wl, d_na, out_na, stream), status.data_ptr())
        assert rc == K.KVATTN_OK, K.kvattn_status_string(rc)
        torch.cuda.synchronize()
        assert status.item() == 0
        a, b = out_f64(out_na), out_f64(out_ws)
        err = np.abs(a - b)
        assert np.all(np.isfinite(a))
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
        assert np.array_equal(pool_bits(d_na["k_pages"]), pool_bits(d_ws["k_pages"]))
        assert np.array_equal(pool_bits(d_na["v_pages"]), pool_bits(d_ws["v_pages"]))
        # and both against the oracle: pools (and int8 scales) bit for bit,
        # outputs within the stated tolerance
        _assert_pools_equal(d_na, kp, vp, ks, vs)
        assert_close(a, ref)


def test_noalloc_status_word_is_reported_then_cleared(lib):
    # a block-table entry outside the pool makes the device skip that page and
    # set KVATTN_DEV_BAD_PAGE in the array's status word; the next call on the
    # same stream starts from a cleared word and reports 0
    stream = torch.cuda.current_stream().cuda_stream
    wl, h = _case(23, "bf16", 128)
    bad = dict(h)
    bad["block_table"] = h["block_table"].copy()
    bad["block_table"][0, 3] = -1
    d_bad = to_dev(bad)
    out_bad = torch.zeros(d_bad["q"].shape, dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.kvattn_decode_noalloc(*_common_args(wl, d_bad, out_bad, stream), status.data_ptr())
    assert rc == K.KVATTN_OK
    torch.cuda.synchronize()
    assert status.item() & K.KVATTN_DEV_BAD_PAGE
    # the clean call: status 0 and the oracle's result
    ref, ost, kp, vp, ks, vs = oracle_decode(wl, h)
    d_ok = to_dev(h)
    out_ok = torch.full(d_ok["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    status.fill_(-1)
    rc = lib.kvattn_decode_noalloc(*_common_args(wl, d_ok, out_ok, stream), status.data_ptr())
    assert rc == K.KVATTN_OK
    torch.cuda.synchronize()
    assert status.item() == 0
    _assert_pools_equal(d_ok, kp, vp, ks, vs)
    assert_close(out_f64(out_ok), ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # 8192 sequences x 64 query heads x d 128 need far more than the fixed array;
    # the call is refused before anything is queued (fake, never-used pointers)
    need = K.kvattn_workspace_size(8192, 64, 8, 128)
    assert need > K.KVATTN_NOALLOC_SCRATCH_BYTES
    fake = 0x10000
    args = [fake] * 9 + [8192, 64, 8, 128, 16, 1e4, 0.1, K.KVATTN_KV_BF16, None, 4, 8,
                         None, None]
    assert lib.kvattn_decode_noalloc(*args, None) == K.KVATTN_EUNSUPPORTED
