"""Child process of tests/test_gpu_timeout.py (run as ``python -m tests.stall_child LIB``).

It loads only the test build of the library at LIB (compiled with
KVATTN_TEST_STALL), so that no other copy of the library shares the process.
With the request bit set in the workspace's status word, a decode call's warps
wait on a barrier nothing arrives at until their short limit runs out; the call
must report KVATTN_DEV_TIMEOUT.  The same process then re-initialises the
workspace and decodes again without the request: the context is intact and the
result matches the oracle.  Prints "stall-child ok" on success.
"""
import ctypes
import sys

import numpy as np
import torch

from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests.gpu_helpers import assert_close, out_f64, pool_bits, to_dev
from tests.helpers import host_inputs, oracle_decode

STALL_REQUEST = 0x80000000


def _args(lib_kv, wl, d, out, ws, stream):
    n_seq, n_qh, hd = d["q"].shape
    num_pages, n_kvh, page, _ = d["k_pages"].shape
    ptr = lambda t: None if t is None else t.data_ptr()
    return [d["q"].data_ptr(), d["k_new"].data_ptr(), d["v_new"].data_ptr(),
            d["k_pages"].data_ptr(), d["v_pages"].data_ptr(), d["block_table"].data_ptr(),
            d["seq_lens"].data_ptr(), d["positions"].data_ptr(), out.data_ptr(),
            n_seq, n_qh, n_kvh, hd, page, float(wl.rope_theta), float(wl.scale), lib_kv, stream,
            d["block_table"].shape[1], num_pages, ptr(d["k_scales"]), ptr(d["v_scales"]),
            ws.data_ptr(), ws.numel()]


def main(path):
    lib = K.bind(path)
    stream = torch.cuda.current_stream().cuda_stream
    for kv in ("bf16", "int8"):
        wl = W.make_workload("custom", seed=31, n_seq=5, n_qh=16, n_kvh=4, head_dim=128,
                             page_size=16, rope_theta=1e6, kv_dtype=kv,
                             lengths=[2000, 40, 777, 0, 3001], spare=0.1)
        h = host_inputs(wl)
        kv_code = K.KVATTN_KV_INT8 if kv == "int8" else K.KVATTN_KV_BF16
        size = lib.kvattn_workspace_size(wl.n_seq, wl.n_qh, wl.n_kvh, wl.head_dim)
        raw = torch.empty(size + 256, dtype=torch.uint8, device="cuda")
        off = (-raw.data_ptr()) % 256
        ws = raw[off:off + size]
        assert lib.kvattn_workspace_init(ws.data_ptr(), size, stream) == 0
        # the request bit in the status word (bit 31 of the first 4 bytes)
        ws[:4].view(torch.int32).fill_(-2 ** 31)
        d = to_dev(h)
        out = torch.zeros(d["q"].shape, dtype=torch.bfloat16, device="cuda")
        rc = lib.kvattn_decode(*_args(kv_code, wl, d, out, ws, stream))
        assert rc == K.KVATTN_OK, (rc, lib.kvattn_last_cuda_error())
        bits = ctypes.c_uint32(0)
        assert lib.kvattn_read_device_status(ws.data_ptr(), stream, ctypes.byref(bits)) == 0
        assert bits.value & K.KVATTN_DEV_TIMEOUT, hex(bits.value)
        # the context still runs work and reads back
        torch.cuda.synchronize()
        assert float(torch.ones(1024, device="cuda").sum()) == 1024.0
        assert torch.isfinite(out.float()).all()
        # re-initialised workspace, no request: the oracle's result
        assert lib.kvattn_workspace_init(ws.data_ptr(), size, stream) == 0
        d = to_dev(h)
        out = torch.full(d["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.kvattn_decode(*_args(kv_code, wl, d, out, ws, stream))
        assert rc == K.KVATTN_OK, (rc, lib.kvattn_last_cuda_error())
        assert lib.kvattn_read_device_status(ws.data_ptr(), stream, ctypes.byref(bits)) == 0
        assert bits.value == 0, hex(bits.value)
        ref, ost, kp, vp, ks, vs = oracle_decode(wl, h)
        assert ost == 0
        assert np.array_equal(pool_bits(d["k_pages"]), kp)
        assert np.array_equal(pool_bits(d["v_pages"]), vp)
        assert_close(out_f64(out), ref)
    print("stall-child ok")


if __name__ == "__main__":
    main(sys.argv[1])
