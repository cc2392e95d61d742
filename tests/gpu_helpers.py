"""GPU-side test plumbing: run the library on host inputs and compare with the oracle."""
import numpy as np
import torch

from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests import refmath as R
from tests.helpers import oracle_decode

# tolerance stated for the attention output (bf16 out, fp32 accumulate)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def to_dev(h, dev="cuda"):
    """Host numpy inputs (bf16 as uint16) -> device tensors of the right dtypes."""
    d = {}
    for k in ("q", "k_new", "v_new"):
        d[k] = torch.from_numpy(h[k].view(np.int16)).view(torch.bfloat16).to(dev)
    for k in ("k_pages", "v_pages"):
        a = h[k]
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
            else torch.from_numpy(a)
        d[k] = t.to(dev)
    for k in ("k_scales", "v_scales"):
        d[k] = None if h[k] is None else torch.from_numpy(h[k]).to(dev)
    for k in ("block_table", "seq_lens", "positions"):
        d[k] = torch.from_numpy(np.ascontiguousarray(h[k])).to(dev)
    return d


def pool_bits(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_gpu(wl: W.Workload, d, num_splits=0, ws=None, out=None):
    n_seq, n_qh, hd = d["q"].shape
    if ws is None:
        ws = K.alloc_workspace(n_seq, n_qh, wl.n_kvh, hd)
    if out is None:
        out = torch.full((n_seq, n_qh, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    K.kvattn_decode(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"], d["block_table"],
                    d["seq_lens"], d["positions"], out, rope_theta=wl.rope_theta, scale=wl.scale,
                    workspace=ws, k_scales=d["k_scales"], v_scales=d["v_scales"],
                    num_splits=num_splits)
    status = K.kvattn_read_device_status(ws)
    return out, status, ws


def out_f64(out):
    return out.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, rows=None):
    """max-abs <= 2e-2 and mean-abs <= 2e-3 over the compared rows."""
    g = gpu if rows is None else gpu[rows]
    r = ref if rows is None else ref[rows]
    err = np.abs(g - r)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3g}"
    assert err.mean() <= MEAN_ABS, f"mean abs err {err.mean():.3g}"
    return float(err.max()), float(err.mean())


def check_against_oracle(wl, h, num_splits=0, seq_mask=None):
    """Run GPU and oracle on the same inputs; check pools bit-exact and outputs in tolerance."""
    d = to_dev(h)
    out, status, _ = run_gpu(wl, d, num_splits)
    ref, ost, kp, vp, ks, vs = oracle_decode(wl, h, seq_mask=seq_mask)
    assert status == ost == 0
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)
    if ks is not None:
        assert np.array_equal(d["k_scales"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(d["v_scales"].cpu().numpy().view(np.uint32), vs.view(np.uint32))
    rows = None if seq_mask is None else np.flatnonzero(seq_mask)
    errs = assert_close(out_f64(out), ref, rows)
    return out, ref, errs
