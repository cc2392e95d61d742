"""Parity of the multi-layer entry (kvattn_decode_layers) with the oracle (needs a GB300).

Several layer caches that share the block table, lengths and positions are
decoded in one call; every layer must come out as the oracle's decode step of
that layer alone: its K/V pool (and int8 scales) bit for bit after the
append, its output within max-abs 2e-2 / mean-abs 2e-3.  One layer through the
multi-layer entry is the single-layer call bit for bit.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests.gpu_helpers import assert_close, out_f64, pool_bits, run_gpu, to_dev
from tests.helpers import host_inputs, oracle_decode

pytestmark = pytest.mark.gpu

STACKED = ("q", "k_new", "v_new", "k_pages", "v_pages", "k_scales", "v_scales")


def stack_layers(wl, n_layers, device="cuda", tensors=None):
    """Layer-major device inputs of n_layers layer caches, and each layer's host copy."""
    layers = tensors if tensors is not None else [
        W.make_tensors(wl, layer=l, device="cpu") for l in range(n_layers)]
    hosts = [host_inputs(wl, tensors=t) for t in layers]
    d = {}
    for k in STACKED:
        d[k] = None if layers[0][k] is None else torch.stack(
            [t[k].to(device) for t in layers]).contiguous()
    for k in ("block_table", "seq_lens", "positions"):
        d[k] = torch.from_numpy(np.ascontiguousarray(hosts[0][k])).to(device)
    return d, hosts


def run_layers(wl, d, layer_rope=None):
    L, B, Hq, hd = d["q"].shape
    ws = K.alloc_workspace(B, Hq, wl.n_kvh, hd, n_layers=L)
    out = torch.full((L, B, Hq, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    K.kvattn_decode_layers(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                           d["block_table"], d["seq_lens"], d["positions"], out,
                           rope_theta=wl.rope_theta, scale=wl.scale, workspace=ws,
                           k_scales=d["k_scales"], v_scales=d["v_scales"],
                           layer_rope=layer_rope)
    return out, K.kvattn_read_device_status(ws)


def check_layers(wl, d, hosts, out, seq_mask=None, layer_rope=None):
    rows = None if seq_mask is None else np.flatnonzero(seq_mask)
    for l, h in enumerate(hosts):
        # a layer without RoPE is the oracle's step with RoPE off (theta <= 0)
        wl_l = wl if layer_rope is None or layer_rope[l] else replace(wl, rope_theta=0.0)
        ref, ost, kp, vp, ks, vs = oracle_decode(wl_l, h, seq_mask=seq_mask)
        assert ost == 0
        assert np.array_equal(pool_bits(d["k_pages"][l]), kp), f"layer {l} K pool"
        assert np.array_equal(pool_bits(d["v_pages"][l]), vp), f"layer {l} V pool"
        if ks is not None:
            assert np.array_equal(d["k_scales"][l].cpu().numpy().view(np.uint32), ks.view(np.uint32))
            assert np.array_equal(d["v_scales"][l].cpu().numpy().view(np.uint32), vs.view(np.uint32))
        got = out_f64(out[l])
        assert np.all(np.isfinite(got if rows is None else got[rows])), f"layer {l} rows unwritten"
        assert_close(got, ref, rows)


def custom(n_qh, n_kvh, lens, d=128, kv="bf16", seed=0, page=16):
    return W.make_workload("custom", seed=seed, n_seq=len(lens), n_qh=n_qh, n_kvh=n_kvh,
                           head_dim=d, page_size=page, rope_theta=1e6, kv_dtype=kv,
                           lengths=list(lens), spare=0.1)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_layers", [2, 5])
def test_every_layer_matches_the_oracle(kv, d, n_layers):
    # ragged tails, a new token alone in a new page, an empty cache, several tiles
    wl = custom(16, 4, [0, 15, 16, 17, 100, 257, 511], d=d, kv=kv, seed=n_layers + d)
    dd, hosts = stack_layers(wl, n_layers)
    out, status = run_layers(wl, dd)
    assert status == 0
    check_layers(wl, dd, hosts, out)


@pytest.mark.parametrize("n_qh,n_kvh,lens", [
    (4, 1, [256]),                      # the tiny shape: shares spread, helper warps
    (32, 8, [3000, 1, 40]),             # streams cut across warps and across layers
    (8, 8, [5] * 40),                   # many short sequences, no GQA sharing
])
def test_layer_boundaries_inside_shares(n_qh, n_kvh, lens):
    wl = custom(n_qh, n_kvh, lens, d=64, seed=len(lens))
    dd, hosts = stack_layers(wl, 3)
    out, status = run_layers(wl, dd)
    assert status == 0
    check_layers(wl, dd, hosts, out)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_one_layer_is_the_single_layer_call(kv):
    wl = custom(32, 8, [700, 3, 2048, 129], d=128, kv=kv, seed=11)
    h = host_inputs(wl)
    d1 = to_dev(h)
    single, st1, _ = run_gpu(wl, d1)
    dd, _ = stack_layers(wl, 1)
    layered, st2 = run_layers(wl, dd)
    assert st1 == st2 == 0
    assert torch.equal(single.view(torch.int16), layered[0].view(torch.int16))
    assert np.array_equal(pool_bits(d1["k_pages"]), pool_bits(dd["k_pages"][0]))
    assert np.array_equal(pool_bits(d1["v_pages"]), pool_bits(dd["v_pages"][0]))


def test_qwen3_shaped_layers_at_full_size():
    """Four of the Qwen3-8B-shaped step's layer caches (batch 64, 32/8 heads,
    d 128, lengths log-uniform in [128, 8192]) in one call with the default
    split, as the benchmark times the step: every pool bit for bit, the
    output on the longest, shortest and a seeded few sequences."""
    wl = W.make_workload("qwen3", seed=0)
    dev = torch.device("cuda")
    layers = [W.make_tensors(wl, layer=l, device=dev) for l in range(4)]
    dd, hosts = stack_layers(wl, 4, tensors=layers)
    del layers
    out, status = run_layers(wl, dd)
    assert status == 0
    L = wl.seq_lens
    pick = {int(np.argmax(L)), int(np.argmin(L))}
    pick.update(int(b) for b in np.random.default_rng(5).choice(wl.n_seq, 4, replace=False))
    mask = np.zeros(wl.n_seq, np.uint8)
    mask[sorted(pick)] = 1
    check_layers(wl, dd, hosts, out, seq_mask=mask)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_rope_and_nope_layers(kv):
    """SmolLM3's pattern: RoPE on three layers, none on the fourth (its query
    and new key are not rotated), in one call."""
    pattern = [True, True, True, False, True, True, True, False]
    wl = custom(16, 4, [3, 64, 200, 1000], d=128, kv=kv, seed=21)
    dd, hosts = stack_layers(wl, len(pattern))
    out, status = run_layers(wl, dd, layer_rope=pattern)
    assert status == 0
    check_layers(wl, dd, hosts, out, layer_rope=pattern)


def test_bad_length_and_bad_page_in_every_layer():
    """The layers share the lengths and the block table, so a bad length or
    page is bad in every layer: each layer skips the same sequence and leaves
    out the same page's tokens as its own decode step would, and the status
    word reports both."""
    wl = custom(8, 2, [50, 60, 70, 90], d=64, seed=8)
    layers = [W.make_tensors(wl, layer=l, device="cpu") for l in range(3)]
    bt = wl.block_table.copy()
    bt[2, 1] = 10 ** 6      # out of range: tokens 16-31 of sequence 2 left out
    bt[3, 0] = -7           # negative: tokens 0-15 of sequence 3 left out
    wl = replace(wl, block_table=bt, seq_lens=np.array([50, -3, 70, 90], np.int32))
    dd, hosts = stack_layers(wl, 3, tensors=layers)
    out, status = run_layers(wl, dd)
    assert status & K.KVATTN_DEV_BAD_LEN and status & K.KVATTN_DEV_BAD_PAGE
    for l, h in enumerate(hosts):
        ref, ost, kp, vp, _, _ = oracle_decode(wl, h)
        assert ost & 1 and ost & 2
        o = out_f64(out[l])
        assert np.all(np.isnan(o[1])), "the skipped sequence's rows were written"
        assert_close(o, ref, rows=[0, 2, 3])
        assert np.array_equal(pool_bits(dd["k_pages"][l]), kp)
        assert np.array_equal(pool_bits(dd["v_pages"][l]), vp)


def test_layers_captured_in_cuda_graph():
    """One layered call captured in a CUDA graph and replayed twice (the append
    rewrites the same slot with the same row, so a replay repeats the step)."""
    wl = custom(32, 8, [1000, 20, 333, 4096], d=128, seed=13)
    dd, hosts = stack_layers(wl, 4)
    L, B, Hq, hd = dd["q"].shape
    ws = K.alloc_workspace(B, Hq, wl.n_kvh, hd, n_layers=L)
    out = torch.empty((L, B, Hq, hd), dtype=torch.bfloat16, device="cuda")

    def call(stream):
        K.kvattn_decode_layers(dd["q"], dd["k_new"], dd["v_new"], dd["k_pages"], dd["v_pages"],
                               dd["block_table"], dd["seq_lens"], dd["positions"], out,
                               rope_theta=wl.rope_theta, scale=wl.scale, workspace=ws,
                               stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(s)            # the library's per-device set-up, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert K.kvattn_read_device_status(ws) == 0
        check_layers(wl, dd, hosts, out)
