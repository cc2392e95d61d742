"""Parity of the CUDA decode path with the CPU oracle (needs a GB300).

Every case runs the library through the C ABI and the oracle on the same
seeded inputs, then checks: the whole K/V pool (and int8 scales) bit for bit
after the append, the attention output within max-abs 2e-2 / mean-abs 2e-3,
and a clean device status word.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests import refmath as R
from tests.gpu_helpers import (assert_close, check_against_oracle, out_f64, pool_bits,
                               run_gpu, to_dev)
from tests.helpers import host_inputs, oracle_decode

pytestmark = pytest.mark.gpu


def custom(n_qh, n_kvh, lens, d=128, page=16, kv="bf16", seed=0, theta=1e4, spare=0.1,
           max_len=None):
    wl = W.make_workload("custom", seed=seed, n_seq=len(lens), n_qh=n_qh, n_kvh=n_kvh,
                         head_dim=d, page_size=page, rope_theta=theta, kv_dtype=kv,
                         lengths=list(lens), spare=spare, max_len=max_len)
    return wl, host_inputs(wl)


def test_tiny_config():
    wl = W.make_workload("tiny", seed=0)
    check_against_oracle(wl, host_inputs(wl))


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_qh,n_kvh", [(4, 1), (16, 4), (8, 8), (4, 2), (12, 4), (24, 2), (6, 2)])
def test_head_layouts(kv, d, n_qh, n_kvh):
    # several 16-token tiles, ragged tails, the new token alone in a new page
    lens = [0, 15, 16, 17, 100, 257, 511]
    wl, h = custom(n_qh, n_kvh, lens, d=d, kv=kv, seed=n_qh * 7 + n_kvh)
    check_against_oracle(wl, h)


@pytest.mark.parametrize("page", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_page_sizes(page, kv):
    lens = [1, page - 1, page, 3 * page + 5, 700]
    wl, h = custom(8, 2, lens, d=64, page=page, kv=kv, seed=page)
    check_against_oracle(wl, h)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 5, 17, 64, 333, 4096])
def test_split_counts_agree(num_splits):
    wl, h = custom(16, 4, [3000, 1, 40, 777, 2048], d=128, seed=3)
    out, ref, _ = check_against_oracle(wl, h, num_splits=num_splits)
    # and against the single-share result: fp32 reordering only (1 bf16 ulp)
    d = to_dev(host_inputs(wl))
    one, _, _ = run_gpu(wl, d, num_splits=1)
    a, b = out_f64(out), out_f64(one)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6)


def test_results_are_deterministic():
    wl, h = custom(32, 8, [5000, 300, 12, 4096], d=128, seed=11)
    outs = []
    for _ in range(3):
        d = to_dev(h)
        o, st, _ = run_gpu(wl, d)
        assert st == 0
        outs.append(pool_bits(o))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_page_permutation_is_bit_identical():
    wl, h = custom(8, 2, [200, 64, 1000], d=128, seed=5, spare=0.0)
    d1 = to_dev(h)
    o1, _, _ = run_gpu(wl, d1)
    perm = np.random.default_rng(1).permutation(wl.num_pages).astype(np.int32)
    h2 = dict(h)
    for k in ("k_pages", "v_pages"):
        h2[k] = np.empty_like(h[k])
        h2[k][perm] = h[k]
    h2["block_table"] = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)],
                                 -1).astype(np.int32)
    o2, _, _ = run_gpu(wl, to_dev(h2))
    assert np.array_equal(pool_bits(o1), pool_bits(o2))


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_single_token_returns_value(kv):
    wl, h = custom(8, 2, [0, 0, 0], d=128, kv=kv, seed=2)
    d = to_dev(h)
    out, st, _ = run_gpu(wl, d)
    assert st == 0
    ref, _, kp, vp, ks, vs = oracle_decode(wl, h)
    if kv == "bf16":
        # one weight of exactly 1: the stored value comes back bit for bit
        want = np.repeat(h["v_new"], 4, axis=1)
        assert np.array_equal(pool_bits(out), want)
    else:
        assert_close(out_f64(out), ref)


def test_identical_keys_give_mean_of_values():
    wl, h = custom(4, 1, [300], d=64, seed=4, theta=0.0)
    # every cached key equals the new key (NoPE, so it is stored unchanged)
    P = wl.page_size
    for t in range(300):
        h["k_pages"][wl.block_table[0, t // P], :, t % P] = h["k_new"][0]
    out, st, _ = run_gpu(wl, to_dev(h))
    vr = R.gather_rows(h["v_pages"], None, wl.block_table, 0, 299, P, False)[:, 0]
    vmean = (vr.sum(axis=0) + R.bf16_bits_to_f64(h["v_new"][0, 0])) / 301
    assert np.max(np.abs(out_f64(out)[0] - vmean)) < 2e-3


def test_new_token_dominates_when_aligned():
    wl, h = custom(1, 1, [900], d=128, seed=6, theta=0.0)
    h["k_new"][0, 0] = h["q"][0, 0]
    wl.scale = 30.0
    out, st, _ = run_gpu(wl, to_dev(h))
    assert np.max(np.abs(out_f64(out)[0, 0] - R.bf16_bits_to_f64(h["v_new"][0, 0]))) < 1e-2


@pytest.mark.parametrize("num_splits", [0, 7])
@pytest.mark.parametrize("factor", [1e-7, 1e5])
def test_int8_value_scales_far_from_one(factor, num_splits):
    """Every value row, cached and the new token's, times 1e-7 (dequantised
    values below f16's smallest subnormal) or 1e5 (past f16's largest finite
    value): the outputs move with them.  Compared with the oracle relative to
    each output row's size, whole streams and streams cut into parts."""
    wl, h = custom(8, 2, [0, 15, 300, 2000], d=128, kv="int8", seed=71)
    h["v_scales"] = h["v_scales"] * np.float32(factor)
    h["v_new"] = R.f32_to_bf16_bits(R.bf16_bits_to_f64(h["v_new"]) * factor)
    out, st, _ = run_gpu(wl, to_dev(h), num_splits=num_splits)
    ref, ost, *_ = oracle_decode(wl, h)
    assert st == ost == 0
    got = out_f64(out)
    assert np.all(np.isfinite(got))
    size = np.abs(ref).max(axis=-1, keepdims=True)
    assert size.min() > 0
    assert np.all(np.abs(got - ref) <= 2e-2 * size)


@pytest.mark.parametrize("num_splits", [0, 7])
def test_int8_key_scales_far_from_one(num_splits):
    """Cached key rows with 1e-7 times their scales (scores near zero), and one
    row per sequence with 3e4 times its scale (dequantised values past f16's
    range, scores near 3e5) that the query is aligned with (NoPE): that row
    takes the whole softmax."""
    wl, h = custom(8, 2, [40, 300, 2000], d=128, kv="int8", seed=73, theta=0.0)
    P = wl.page_size
    ks = h["k_scales"]
    for b, L in enumerate(wl.seq_lens):
        big = int(L) // 3
        for t in range(0, int(L), 5):
            if t != big:
                ks[wl.block_table[b, t // P], :, t % P] *= np.float32(1e-7)
        pg, off = wl.block_table[b, big // P], big % P
        for hq in range(8):   # aligned with the row before it grows
            h["q"][b, hq] = R.f32_to_bf16_bits(
                h["k_pages"][pg, hq // 4, off].astype(np.float64) * ks[pg, hq // 4, off])
        ks[pg, :, off] *= np.float32(3e4)
    check_against_oracle(wl, h, num_splits=num_splits)


def test_relative_position_invariance_through_appends():
    # fill two caches token by token through the library, positions t and t + s,
    # then decode at m and m + s: scores depend on m - t only
    d, n = 64, 40
    rng = np.random.default_rng(0)
    raw_k = R.f32_to_bf16_bits(rng.standard_normal((n + 1, 1, d)))
    raw_v = R.f32_to_bf16_bits(rng.standard_normal((n + 1, 1, d)))
    q = R.f32_to_bf16_bits(rng.standard_normal((1, 4, d)))
    outs = []
    for shift in (0, 1000):
        wl, h = custom(4, 1, [n], d=d, seed=0, theta=1e4)
        dev = to_dev(h)
        ws = K.alloc_workspace(1, 4, 1, d)
        out = torch.empty((1, 4, d), dtype=torch.bfloat16, device="cuda")
        for t in range(n + 1):
            dev["seq_lens"].fill_(t)
            dev["positions"].fill_(t + shift)
            dev["k_new"].copy_(torch.from_numpy(raw_k[t:t + 1].view(np.int16)).view(torch.bfloat16))
            dev["v_new"].copy_(torch.from_numpy(raw_v[t:t + 1].view(np.int16)).view(torch.bfloat16))
            if t == n:
                dev["q"].copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16))
            K.kvattn_decode(dev["q"], dev["k_new"], dev["v_new"], dev["k_pages"], dev["v_pages"],
                            dev["block_table"], dev["seq_lens"], dev["positions"], out,
                            rope_theta=1e4, scale=wl.scale, workspace=ws)
        assert K.kvattn_read_device_status(ws) == 0
        outs.append(out_f64(out))
    assert np.max(np.abs(outs[0] - outs[1])) < 2e-2


def test_bad_length_and_bad_page_are_skipped_and_reported():
    wl, h = custom(8, 2, [50, 60, 70], d=64, seed=8)
    h["seq_lens"] = np.array([50, -3, 70], np.int32)
    d = to_dev(h)
    out, st, _ = run_gpu(wl, d)
    assert st & K.KVATTN_DEV_BAD_LEN
    o = out_f64(out)
    assert np.all(np.isnan(o[1])) and np.all(np.isfinite(o[[0, 2]]))
    ref, ost, *_ = oracle_decode(wl, h)
    assert ost & 1
    assert_close(o, ref, rows=[0, 2])
    # an out-of-range page: its tokens are left out, everything else is exact
    wl2, h2 = custom(8, 2, [50, 60, 70], d=64, seed=8)
    bt = h2["block_table"].copy()
    bt[1, 1] = 10 ** 6
    bt[2, 0] = -7
    h2["block_table"] = bt
    wl2.block_table = bt
    d2 = to_dev(h2)
    out2, st2, _ = run_gpu(wl2, d2)
    assert st2 & K.KVATTN_DEV_BAD_PAGE
    ref2, ost2, kp, vp, _, _ = oracle_decode(wl2, h2)
    assert ost2 & 2
    assert_close(out_f64(out2), ref2)
    assert np.array_equal(pool_bits(d2["k_pages"]), kp)


def test_length_at_table_capacity():
    # L + 1 == max_pages * page: the last slot of the last page
    wl, h = custom(8, 2, [127, 63], d=128, seed=9, max_len=127)
    assert wl.max_pages_per_seq == 8
    check_against_oracle(wl, h)


def test_many_short_sequences():
    lens = list(np.random.default_rng(2).integers(0, 40, size=300))
    wl, h = custom(8, 2, lens, d=64, seed=12)
    check_against_oracle(wl, h)


def test_empty_batch_is_a_no_op():
    ws = K.alloc_workspace(0, 8, 2, 64)
    z = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device="cuda")
    K.kvattn_decode(z(0, 8, 64), z(0, 2, 64), z(0, 2, 64), z(4, 2, 16, 64), z(4, 2, 16, 64),
                    z(0, 4, dt=torch.int32), z(0, dt=torch.int32), z(0, dt=torch.int32),
                    z(0, 8, 64), rope_theta=1e4, scale=0.125, workspace=ws)
    assert K.kvattn_read_device_status(ws) == 0


def test_captured_in_cuda_graph():
    wl, h = custom(16, 4, [1000, 20, 333], d=128, seed=13)
    d = to_dev(h)
    ws = K.alloc_workspace(3, 16, 4, 128)
    out = torch.empty((3, 16, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.kvattn_decode(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                        d["block_table"], d["seq_lens"], d["positions"], out,
                        rope_theta=wl.rope_theta, scale=wl.scale, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        K.kvattn_decode(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                        d["block_table"], d["seq_lens"], d["positions"], out,
                        rope_theta=wl.rope_theta, scale=wl.scale, workspace=ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref, *_ = oracle_decode(wl, h)
    assert_close(out_f64(out), ref)


@pytest.mark.parametrize("kv,d,theta", [("bf16", 128, 1e4), ("int8", 64, 5e5), ("bf16", 64, 1e6)])
def test_appended_keys_over_many_positions(kv, d, theta):
    # 384 short sequences whose RoPE positions spread over [0, 2^21): the stored
    # key's cos/sin take the float-float path below angles of 2^18 and the
    # double fallback above; every appended slot must equal the oracle's
    # recipe bit for bit, and the outputs stay within tolerance
    n = 384
    lens = list(np.random.default_rng(d).integers(0, 20, size=n))
    wl, h = custom(8, 2, lens, d=d, kv=kv, seed=d + 3, theta=theta)
    pos = np.random.default_rng(7).integers(0, 1 << 21, size=n).astype(np.int32)
    pos[:8] = [0, 1, 2, 3, 255, 256, 1 << 17, (1 << 18) + 1]
    wl.positions = pos
    h["positions"] = pos.copy()
    check_against_oracle(wl, h)


@pytest.mark.parametrize("theta", [1e4, 1e6])
def test_appended_keys_at_many_fast_path_positions(theta):
    # 2048 sequences whose positions spread over [0, 2^18), where the stored
    # key's angle is formed from the integer product pos * inv_freq and the
    # float-float reduction: 131072 angles, every appended slot bit for bit
    n = 2048
    lens = list(np.random.default_rng(11).integers(0, 4, size=n))
    wl, h = custom(4, 1, lens, d=128, seed=31, theta=theta)
    pos = np.random.default_rng(13).integers(0, 1 << 18, size=n).astype(np.int32)
    pos[:6] = [1, 2, 3, (1 << 18) - 1, 12345, 65536]
    wl.positions = pos
    h["positions"] = pos.copy()
    check_against_oracle(wl, h)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_back_to_back_steps_see_the_previous_append(kv):
    # two decode steps queued on one stream with no other kernel between them:
    # the second step attends over the token the first one appended (lengths
    # at and across unit and page boundaries)
    lens = [14, 15, 16, 31, 100, 255, 0, 47]
    wl, h1 = custom(8, 2, lens, d=128, kv=kv, seed=21, spare=0.5, max_len=300)
    bt = h1["block_table"]
    used = set(int(x) for x in bt.ravel() if x >= 0)
    free = [p for p in range(wl.num_pages) if p not in used]
    for b, L in enumerate(lens):  # the second step's slot L + 1 may start a new page
        n = L // wl.page_size + 1
        if (L + 1) // wl.page_size + 1 > n:
            bt[b, n] = free.pop()
    rng = np.random.default_rng(5)
    h2 = dict(h1)
    for k in ("q", "k_new", "v_new"):
        h2[k] = R.f32_to_bf16_bits(rng.standard_normal(h1[k].shape))
    h2["seq_lens"] = h1["seq_lens"] + 1
    h2["positions"] = h1["positions"] + 1

    d1 = to_dev(h1)
    d2 = dict(d1)
    for k in ("q", "k_new", "v_new", "seq_lens", "positions"):
        d2[k] = to_dev(h2)[k]
    ws = K.alloc_workspace(len(lens), 8, 2, 128)
    outs = []
    for d in (d1, d2):
        out = torch.full((len(lens), 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        K.kvattn_decode(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                        d["block_table"], d["seq_lens"], d["positions"], out,
                        rope_theta=wl.rope_theta, scale=wl.scale, workspace=ws,
                        k_scales=d["k_scales"], v_scales=d["v_scales"])
        outs.append(out)
    assert K.kvattn_read_device_status(ws) == 0

    ref1, st1, kp, vp, ks, vs = oracle_decode(wl, h1)
    h2.update(k_pages=kp, v_pages=vp, k_scales=ks, v_scales=vs)
    ref2, st2, kp, vp, ks, vs = oracle_decode(wl, h2)
    assert st1 == st2 == 0
    assert np.array_equal(pool_bits(d1["k_pages"]), kp)
    assert np.array_equal(pool_bits(d1["v_pages"]), vp)
    if ks is not None:
        assert np.array_equal(d1["k_scales"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(d1["v_scales"].cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert_close(out_f64(outs[0]), ref1)
    assert_close(out_f64(outs[1]), ref2)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_selective_kv_over_a_sparse_block_table(kv):
    """Decode over a selectively kept cache ("C17 CPU-first LLM inference
    engine", section 5.3: initial tokens, recent tokens and a few important
    ones are kept, the rest evicted).  At page granularity the kept cache is a
    sparse block table: the sequence's first page, three middle pages and its
    last four.  seq_lens is the kept token count and positions the new token's
    true position, so the new token lands in the same physical slot, rotated
    the same way, as in the full cache, and attends over exactly the kept
    tokens."""
    L = 1000
    wl, h_full = custom(16, 4, [L], d=128, kv=kv, seed=9)
    keep = [0, 10, 31, 47, 59, 60, 61, 62]       # logical pages; 62 holds slot L
    assert L // wl.page_size == keep[-1]
    sparse = np.full_like(wl.block_table, -1)
    sparse[0, :len(keep)] = wl.block_table[0, keep]
    L_kept = wl.page_size * (len(keep) - 1) + L % wl.page_size
    wl_s = replace(W.with_lengths(wl, [L_kept], positions=[L]), block_table=sparse)
    h = dict(h_full)
    h["block_table"], h["seq_lens"], h["positions"] = sparse, wl_s.seq_lens, wl_s.positions
    check_against_oracle(wl_s, h)
    # the appended row is the full cache's: same slot, same position
    d = to_dev(h)
    run_gpu(wl_s, d)
    _, _, kp, vp, _, _ = oracle_decode(wl, h_full)
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)
