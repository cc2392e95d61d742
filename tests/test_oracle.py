"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check compares the oracle with something other than itself: closed
forms, invariants, degenerate cases that reduce to a mean or to a copy, and an
independent numpy float64 formula (tests/refmath.py) on tiny inputs.
"""
import math

import numpy as np
import pytest

import oracle
from decode_phase_gqa_gb300 import workloads as W
from tests import refmath as R
from tests.helpers import host_inputs, oracle_decode

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ RoPE ---

@pytest.mark.parametrize("d", [2, 8, 64, 128])
@pytest.mark.parametrize("pos", [0, 1, 7, 256, 4095, 32768])
def test_rope_preserves_norm(d, pos):
    x = RNG.standard_normal(d)
    y = oracle.rope_f64(x, pos, 1e4)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)


def test_rope_position_zero_and_nope_are_identity():
    x = RNG.standard_normal(64)
    assert np.array_equal(oracle.rope_f64(x, 0, 1e4), x)
    assert np.array_equal(oracle.rope_f64(x, 123, 0.0), x)
    assert np.array_equal(oracle.rope_f64(x, 123, -1.0), x)


@pytest.mark.parametrize("d", [4, 64, 128])
def test_rope_is_half_split_pairing(d):
    # a unit vector e_i (i < d/2) stays in span{e_i, e_{i+d/2}}: pairs are
    # (i, i + d/2), not adjacent (i, i + 1)
    h = d // 2
    for i in range(h):
        x = np.zeros(d)
        x[i] = 1.0
        y = oracle.rope_f64(x, 5, 1e4)
        mask = np.ones(d, bool)
        mask[[i, i + h]] = False
        assert np.all(y[mask] == 0.0)
        assert abs(y[i] ** 2 + y[i + h] ** 2 - 1.0) < 1e-14


def test_rope_first_pair_turns_by_position_counterclockwise():
    # pair 0 has frequency theta^0 = 1: e_0 goes to (cos p, sin p), e_h to (-sin p, cos p)
    d, h = 8, 4
    for p in (1, 2, 3, 100):
        x = np.zeros(d)
        x[0] = 1.0
        y = oracle.rope_f64(x, p, 1e4)
        assert abs(y[0] - math.cos(p)) < 1e-15 and abs(y[h] - math.sin(p)) < 1e-15
        x = np.zeros(d)
        x[h] = 1.0
        y = oracle.rope_f64(x, p, 1e4)
        assert abs(y[0] + math.sin(p)) < 1e-15 and abs(y[h] - math.cos(p)) < 1e-15


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6), (64, 5e5)])
def test_rope_matches_complex_rotation(d, theta):
    for p in (0, 3, 1000, 32768):
        x = RNG.standard_normal(d)
        # the two evaluate pow/cos/sin through different routines: the angle
        # p * freq agrees to a few double ulps of p, i.e. ~1e-11 at p = 32768
        assert np.allclose(oracle.rope_f64(x, p, theta), R.rope_complex(x, p, theta),
                           rtol=0, atol=1e-10)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6)])
def test_rope_frequencies_fall_geometrically(d, theta):
    # the angle of pair i at position 1 (recovered with atan2) is theta^(-2i/d):
    # first pair turns by 1 rad, each later pair by a factor theta^(-2/d) less
    h = d // 2
    ang = []
    for i in range(h):
        x = np.zeros(d)
        x[i] = 1.0
        y = oracle.rope_f64(x, 1, theta)
        ang.append(math.atan2(y[i + h], y[i]))
    ang = np.array(ang)
    assert abs(ang[0] - 1.0) < 1e-15
    ratio = ang[1:] / ang[:-1]
    assert np.allclose(ratio, theta ** (-2.0 / d), rtol=1e-12)


@pytest.mark.parametrize("d", [64, 128])
def test_rope_scores_depend_on_relative_position_only(d):
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    for m, n, s in ((7, 3, 100), (300, 299, 4000), (0, 0, 32768), (5, 50, 12345)):
        a = oracle.rope_f64(q, m, 1e6) @ oracle.rope_f64(k, n, 1e6)
        b = oracle.rope_f64(q, m + s, 1e6) @ oracle.rope_f64(k, n + s, 1e6)
        assert abs(a - b) < 1e-9 * max(1.0, abs(a))


# ------------------------------------------------------- storage recipe ---

def test_store_recipe_position_zero_keeps_key_bits():
    x = R.f32_to_bf16_bits(RNG.standard_normal(128))
    y = oracle.rope_store_f32(x, 0, 1e6)
    assert np.array_equal(R.f32_to_bf16_bits(y), x)
    y = oracle.rope_store_f32(x, 77, 0.0)
    assert np.array_equal(R.f32_to_bf16_bits(y), x)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6), (64, 5e5)])
def test_store_recipe_is_fp32_accurate_rotation(d, theta):
    for p in (1, 17, 4096, 32768):
        xb = R.f32_to_bf16_bits(RNG.standard_normal(d))
        y32 = oracle.rope_store_f32(xb, p, theta).astype(np.float64)
        y64 = R.rope_complex(R.bf16_bits_to_f64(xb), p, theta)
        mag = np.abs(R.bf16_bits_to_f64(xb)).max()
        # c, s rounded to fp32, two fp32 products and a sum: a few fp32 ulps
        assert np.max(np.abs(y32 - y64)) <= 8 * 2.0 ** -24 * mag * 2


def test_store_recipe_rounds_each_operation():
    # the recipe rounds c, s to fp32 and then every product and sum on its own;
    # c, s come from the double rotation of unit vectors (pinned above) and the
    # fp32 sequence is replayed with numpy float32 scalars (no fused multiply-add)
    d, theta = 128, 1e6
    h = d // 2
    for p in (3, 1000, 32768):
        cs = np.empty((h, 2))
        for i in range(h):
            e = np.zeros(d)
            e[i] = 1.0
            y = oracle.rope_f64(e, p, theta)
            cs[i] = y[i], y[i + h]
        c, s = cs[:, 0].astype(np.float32), cs[:, 1].astype(np.float32)
        xb = R.f32_to_bf16_bits(RNG.standard_normal(d))
        x = R.bf16_bits_to_f64(xb).astype(np.float32)
        lo, hi = x[:h], x[h:]
        want = np.concatenate([np.subtract(lo * c, hi * s, dtype=np.float32),
                               np.add(hi * c, lo * s, dtype=np.float32)])
        assert np.array_equal(oracle.rope_store_f32(xb, p, theta), want)


# ----------------------------------------------------------------- int8 ---

def test_int8_quant_properties():
    for _ in range(50):
        x = (RNG.standard_normal(128) * RNG.uniform(0.01, 100)).astype(np.float32)
        codes, sc = oracle.quant_int8(x)
        amax = np.abs(x).max()
        assert sc == np.float32(amax / np.float32(127.0))
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        assert abs(int(codes[np.argmax(np.abs(x))])) == 127
        err = np.abs(codes.astype(np.float64) * np.float64(sc) - x.astype(np.float64))
        assert np.all(err <= 0.5 * np.float64(sc) * (1 + 1e-6))
        assert np.all(np.sign(codes[np.abs(x) > sc]) == np.sign(x[np.abs(x) > sc]))


def test_int8_quant_zero_row_and_ties():
    codes, sc = oracle.quant_int8(np.zeros(64, np.float32))
    assert sc == 0.0 and not codes.any()
    # scale is exactly 2^-3 when max|x| = 127 * 2^-3; x/scale = 2.5, 3.5, -2.5 -> 2, 4, -2
    s = np.float32(2.0 ** -3)
    x = np.zeros(64, np.float32)
    x[0], x[1], x[2], x[3] = 127 * s, 2.5 * s, 3.5 * s, -2.5 * s
    codes, sc = oracle.quant_int8(x)
    assert sc == s
    assert list(codes[:4]) == [127, 2, 4, -2]


# -------------------------------------------------------------- attention --

def _tiny(n_qh, n_kvh, lens, d=64, page=16, kv="bf16", seed=0, theta=1e4, spare=0.5):
    wl = W.make_workload("custom", seed=seed, n_seq=len(lens), n_qh=n_qh, n_kvh=n_kvh,
                         head_dim=d, page_size=page, rope_theta=theta, kv_dtype=kv,
                         lengths=list(lens), spare=spare)
    return wl, host_inputs(wl)


def _np_reference(wl, h, kp, vp, ks, vs):
    out = np.empty((wl.n_seq, wl.n_qh, wl.head_dim))
    for b in range(wl.n_seq):
        L = int(wl.seq_lens[b])
        kr = R.gather_rows(kp, ks, wl.block_table, b, L, wl.page_size, wl.kv_dtype == "int8")
        vr = R.gather_rows(vp, vs, wl.block_table, b, L, wl.page_size, wl.kv_dtype == "int8")
        out[b] = R.attend_reference(h["q"][b], kr, vr, wl.positions[b], wl.rope_theta,
                                    wl.scale, wl.n_kvh)
    return out


@pytest.mark.parametrize("n_qh,n_kvh", [(1, 1), (2, 1), (4, 1), (4, 2), (8, 2)])
@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_brute_force_tiny(n_qh, n_kvh, kv):
    for lens in ([0], [1], [2], [3], [3, 0, 2], [15, 16, 17, 33]):
        wl, h = _tiny(n_qh, n_kvh, lens, kv=kv, seed=len(lens) + n_qh)
        out, st, kp, vp, ks, vs = oracle_decode(wl, h)
        assert st == 0
        ref = _np_reference(wl, h, kp, vp, ks, vs)
        assert np.max(np.abs(out - ref)) < 1e-12


def test_single_token_returns_its_value():
    for kv in ("bf16", "int8"):
        wl, h = _tiny(8, 2, [0, 0, 0], kv=kv, d=128)
        out, st, kp, vp, ks, vs = oracle_decode(wl, h)
        for b in range(3):
            for hh in range(8):
                j = hh // 4
                if kv == "bf16":
                    v = R.bf16_bits_to_f64(h["v_new"][b, j])
                else:
                    pg = wl.block_table[b, 0]
                    v = vp[pg, j, 0].astype(np.float64) * np.float64(vs[pg, j, 0])
                assert np.array_equal(out[b, hh], v)


def test_gqa_head_mapping_is_consecutive():
    # each KV head holds a constant value vector j+1; query head h must see h // g
    wl, h = _tiny(8, 4, [5], d=64)
    vp = h["v_pages"]
    for j in range(4):
        vp[:, j] = R.f32_to_bf16_bits(np.full(vp.shape[2:], j + 1, np.float32))
        h["v_new"][:, j] = R.f32_to_bf16_bits(np.full(64, j + 1, np.float32))
    out, *_ = oracle_decode(wl, h)
    for hh in range(8):
        assert np.allclose(out[0, hh], hh // 2 + 1, atol=1e-12, rtol=0)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_identical_keys_give_mean_of_values(kv):
    wl, h = _tiny(4, 2, [40], kv=kv, d=64)
    # append first, then copy the stored new key into every cached slot
    kp, vp = h["k_pages"], h["v_pages"]
    ks, vs = h["k_scales"], h["v_scales"]
    oracle.append(h["k_new"], h["v_new"], kp, vp, wl.block_table, wl.seq_lens,
                  wl.positions, wl.rope_theta, ks, vs)
    L, P = 40, wl.page_size
    pl, ol = wl.block_table[0, L // P], L % P
    for t in range(L):
        pg, o = wl.block_table[0, t // P], t % P
        kp[pg, :, o] = kp[pl, :, ol]
        if ks is not None:
            ks[pg, :, o] = ks[pl, :, ol]
    out, st = oracle.attend_paged(h["q"], kp, vp, wl.block_table, wl.seq_lens,
                                  wl.positions, wl.rope_theta, wl.scale, ks, vs)
    vr = R.gather_rows(vp, vs, wl.block_table, 0, L, P, kv == "int8")
    for hh in range(4):
        assert np.max(np.abs(out[0, hh] - vr[:, hh // 2].mean(axis=0))) < 1e-12


def test_zero_query_and_zero_scale_give_mean_of_values():
    wl, h = _tiny(4, 1, [70], d=64)
    h2 = dict(h)
    h2["q"] = np.zeros_like(h["q"])
    out, _, kp, vp, ks, vs = oracle_decode(wl, h2)
    vr = R.gather_rows(vp, None, wl.block_table, 0, 70, 16, False)
    assert np.max(np.abs(out[0] - vr[:, 0].mean(axis=0))) < 1e-12
    wl0 = W.make_workload("custom", seed=0, n_seq=1, n_qh=4, n_kvh=1, head_dim=64,
                          lengths=[70], spare=0.5, scale=0.0)
    out, _, kp, vp, ks, vs = oracle_decode(wl0, host_inputs(wl0))
    vr = R.gather_rows(vp, None, wl0.block_table, 0, 70, 16, False)
    assert np.max(np.abs(out[0] - vr[:, 0].mean(axis=0))) < 1e-12


def test_two_tokens_closed_form():
    wl, h = _tiny(2, 1, [1], d=64, theta=1e4)
    out, _, kp, vp, _, _ = oracle_decode(wl, h)
    kr = R.gather_rows(kp, None, wl.block_table, 0, 1, 16, False)[:, 0]
    vr = R.gather_rows(vp, None, wl.block_table, 0, 1, 16, False)[:, 0]
    for hh in range(2):
        qh = R.rope_complex(R.bf16_bits_to_f64(h["q"][0, hh]), wl.positions[0], 1e4)
        s0, s1 = wl.scale * (qh @ kr[0]), wl.scale * (qh @ kr[1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        assert np.max(np.abs(out[0, hh] - (w0 * vr[0] + w1 * vr[1]))) < 1e-12


def test_new_token_is_attended():
    # a new key aligned with q and huge scale: the output collapses onto v_new
    wl, h = _tiny(1, 1, [30], d=64, theta=0.0)
    h["k_new"][0, 0] = h["q"][0, 0]
    wl.scale = 50.0
    out, *_ = oracle_decode(wl, h)
    assert np.max(np.abs(out[0, 0] - R.bf16_bits_to_f64(h["v_new"][0, 0]))) < 1e-6


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_paged_equals_contiguous_exactly(kv):
    wl, h = _tiny(8, 2, [0, 15, 16, 47, 100], kv=kv, d=64)
    out, _, kp, vp, ks, vs = oracle_decode(wl, h)
    kc = np.concatenate([R.gather_rows(kp, ks, wl.block_table, b, int(L), 16, kv == "int8")
                         for b, L in enumerate(wl.seq_lens)])
    vc = np.concatenate([R.gather_rows(vp, vs, wl.block_table, b, int(L), 16, kv == "int8")
                         for b, L in enumerate(wl.seq_lens)])
    out_c = oracle.attend_contiguous(h["q"], np.ascontiguousarray(kc), np.ascontiguousarray(vc),
                                     wl.seq_lens, wl.positions, wl.n_kvh, wl.rope_theta, wl.scale)
    assert np.array_equal(out, out_c)


def test_page_permutation_does_not_change_result():
    wl, h = _tiny(4, 1, [100, 63], d=64, spare=0.0)
    out1, _, kp, vp, _, _ = oracle_decode(wl, h)
    # relabel the physical pages with a new permutation and move the data along
    perm = np.random.default_rng(9).permutation(wl.num_pages).astype(np.int32)
    h2 = dict(h)
    h2["k_pages"] = np.empty_like(h["k_pages"])
    h2["v_pages"] = np.empty_like(h["v_pages"])
    h2["k_pages"][perm] = h["k_pages"]
    h2["v_pages"][perm] = h["v_pages"]
    bt = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    wl2 = W.with_lengths(wl, wl.seq_lens)
    wl2.block_table = bt
    h2["block_table"] = bt
    out2, *_ = oracle_decode(wl2, h2)
    assert np.array_equal(out1, out2)


def test_large_scores_stay_finite():
    wl, h = _tiny(4, 1, [50], d=64)
    wl.scale = 1e3
    out, _, kp, vp, ks, vs = oracle_decode(wl, h)
    assert np.all(np.isfinite(out))
    ref = _np_reference(wl, h, kp, vp, ks, vs)
    assert np.max(np.abs(out - ref)) < 1e-9


def test_invalid_length_and_page_are_reported():
    wl, h = _tiny(4, 1, [20, 20, 20], d=64)
    bad = dict(h)
    bad["seq_lens"] = np.array([20, -1, 20], np.int32)
    wl_bad = W.with_lengths(wl, bad["seq_lens"], np.array([20, 20, 20], np.int32))
    out, st, *_ = oracle_decode(wl_bad, bad)
    assert st & oracle.BAD_LEN
    assert np.all(np.isnan(out[1])) and np.all(np.isfinite(out[0]))
    # a poisoned first page: those 16 tokens are invisible, the rest attends
    bt = wl.block_table.copy()
    bt[2, 0] = wl.num_pages + 5
    wl2 = W.with_lengths(wl, wl.seq_lens)
    wl2.block_table = bt
    h2 = dict(h)
    h2["block_table"] = bt
    out2, st2, kp, vp, _, _ = oracle_decode(wl2, h2)
    assert st2 & oracle.BAD_PAGE
    t = np.arange(16, 21)
    kr = R.bf16_bits_to_f64(kp[bt[2, t // 16], :, t % 16])
    vr = R.bf16_bits_to_f64(vp[bt[2, t // 16], :, t % 16])
    ref = R.attend_reference(h["q"][2], kr, vr, 20, wl.rope_theta, wl.scale, 1)
    assert np.max(np.abs(out2[2] - ref)) < 1e-12


def test_append_touches_only_the_new_slot():
    wl, h = _tiny(8, 2, [0, 17, 31], d=64, kv="bf16")
    before = h["k_pages"].copy(), h["v_pages"].copy()
    _, _, kp, vp, _, _ = oracle_decode(wl, h)
    changed = np.zeros(kp.shape[:3], bool)
    for b, L in enumerate(wl.seq_lens):
        changed[wl.block_table[b, L // 16], :, L % 16] = True
    for new, old in ((kp, before[0]), (vp, before[1])):
        diff = np.any(new != old, axis=-1)
        assert not np.any(diff & ~changed)
    # value rows are copied bit for bit
    for b, L in enumerate(wl.seq_lens):
        assert np.array_equal(vp[wl.block_table[b, L // 16], :, L % 16], h["v_new"][b])


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("n_kvh,d,page,theta", [(1, 64, 16, 1e4), (2, 128, 16, 1e6),
                                                 (4, 64, 32, 5e5), (2, 128, 8, 0.0)])
def test_append_stores_the_recipe_values(kv, n_kvh, d, page, theta):
    # Every appended slot is rebuilt from the storage recipe of the pages
    # ("LLM inference from smollm3.go": the new k/v are written at the current
    # slot after RoPE, section "KV cache"; a quantised row is int8 codes with
    # one fp32 scale max|x|/127, section "int8 weight-only quantization"),
    # replayed in numpy float32 by tests/refmath.py, and compared bit for bit
    # with what the oracle wrote.  RoPE positions differ from the slots, so a
    # key rotated at its slot (or not at all) shows; one key row and one value
    # row are zero, so the zero-row rule of the quantiser shows.
    rng = np.random.default_rng(d * 7 + page + n_kvh)
    lens = [0, 5, page - 1, page, 3 * page + 2]
    wl, h = _tiny(2 * n_kvh, n_kvh, lens, d=d, page=page, kv=kv, theta=theta,
                  seed=d + n_kvh)
    pos = (wl.seq_lens + rng.integers(1, 40000, size=len(lens))).astype(np.int32)
    h["positions"] = pos
    wl.positions = pos
    h["k_new"][1, 0, :] = 0
    h["v_new"][2, n_kvh - 1, :] = 0
    kp, vp = h["k_pages"].copy(), h["v_pages"].copy()
    ks = None if h["k_scales"] is None else h["k_scales"].copy()
    vs = None if h["v_scales"] is None else h["v_scales"].copy()
    st = oracle.append(h["k_new"], h["v_new"], kp, vp, wl.block_table, wl.seq_lens, pos,
                       theta, ks, vs)
    assert st == 0
    for b, L in enumerate(wl.seq_lens):
        pg, off = wl.block_table[b, L // page], L % page
        for j in range(n_kvh):
            kf = R.store_key_f32(h["k_new"][b, j], int(pos[b]), theta)
            if kv == "bf16":
                assert np.array_equal(kp[pg, j, off], R.f32_to_bf16_bits(kf))
                assert np.array_equal(vp[pg, j, off], h["v_new"][b, j])
            else:
                kc, kscale = R.quant_row_int8(kf)
                vc, vscale = R.quant_row_int8(R.bf16_bits_to_f64(h["v_new"][b, j]))
                assert np.array_equal(kp[pg, j, off], kc)
                assert np.array_equal(vp[pg, j, off], vc)
                assert ks[pg, j, off].view(np.uint32) == np.float32(kscale).view(np.uint32)
                assert vs[pg, j, off].view(np.uint32) == np.float32(vscale).view(np.uint32)
    # the zero rows really are zero after storage
    if kv == "int8":
        b1 = wl.block_table[1, wl.seq_lens[1] // page]
        assert ks[b1, 0, wl.seq_lens[1] % page] == 0 and not kp[b1, 0, wl.seq_lens[1] % page].any()


def test_tiny_config_end_to_end_against_numpy():
    wl = W.make_workload("tiny", seed=0)
    assert wl.num_pages == 17 and list(wl.seq_lens) == [256]
    assert sorted(wl.block_table[0, :17]) == list(range(17))
    h = host_inputs(wl)
    out, st, kp, vp, ks, vs = oracle_decode(wl, h)
    assert st == 0
    ref = _np_reference(wl, h, kp, vp, ks, vs)
    assert np.max(np.abs(out - ref)) < 1e-12
