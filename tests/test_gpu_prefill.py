"""Paged chunked prefill (kvattn_prefill) against the oracle (needs a GB300).

The oracle's prefill is the decode steps it is made of (tests/helpers.py,
oracle_prefill): step i appends new token i of every sequence and attends over
the cache up to it.  Checks: the whole pool bit for bit after the appends,
every output row within max-abs 2e-2 / mean-abs 2e-3, the status word.
"""
import numpy as np
import pytest
import torch

from decode_phase_gqa_gb300 import kvattn as K
from decode_phase_gqa_gb300 import workloads as W
from tests import refmath as R
from tests.gpu_helpers import assert_close, out_f64, pool_bits, run_gpu, to_dev
from tests.helpers import bits, host_inputs, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu


def make_case(n_qh, n_kvh, ctx, n_new, d=128, page=16, seed=0, theta=1e6, kv="bf16"):
    """A pool and table covering ctx + n_new tokens per sequence, and the new
    tokens' q / k / v (N(0,1), bf16), back to back."""
    ctx = np.asarray(ctx, np.int32)
    n_new = np.asarray(n_new, np.int32)
    wl = W.make_workload("custom", seed=seed, n_seq=len(ctx), n_qh=n_qh, n_kvh=n_kvh,
                         head_dim=d, page_size=page, rope_theta=theta, kv_dtype=kv,
                         lengths=[int(x) for x in np.maximum(ctx + n_new - 1, 0)], spare=0.1)
    h = host_inputs(wl)
    g = torch.Generator().manual_seed(1000 + seed)
    T = int(n_new.sum())
    h["q"] = bits(torch.randn((T, n_qh, d), generator=g).to(torch.bfloat16))
    h["k_new"] = bits(torch.randn((T, n_kvh, d), generator=g).to(torch.bfloat16))
    h["v_new"] = bits(torch.randn((T, n_kvh, d), generator=g).to(torch.bfloat16))
    starts = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    return wl, h, starts, ctx


def run_prefill(wl, h, starts, ctx, max_new=None, split=True):
    d = to_dev(h)
    ss = torch.from_numpy(starts).cuda()
    cl = torch.from_numpy(np.ascontiguousarray(ctx)).cuda()
    out = torch.full_like(d["q"], float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx = int(np.diff(starts).max(initial=0)) if max_new is None else max_new
    ws = None
    if split:   # NaN-filled: no split may read what it did not write
        n = K.kvattn_prefill_workspace_size(d["q"].shape[0], d["q"].shape[1], d["q"].shape[2])
        ws = torch.full((n // 4,), float("nan"), dtype=torch.float32, device="cuda")
    K.kvattn_prefill(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                     d["block_table"], ss, cl, out, rope_theta=wl.rope_theta, scale=wl.scale,
                     max_new_tokens=mx, k_scales=d["k_scales"], v_scales=d["v_scales"],
                     dev_status=st, workspace=ws)
    torch.cuda.synchronize()
    return out, int(st.item()), d


def check(wl, h, starts, ctx, split=True):
    out, st, d = run_prefill(wl, h, starts, ctx, split=split)
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, wl.rope_theta, wl.scale)
    assert st == 0 and ost == 0, (st, ost)
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)
    ks, vs = oracle_prefill.scales
    if ks is not None:
        assert np.array_equal(d["k_scales"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(d["v_scales"].cpu().numpy().view(np.uint32), vs.view(np.uint32))
    return assert_close(out_f64(out), ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_qh,n_kvh", [(4, 1), (16, 4), (8, 2)])
def test_prompts_into_empty_caches(d, n_qh, n_kvh):
    # ragged prompts: one token, exactly a 16-token tile, one past, several key tiles
    wl, h, starts, ctx = make_case(n_qh, n_kvh, [0, 0, 0, 0], [1, 16, 17, 150], d=d, seed=d + n_qh)
    check(wl, h, starts, ctx)


@pytest.mark.parametrize("d", [64, 128])
def test_chunked_prefill_after_cached_tokens(d):
    wl, h, starts, ctx = make_case(16, 4, [100, 0, 37, 511], [20, 5, 64, 33], d=d, seed=3)
    check(wl, h, starts, ctx)


@pytest.mark.parametrize("split", [True, False])
def test_speculative_verification_of_draft_tokens(split):
    """Four draft tokens per sequence over long caches (Qwen3-8B-shaped heads),
    with the key tiles split among 16 CTAs and merged, and without."""
    wl, h, starts, ctx = make_case(32, 8, [1000, 3, 257, 4000], [4, 4, 4, 4], d=128, seed=5)
    check(wl, h, starts, ctx, split=split)


@pytest.mark.parametrize("page", [32, 64, 256])
def test_page_sizes(page):
    wl, h, starts, ctx = make_case(8, 2, [30, 300, 0], [40, 9, 70], d=64, page=page, seed=page)
    check(wl, h, starts, ctx)


def test_long_prompt():
    wl, h, starts, ctx = make_case(16, 4, [0, 64], [600, 333], d=128, seed=7)
    check(wl, h, starts, ctx)


@pytest.mark.parametrize("d", [64, 128])
def test_long_prompts_without_splits(d):
    # no workspace: every query tile's keys go through one CTA of the
    # tensor-core kernel (prompts above 64 new tokens over a bf16 cache)
    wl, h, starts, ctx = make_case(16, 4, [0, 0, 130, 0], [65, 200, 97, 300], d=d, seed=13)
    check(wl, h, starts, ctx, split=False)


@pytest.mark.parametrize("split", [False, True])
def test_more_prompt_tiles_than_sms(split):
    """More 64-token query tiles than the GPU has SMs, so each CTA of the
    persistent tensor-core kernel walks several of them (query rows reloaded,
    tensor memory and rings reused, barrier phases carried on), with
    prompts of 65..160 tokens over short cached prefixes and a page mix."""
    rng = np.random.default_rng(29)
    n = 180
    ctx = [int(x) for x in rng.integers(0, 40, n)]
    n_new = [int(x) for x in rng.integers(65, 161, n)]
    wl, h, starts, ctx = make_case(4, 1, ctx, n_new, d=128, seed=29)
    check(wl, h, starts, ctx, split=split)


def test_long_prompt_eight_query_heads_per_kv_head():
    # a group of 8 query heads is two CTAs of 4 heads each
    wl, h, starts, ctx = make_case(16, 2, [0, 40], [400, 129], d=128, seed=17)
    check(wl, h, starts, ctx)
    check(wl, h, starts, ctx, split=False)


@pytest.mark.parametrize("d", [64, 128])
def test_pool_slots_past_the_keys_may_hold_nan(d):
    # every pool slot no key occupies (before or after the step) is a NaN:
    # the rows past a sequence's last key inside its last 16-key block must
    # not reach the weighted sum
    wl, h, starts, ctx = make_case(16, 4, [0, 0, 0], [77, 130, 250], d=d, seed=19)
    nan = np.uint16(0x7FC1)
    h["k_pages"][:] = nan
    h["v_pages"][:] = nan
    check(wl, h, starts, ctx)
    check(wl, h, starts, ctx, split=False)


def test_bad_page_in_a_long_prompt_is_reported():
    wl, h, starts, ctx = make_case(8, 2, [64, 0], [100, 180], d=128, seed=23)
    bt = h["block_table"].copy()
    bt[0, 2] = -7                # cached tokens 32-47 of sequence 0 left out
    h["block_table"] = bt
    out, st, d = run_prefill(wl, h, starts, ctx, split=False)
    assert st & K.KVATTN_DEV_BAD_PAGE
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, wl.rope_theta, wl.scale)
    assert ost & 2
    assert_close(out_f64(out), ref)
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)


def test_one_new_token_is_the_decode_step():
    """n_b = 1 is kvattn_decode with seq_lens = positions = ctx: the same
    appended rows bit for bit, outputs within the tolerance of the oracle."""
    wl, h, starts, ctx = make_case(16, 4, [50, 0, 300, 1023], [1, 1, 1, 1], d=128, seed=9)
    out, st, d = run_prefill(wl, h, starts, ctx)
    hd = dict(h, seq_lens=ctx.copy(), positions=ctx.copy())
    wld = W.with_lengths(wl, ctx)
    dd = to_dev(hd)
    dec, st2, _ = run_gpu(wld, dd)
    assert st == st2 == 0
    assert np.array_equal(pool_bits(d["k_pages"]), pool_bits(dd["k_pages"]))
    assert np.array_equal(pool_bits(d["v_pages"]), pool_bits(dd["v_pages"]))
    ref, *_ = oracle_decode(wld, hd)
    assert_close(out_f64(out), ref)
    assert_close(out_f64(dec), ref)


def test_bad_page_and_overfull_sequence_are_reported():
    wl, h, starts, ctx = make_case(8, 2, [40, 20, 10], [30, 10, 10], d=64, seed=11)
    bt = h["block_table"].copy()
    bt[0, 1] = 10 ** 6           # cached tokens 16-31 of sequence 0 left out
    h["block_table"] = bt
    cap = bt.shape[1] * wl.page_size
    ctx = ctx.copy()
    ctx[2] = cap - 5             # 10 new tokens cannot fit: sequence 2 is skipped
    out, st, d = run_prefill(wl, h, starts, ctx)
    assert st & K.KVATTN_DEV_BAD_PAGE and st & K.KVATTN_DEV_BAD_LEN
    got = out_f64(out)
    assert np.all(np.isnan(got[starts[2]:starts[3]])), "the skipped sequence's rows were written"
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, wl.rope_theta, wl.scale, seqs=[0, 1])
    assert ost & 2
    assert_close(got[:starts[2]], ref[:starts[2]])
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)


@pytest.mark.parametrize("kind", ["prefill", "verify", "verify_int8"])
def test_benchmark_shapes_at_full_size(kind):
    """The shapes the benchmark times, drawn as it draws them (on the GPU,
    same seeds) and run with its workspace: 8 SmolLM3-shaped prompts of 2048
    tokens into empty caches, and 4 draft tokens over each of the Qwen3-shaped
    batch's 64 caches, bf16 and int8.  Every pool (and int8 scale) bit for bit,
    every output row in tolerance."""
    import math
    if kind == "prefill":
        n_qh, n_kvh, d, theta = 16, 4, 128, 1e6
        ctx = np.zeros(8, np.int64)
        n_new = np.full(8, 2048, np.int64)
    else:
        q3 = W.make_workload("qwen3", seed=0)
        n_qh, n_kvh, d, theta = q3.n_qh, q3.n_kvh, q3.head_dim, q3.rope_theta
        ctx = q3.seq_lens.astype(np.int64)
        n_new = np.full(len(ctx), 4, np.int64)
    wl = W.make_workload("custom", seed=0, n_seq=len(ctx), n_qh=n_qh, n_kvh=n_kvh, head_dim=d,
                         page_size=16, rope_theta=theta,
                         kv_dtype="int8" if kind == "verify_int8" else "bf16",
                         lengths=[int(x) for x in ctx + n_new - 1], spare=0.05)
    dev = torch.device("cuda")
    t = W.make_tensors(wl, device=dev)
    g = torch.Generator(device=dev).manual_seed(77)
    T = int(n_new.sum())
    q = torch.randn((T, n_qh, d), generator=g, device=dev).to(torch.bfloat16)
    kn = torch.randn((T, n_kvh, d), generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn((T, n_kvh, d), generator=g, device=dev).to(torch.bfloat16)
    h = {"q": bits(q), "k_new": bits(kn), "v_new": bits(vn), "k_pages": bits(t["k_pages"]),
         "v_pages": bits(t["v_pages"]), "block_table": wl.block_table.copy()}
    if t.get("k_scales") is not None:
        h["k_scales"], h["v_scales"] = bits(t["k_scales"]), bits(t["v_scales"])
    starts = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    out = torch.full_like(q, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(K.kvattn_prefill_workspace_size(T, n_qh, d), dtype=torch.uint8, device=dev)
    K.kvattn_prefill(q, kn, vn, t["k_pages"], t["v_pages"], torch.from_numpy(wl.block_table).to(dev),
                     torch.from_numpy(starts).to(dev), torch.from_numpy(ctx.astype(np.int32)).to(dev),
                     out, rope_theta=theta, scale=1.0 / math.sqrt(d),
                     max_new_tokens=int(n_new.max()), k_scales=t.get("k_scales"),
                     v_scales=t.get("v_scales"), dev_status=st, workspace=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, theta, 1.0 / math.sqrt(d))
    assert ost == 0
    assert np.array_equal(pool_bits(t["k_pages"]), kp)
    assert np.array_equal(pool_bits(t["v_pages"]), vp)
    ks, vs = oracle_prefill.scales
    if ks is not None:
        assert np.array_equal(t["k_scales"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(t["v_scales"].cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert_close(out_f64(out), ref)


@pytest.mark.parametrize("ctx0,prompt", [([0, 40], [70, 9]),      # 16-token query tiles
                                         ([100, 700], [3, 4])])   # the short-chunk kernel
def test_decode_after_prefill_reads_the_prefilled_cache(ctx0, prompt):
    """A prompt (or drafts) through kvattn_prefill, then two decode steps
    through kvattn_decode: the steps attend over the keys the prefill
    appended, and the whole sequence equals the oracle's decode steps one
    token at a time."""
    n_qh, n_kvh, d = 16, 4, 128
    ctx0, prompt, steps = np.array(ctx0, np.int32), np.array(prompt, np.int32), 2
    # pages for the prompt and the decode steps that follow
    wl, h, starts, ctx = make_case(n_qh, n_kvh, ctx0, prompt + steps, d=d, seed=17)
    T = int(prompt.sum())
    rows = np.concatenate([np.arange(starts[b], starts[b] + prompt[b]) for b in range(2)])
    later = [starts[:-1] + prompt + s for s in range(steps)]  # rows of each decode token
    hp = dict(h, q=h["q"][rows].copy(), k_new=h["k_new"][rows].copy(), v_new=h["v_new"][rows].copy())
    pstarts = np.concatenate([[0], np.cumsum(prompt)]).astype(np.int32)
    out, st, dv = run_prefill(wl, hp, pstarts, ctx0)
    assert st == 0
    ref_p, ost, kp, vp = oracle_prefill(hp, pstarts, ctx0, wl.rope_theta, wl.scale)
    assert ost == 0
    assert_close(out_f64(out), ref_p)
    hd = {"k_pages": kp, "v_pages": vp, "block_table": h["block_table"], "k_scales": None,
          "v_scales": None}
    for s in range(steps):
        L = (ctx0 + prompt + s).astype(np.int32)
        hs = dict(hd, q=h["q"][later[s]].copy(), k_new=h["k_new"][later[s]].copy(),
                  v_new=h["v_new"][later[s]].copy(), seq_lens=L, positions=L)
        wls = W.with_lengths(wl, L)
        dd = to_dev(hs)
        dd["k_pages"], dd["v_pages"] = dv["k_pages"], dv["v_pages"]   # the GPU's own cache
        dec, st2, _ = run_gpu(wls, dd)
        ref, ost2, kp, vp, _, _ = oracle_decode(wls, hs)
        assert st2 == 0 and ost2 == 0
        assert np.array_equal(pool_bits(dv["k_pages"]), kp)
        assert np.array_equal(pool_bits(dv["v_pages"]), vp)
        assert_close(out_f64(dec), ref)
        hd = dict(hd, k_pages=kp, v_pages=vp)


def test_tokens_past_max_new_tokens_are_left_out():
    """A sequence with more new tokens than max_new_tokens: the first
    max_new_tokens are appended and attended, the rest neither, and the status
    says so; the other sequences are untouched by it."""
    wl, h, starts, ctx = make_case(8, 2, [10, 30], [20, 50], d=64, seed=19)
    out, st, d = run_prefill(wl, h, starts, ctx, max_new=32)
    assert st & K.KVATTN_DEV_BAD_LEN
    got = out_f64(out)
    cut = starts[1] + 32            # rows of sequence 1 past the launch's 32 tokens
    assert np.all(np.isnan(got[cut:starts[2]]))
    short = np.concatenate([[0], np.cumsum([20, 32])]).astype(np.int32)
    keep = np.r_[0:starts[1] + 32]
    hs = dict(h, q=h["q"][keep].copy(), k_new=h["k_new"][keep].copy(), v_new=h["v_new"][keep].copy())
    ref, ost, kp, vp = oracle_prefill(hs, short, ctx, wl.rope_theta, wl.scale)
    assert ost == 0
    assert_close(got[:cut], ref)
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("ctx,n_new", [([0, 0, 0], [1, 17, 150]),            # prompts
                                       ([100, 37, 511], [20, 64, 33]),       # chunks
                                       ([1000, 3, 4000], [4, 4, 4])])        # drafts
def test_int8_cache(d, ctx, n_new):
    """The int8 cache: appended rows quantised by the decode step's recipe
    (codes and scales bit for bit), attention over the dequantised rows."""
    wl, h, starts, ctx = make_case(16, 4, ctx, n_new, d=d, seed=d + len(n_new), kv="int8")
    check(wl, h, starts, ctx)


def test_int8_one_new_token_is_the_decode_step():
    wl, h, starts, ctx = make_case(32, 8, [50, 0, 300, 1023], [1, 1, 1, 1], d=128, seed=23, kv="int8")
    out, st, d = run_prefill(wl, h, starts, ctx)
    hd = dict(h, seq_lens=ctx.copy(), positions=ctx.copy())
    wld = W.with_lengths(wl, ctx)
    dd = to_dev(hd)
    dec, st2, _ = run_gpu(wld, dd)
    assert st == st2 == 0
    for k in ("k_pages", "v_pages"):
        assert np.array_equal(pool_bits(d[k]), pool_bits(dd[k]))
    for k in ("k_scales", "v_scales"):
        assert torch.equal(d[k], dd[k])
    ref, *_ = oracle_decode(wld, hd)
    assert_close(out_f64(out), ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_qh,n_kvh", [(4, 1), (32, 8), (16, 2)])
def test_short_chunks(d, n_qh, n_kvh):
    """At most 4 new tokens a sequence (the kernel whose MMA rows are tokens x
    heads): ragged chunks of 1..4 and none, caches from empty to several
    64-key stages and splits, groups of one and of two head quads."""
    wl, h, starts, ctx = make_case(n_qh, n_kvh, [0, 63, 64, 700, 5, 2000], [4, 1, 3, 2, 0, 4],
                                   d=d, seed=d + n_qh + n_kvh)
    check(wl, h, starts, ctx)
    check(wl, h, starts, ctx, split=False)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_short_chunk_over_the_most_splits(kv):
    """Drafts of 4 and 2 tokens over 24000 and 3 cached keys: the long one's
    376 stages go to the most splits a query tile takes (16), each a quarter
    shorter than the one before, the last ones a few stages long; every split's
    partial state meets the others in the merge."""
    wl, h, starts, ctx = make_case(8, 2, [24000, 3], [4, 2], kv=kv, seed=5)
    check(wl, h, starts, ctx)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("page", [16, 64, 256])
def test_short_chunks_page_sizes(page, kv):
    wl, h, starts, ctx = make_case(8, 2, [30, 600, 0, 4095], [4, 2, 1, 3], d=128, page=page,
                                   seed=page + 1, kv=kv)
    check(wl, h, starts, ctx)


@pytest.mark.parametrize("d", [64, 128])
def test_short_chunks_int8(d):
    """Short chunks over an int8 cache: ragged 0..4 new tokens, caches from
    empty to several splits, with and without splits."""
    wl, h, starts, ctx = make_case(16, 4, [0, 63, 64, 700, 5, 2000], [4, 1, 3, 2, 0, 4], d=d,
                                   seed=d + 43, kv="int8")
    check(wl, h, starts, ctx)
    check(wl, h, starts, ctx, split=False)


def test_short_chunks_bad_page_and_tokens_past_the_bound():
    """max_new_tokens = 4 with a 6-token sequence: its first 4 tokens only,
    and the status says so; a page out of range is reported, its keys left out."""
    wl, h, starts, ctx = make_case(8, 2, [40, 300], [3, 6], d=64, seed=29)
    bt = h["block_table"].copy()
    bt[0, 1] = 10 ** 6           # cached tokens 16-31 of sequence 0
    h["block_table"] = bt
    out, st, d = run_prefill(wl, h, starts, ctx, max_new=4)
    assert st & K.KVATTN_DEV_BAD_PAGE and st & K.KVATTN_DEV_BAD_LEN
    got = out_f64(out)
    cut = starts[1] + 4
    assert np.all(np.isnan(got[cut:]))
    keep = np.r_[0:cut]
    hs = dict(h, q=h["q"][keep].copy(), k_new=h["k_new"][keep].copy(), v_new=h["v_new"][keep].copy())
    short = np.array([0, 3, 7], np.int32)
    ref, ost, kp, vp = oracle_prefill(hs, short, ctx, wl.rope_theta, wl.scale)
    assert ost & 2
    assert_close(got[:cut], ref)
    assert np.array_equal(pool_bits(d["k_pages"]), kp)
    assert np.array_equal(pool_bits(d["v_pages"]), vp)


def test_short_chunks_workspace_reused_across_calls():
    """The split counters live in the workspace and are reset by every call:
    two calls on one workspace (the second re-appends the same rows) give the
    oracle's outputs both times."""
    wl, h, starts, ctx = make_case(32, 8, [3000, 1500, 5000], [4, 3, 4], d=128, seed=31)
    d = to_dev(h)
    ss = torch.from_numpy(starts).cuda()
    cl = torch.from_numpy(np.ascontiguousarray(ctx)).cuda()
    n = K.kvattn_prefill_workspace_size(d["q"].shape[0], d["q"].shape[1], d["q"].shape[2])
    ws = torch.full((n // 4,), float("nan"), dtype=torch.float32, device="cuda")
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, wl.rope_theta, wl.scale)
    assert ost == 0
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        K.kvattn_prefill(d["q"], d["k_new"], d["v_new"], d["k_pages"], d["v_pages"],
                         d["block_table"], ss, cl, out, rope_theta=wl.rope_theta, scale=wl.scale,
                         max_new_tokens=4, dev_status=st, workspace=ws)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(pool_bits(d["k_pages"]), kp)
        assert_close(out_f64(out), ref)


@pytest.mark.parametrize("max_new", [3, 20])
def test_many_sequences_with_empty_chunks(max_new):
    """1100 sequences (three rounds of the row -> sequence search), a third of
    them with no new token (equal starts), short caches: both kernels."""
    rng = np.random.default_rng(37 + max_new)
    n_new = rng.integers(0, 4, 1100)
    n_new[-1] = 3
    if max_new > 4:
        n_new[::97] = 20
    ctx = rng.integers(0, 41, 1100)
    wl, h, starts, ctx = make_case(4, 1, ctx, n_new, d=64, seed=41 + max_new)
    check(wl, h, starts, ctx)


# ---- range: peaked scores, int8 row scales far from 1 -------------------------

def _stored_key(h, wl, starts, ctx, b, kk, j):
    """The key attention sees at index kk of sequence b, KV head j (NoPE): a
    cached row (bf16 bits, or int8 codes x scale rounded to bf16), else the new
    token's k_new row."""
    P = wl.page_size
    if kk < ctx[b]:
        pg, off = h["block_table"][b, kk // P], kk % P
        if wl.kv_dtype == "int8":
            return R.f32_to_bf16_bits(h["k_pages"][pg, j, off].astype(np.float64) * h["k_scales"][pg, j, off])
        return h["k_pages"][pg, j, off].copy()
    return h["k_new"][starts[b] + kk - ctx[b], j].copy()


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("kind", ["prompts", "chunks", "drafts"])
def test_peaked_scores(kind, kv):
    """Scale 30 and every query equal to one key it sees (NoPE): one score
    exceeds the others by thousands, so the softmax is a single weight of 1.
    Through every attention kernel: the tcgen05 one (prompts over a bf16
    cache), the 16-token one (chunks, and int8 prompts) and the short one
    (drafts)."""
    ctx, n_new = {"prompts": ([0, 40], [130, 97]), "chunks": ([300, 17], [33, 50]),
                  "drafts": ([900, 70], [4, 3])}[kind]
    wl, h, starts, ctx = make_case(8, 2, ctx, n_new, d=128, seed=51, theta=0.0, kv=kv)
    wl.scale = 30.0
    g = 4
    for b in range(len(ctx)):
        for i in range(int(np.diff(starts)[b])):
            kk = (int(ctx[b]) + i) // 2
            for hq in range(8):
                h["q"][starts[b] + i, hq] = _stored_key(h, wl, starts, ctx, b, kk, hq // g)
    check(wl, h, starts, ctx)


def _scaled_bf16(u16, factor):
    return R.f32_to_bf16_bits(R.bf16_bits_to_f64(u16) * factor)


_RANGE_CASES = {"prompts": ([200, 0], [100, 80]), "chunks": ([300, 170], [33, 20]),
                "drafts": ([900, 170], [4, 3])}


@pytest.mark.parametrize("factor", [1e-7, 1e5])
@pytest.mark.parametrize("kind", ["prompts", "chunks", "drafts"])
def test_int8_value_scales_far_from_one(kind, factor):
    """Every value row, cached and new, multiplied by 1e-7 (dequantised values
    below f16's smallest subnormal) or by 1e5 (beyond f16's largest finite
    value): the outputs move with them, compared with the oracle relative to
    each output row's size."""
    ctx, n_new = _RANGE_CASES[kind]
    wl, h, starts, ctx = make_case(8, 2, ctx, n_new, d=128, seed=53, kv="int8")
    P = wl.page_size
    for b in range(len(ctx)):
        for t in range(int(ctx[b])):
            pg, off = h["block_table"][b, t // P], t % P
            h["v_scales"][pg, :, off] *= np.float32(factor)
    h["v_new"] = _scaled_bf16(h["v_new"], factor)
    out, st, d = run_prefill(wl, h, starts, ctx)
    ref, ost, kp, vp = oracle_prefill(h, starts, ctx, wl.rope_theta, wl.scale)
    assert st == 0 and ost == 0
    got = out_f64(out)
    assert np.all(np.isfinite(got))
    size = np.abs(ref).max(axis=-1, keepdims=True)
    assert size.min() > 0
    assert np.all(np.abs(got - ref) <= 2e-2 * size)


@pytest.mark.parametrize("kind", ["prompts", "chunks", "drafts"])
def test_int8_key_scales_far_from_one(kind):
    """Cached key rows with scales of 1e-7 of their own (scores near zero), and
    one row per sequence with 3e4 times its scale (dequantised values past
    f16's range) that every query of the sequence is aligned with (NoPE):
    that row takes the whole softmax, the output is its value row."""
    ctx, n_new = _RANGE_CASES[kind]
    ctx = [max(c, 60) for c in ctx]
    wl, h, starts, ctx = make_case(8, 2, ctx, n_new, d=128, seed=57, theta=0.0, kv="int8")
    P = wl.page_size
    ks = h["k_scales"]
    for b in range(len(ctx)):
        big = int(ctx[b]) // 3
        for t in range(0, int(ctx[b]), 5):
            if t != big:
                pg, off = h["block_table"][b, t // P], t % P
                ks[pg, :, off] *= np.float32(1e-7)
        pg, off = h["block_table"][b, big // P], big % P
        for i in range(int(np.diff(starts)[b])):   # aligned with the row before it grows
            for hq in range(8):
                h["q"][starts[b] + i, hq] = _stored_key(h, wl, starts, ctx, b, big, hq // 4)
        ks[pg, :, off] *= np.float32(3e4)
    check(wl, h, starts, ctx)
