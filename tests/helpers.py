"""Shared test plumbing: turn generated torch tensors into oracle-ready numpy arrays."""
import numpy as np
import torch

from decode_phase_gqa_gb300 import workloads as W


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns; other dtypes -> numpy as is."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def host_inputs(wl: W.Workload, layer: int = 0, tensors=None):
    """Numpy copies (bf16 as uint16) of one layer's inputs plus the workload metadata."""
    t = tensors if tensors is not None else W.make_tensors(wl, layer=layer, device="cpu")
    h = {k: (None if v is None else bits(v)) for k, v in t.items()}
    h["block_table"] = wl.block_table.copy()
    h["seq_lens"] = wl.seq_lens.copy()
    h["positions"] = wl.positions.copy()
    return h


def oracle_decode(wl: W.Workload, h, seq_mask=None, n_threads=0):
    """Run the oracle's decode step on copies of the host inputs.

    Returns (out float64, status, k_pages_after, v_pages_after, k_scales, v_scales).
    """
    import oracle
    kp, vp = h["k_pages"].copy(), h["v_pages"].copy()
    ks = None if h["k_scales"] is None else h["k_scales"].copy()
    vs = None if h["v_scales"] is None else h["v_scales"].copy()
    out, st = oracle.decode(h["q"], h["k_new"], h["v_new"], kp, vp, h["block_table"],
                            h["seq_lens"], h["positions"], wl.rope_theta, wl.scale,
                            ks, vs, seq_mask=seq_mask, n_threads=n_threads)
    return out, st, kp, vp, ks, vs


def oracle_prefill(h, seq_starts, ctx_lens, rope_theta, scale, seqs=None):
    """The oracle's chunked prefill, as the decode steps it is made of: step i
    appends new token i of every sequence that has one (slot and RoPE position
    ctx + i) and attends over the cache up to it, which is the causal
    attention over the cache and the earlier new tokens.

    h: q [T, Hq, d], k_new / v_new [T, Hk, d] (bf16 bits), k_pages / v_pages,
    block_table [B, max_pages].  `seqs`: the sequences to run (default all).
    Returns (out float64 [T, Hq, d], NaN for rows not run; status; the pools
    after the appends); int8 caches: h["k_scales"] / h["v_scales"] are
    updated copies too, returned as oracle_prefill.scales.
    """
    import oracle
    kp, vp = h["k_pages"].copy(), h["v_pages"].copy()
    ks = None if h.get("k_scales") is None else h["k_scales"].copy()
    vs = None if h.get("v_scales") is None else h["v_scales"].copy()
    starts = np.asarray(seq_starts, np.int64)
    ctx = np.asarray(ctx_lens, np.int64)
    n_new = np.diff(starts)
    chosen = np.arange(len(ctx)) if seqs is None else np.asarray(seqs)
    out = np.full(h["q"].shape, np.nan)
    st = 0
    for i in range(int(n_new[chosen].max(initial=0))):
        act = chosen[n_new[chosen] > i]
        rows = starts[act] + i
        o, s = oracle.decode(np.ascontiguousarray(h["q"][rows]), np.ascontiguousarray(h["k_new"][rows]),
                             np.ascontiguousarray(h["v_new"][rows]), kp, vp,
                             np.ascontiguousarray(h["block_table"][act]),
                             (ctx[act] + i).astype(np.int32), (ctx[act] + i).astype(np.int32),
                             rope_theta, scale, ks, vs)
        out[rows] = o
        st |= s
    oracle_prefill.scales = (ks, vs)
    return out, st, kp, vp
