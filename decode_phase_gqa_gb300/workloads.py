"""Seeded synthetic inputs for one decode step of GQA attention over a paged KV cache.

This module only draws inputs: sequence lengths, page permutations, block
tables and the q / k_new / v_new / cached K/V tensors.  It computes nothing of
the decode step itself and is shared, as an input source, by the tests, the
smoke check and the benchmark.

Workload shapes follow the head layouts of the models the source pages discuss
(SmolLM3-3B in "LLM inference from smollm3.go", Qwen3-8B in "Qwen3-8B inference
engine from scratch in C++/CUDA", Llama-3.2-1B in "C17 CPU-first LLM inference
engine"); no weights are used, every value is drawn from N(0, 1).

Recipe (all configs):
  * lengths from ``numpy.random.default_rng(seed)``; positions = lengths;
  * every sequence needs ceil((L + 1) / page_size) pages (the new token
    included); the pool holds that total plus 5 % spare pages, its physical
    page ids are a seeded permutation, handed out in sequence order; unused
    block-table entries are -1;
  * tensors from ``torch.Generator(device).manual_seed(...)``: fp32 N(0, 1)
    draws cast to bf16 (round to nearest even);
  * int8 caches: each cached row (token, KV head) is an fp32 N(0, 1) draw
    stored as int8 codes with an fp32 scale max|x| / 127 (the int8 config's
    input recipe); these rows are inputs, the decode step only reads them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

# name -> shape of the workload; lengths are drawn by _draw_lengths.
CONFIGS = {
    # 1 sequence, 4 q heads / 1 KV head, d 64, 256 cached + 1 new at position
    # 256, page 16, theta 1e4, scale 1/8; the 17 pages are a seeded permutation.
    "tiny": dict(n_seq=1, n_qh=4, n_kvh=1, head_dim=64, page_size=16,
                 rope_theta=1e4, scale=1 / 8, kv_dtype="bf16", layers=1,
                 lengths=("fixed", 256), spare=0.0),
    # SmolLM3-3B-shaped layer: 16/4 heads, d 128, batch 8, L ~ U[512, 4096].
    "smollm3": dict(n_seq=8, n_qh=16, n_kvh=4, head_dim=128, page_size=16,
                    rope_theta=1e6, scale=1 / math.sqrt(128), kv_dtype="bf16",
                    layers=1, lengths=("uniform", 512, 4096), spare=0.05),
    # Qwen3-8B-shaped continuous batch: 32/8 heads, d 128, batch 64,
    # L log-uniform in [128, 8192], 36 independent layer caches per step.
    "qwen3": dict(n_seq=64, n_qh=32, n_kvh=8, head_dim=128, page_size=16,
                  rope_theta=1e6, scale=1 / math.sqrt(128), kv_dtype="bf16",
                  layers=36, lengths=("loguniform", 128, 8192), spare=0.05),
    # Llama-3.2-1B-shaped long context: 32/8 heads, d 64, batch 32, half the
    # sequences at 32768 cached tokens, the rest U[1, 2048], order shuffled.
    "llama1b": dict(n_seq=32, n_qh=32, n_kvh=8, head_dim=64, page_size=16,
                    rope_theta=5e5, scale=1 / 8, kv_dtype="bf16", layers=1,
                    lengths=("skewed", 32768, 1, 2048), spare=0.05),
    # Int8 KV cache, Qwen3-8B-shaped: 32/8 heads, d 128, batch 128,
    # L ~ U[1024, 4096], K/V int8 with per-(token, head) fp32 scales.
    "int8": dict(n_seq=128, n_qh=32, n_kvh=8, head_dim=128, page_size=16,
                 rope_theta=1e6, scale=1 / math.sqrt(128), kv_dtype="int8",
                 layers=1, lengths=("uniform", 1024, 4096), spare=0.05),
    # A large continuous batch of the Qwen3-8B shape: 512 sequences, L
    # log-uniform in [128, 8192], one layer cache (what a serving engine's
    # batch grows to; checks that throughput holds above 128 sequences).
    "qwen3_b512": dict(n_seq=512, n_qh=32, n_kvh=8, head_dim=128, page_size=16,
                       rope_theta=1e6, scale=1 / math.sqrt(128), kv_dtype="bf16",
                       layers=1, lengths=("loguniform", 128, 8192), spare=0.05),
}

# The configs in the order the benchmark configuration list states them.
CONFIG_ORDER = ["tiny", "smollm3", "qwen3", "llama1b", "int8"]
# Further shapes the benchmark times beside them.
EXTRA_CONFIGS = ["qwen3_b512"]


@dataclass
class Workload:
    name: str
    n_seq: int
    n_qh: int
    n_kvh: int
    head_dim: int
    page_size: int
    rope_theta: float
    scale: float
    kv_dtype: str
    layers: int
    seq_lens: np.ndarray          # int32 [n_seq], cached tokens before the step
    positions: np.ndarray         # int32 [n_seq], RoPE position of the new token
    block_table: np.ndarray       # int32 [n_seq, max_pages_per_seq], -1 = unused
    num_pages: int
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V the step must read: sum_b (L_b + 1) * n_kvh * d per
        tensor, times 2 (K and V); int8 adds one fp32 scale per row."""
        tokens = int((self.seq_lens.astype(np.int64) + 1).sum())
        if self.kv_dtype == "int8":
            per_row = self.head_dim + 4
        else:
            per_row = 2 * self.head_dim
        return tokens * self.n_kvh * per_row * 2


def _draw_lengths(spec, n_seq, rng):
    kind = spec[0]
    if kind == "fixed":
        return np.full(n_seq, spec[1], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(spec[1], spec[2], size=n_seq, endpoint=True)
    if kind == "loguniform":
        u = rng.uniform(math.log(spec[1]), math.log(spec[2]), size=n_seq)
        return np.floor(np.exp(u)).astype(np.int64)
    if kind == "skewed":
        n_long = n_seq // 2
        short = rng.integers(spec[2], spec[3], size=n_seq - n_long, endpoint=True)
        lens = np.concatenate([np.full(n_long, spec[1], dtype=np.int64), short])
        return lens[rng.permutation(n_seq)]
    if kind == "list":
        return np.asarray(spec[1], dtype=np.int64)
    raise ValueError(f"unknown length spec {spec!r}")


def make_workload(name: str = "custom", seed: int = 0, *, lengths=None,
                  max_len: Optional[int] = None, spare: Optional[float] = None,
                  **shape) -> Workload:
    """Draw lengths, pool size and block table for a named config or a custom shape.

    ``lengths`` may be a length spec tuple or an explicit list; ``max_len`` sets
    the block-table width (default: the config's largest possible length).
    """
    cfg = dict(CONFIGS.get(name, {}))
    cfg.update(shape)
    if lengths is not None:
        cfg["lengths"] = lengths if isinstance(lengths, tuple) else ("list", list(lengths))
    if spare is not None:
        cfg["spare"] = spare
    for key, default in (("page_size", 16), ("kv_dtype", "bf16"), ("layers", 1),
                         ("spare", 0.05), ("rope_theta", 1e4)):
        cfg.setdefault(key, default)
    cfg.setdefault("scale", 1 / math.sqrt(cfg["head_dim"]))
    rng = np.random.default_rng(seed)
    lens = _draw_lengths(cfg["lengths"], cfg["n_seq"], rng)
    P = cfg["page_size"]
    spec = cfg["lengths"]
    if max_len is None:
        top = {"fixed": lambda s: s[1], "uniform": lambda s: s[2],
               "loguniform": lambda s: s[2], "skewed": lambda s: max(s[1], s[3]),
               "list": lambda s: max(s[1]) if len(s[1]) else 0}[spec[0]](spec)
        max_len = int(top)
    mpps = max(1, -(-(max_len + 1) // P))
    pages_needed = [-(-(int(L) + 1) // P) for L in lens]
    total = int(sum(pages_needed))
    num_pages = max(1, total + int(math.ceil(cfg["spare"] * total)))
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((cfg["n_seq"], mpps), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(pages_needed):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    seq_lens = lens.astype(np.int32)
    return Workload(name=name, n_seq=cfg["n_seq"], n_qh=cfg["n_qh"], n_kvh=cfg["n_kvh"],
                    head_dim=cfg["head_dim"], page_size=P, rope_theta=float(cfg["rope_theta"]),
                    scale=float(cfg["scale"]), kv_dtype=cfg["kv_dtype"], layers=cfg["layers"],
                    seq_lens=seq_lens, positions=seq_lens.copy(), block_table=bt,
                    num_pages=num_pages, seed=seed)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _int8_rows(x: torch.Tensor):
    """Input synthesis of an int8 cache: fp32 rows -> (codes, per-row scales)."""
    a = x.abs().amax(dim=-1)
    sc = a / 127.0
    safe = torch.where(sc > 0, sc, torch.ones_like(sc))
    codes = torch.round(x / safe.unsqueeze(-1)).clamp_(-127, 127)
    codes = torch.where(sc.unsqueeze(-1) > 0, codes, torch.zeros_like(codes))
    return codes.to(torch.int8), sc.contiguous()


def make_tensors(wl: Workload, layer: int = 0, device="cpu", chunk_rows: int = 1 << 22):
    """Draw q, k_new, v_new and one layer's K/V pool for a workload.

    Returns a dict of torch tensors on ``device``: q [B, Hq, d], k_new and
    v_new [B, Hk, d] (bf16), k_pages / v_pages [num_pages, Hk, P, d] (bf16 or
    int8) and k_scales / v_scales [num_pages, Hk, P] fp32 (int8 only, else None).
    """
    device = torch.device(device)
    g = _gen(device, 1_000_003 * wl.seed + 7919 * layer + 17)
    B, Hq, Hk, d, P = wl.n_seq, wl.n_qh, wl.n_kvh, wl.head_dim, wl.page_size
    out = {
        "q": _normal((B, Hq, d), g, device).to(torch.bfloat16),
        "k_new": _normal((B, Hk, d), g, device).to(torch.bfloat16),
        "v_new": _normal((B, Hk, d), g, device).to(torch.bfloat16),
    }
    pool_shape = (wl.num_pages, Hk, P, d)
    rows = wl.num_pages * Hk * P
    for name in ("k", "v"):
        if wl.kv_dtype == "bf16":
            pool = torch.empty(pool_shape, dtype=torch.bfloat16, device=device)
            flat = pool.view(rows, d)
            for r0 in range(0, rows, chunk_rows):
                r1 = min(rows, r0 + chunk_rows)
                flat[r0:r1] = _normal((r1 - r0, d), g, device).to(torch.bfloat16)
            out[f"{name}_pages"] = pool
            out[f"{name}_scales"] = None
        else:
            pool = torch.empty(pool_shape, dtype=torch.int8, device=device)
            scales = torch.empty((wl.num_pages, Hk, P), dtype=torch.float32, device=device)
            flat, sflat = pool.view(rows, d), scales.view(rows)
            for r0 in range(0, rows, chunk_rows):
                r1 = min(rows, r0 + chunk_rows)
                codes, sc = _int8_rows(_normal((r1 - r0, d), g, device))
                flat[r0:r1] = codes
                sflat[r0:r1] = sc
            out[f"{name}_pages"] = pool
            out[f"{name}_scales"] = scales
    return out


def with_lengths(wl: Workload, seq_lens, positions=None) -> Workload:
    """Copy of a workload with other lengths/positions (same table and pool)."""
    sl = np.asarray(seq_lens, dtype=np.int32)
    pos = sl.copy() if positions is None else np.asarray(positions, dtype=np.int32)
    return replace(wl, seq_lens=sl, positions=pos)
