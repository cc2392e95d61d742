"""Independent float64 formulas used to pin the oracle (tests only).

Written in a different style from the C oracle on purpose: RoPE as a complex
multiplication, the paged gather as numpy fancy indexing, softmax from scipy.
A plausible slip in either implementation (swapped pair, wrong sign, dropped
token, wrong head mapping) makes the two disagree.
"""
import math

import numpy as np
from scipy.special import softmax


def bf16_bits_to_f64(u16):
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def rope_complex(x, pos, theta):
    """Half-split RoPE as z_i = x_i + i*x_{i+h} times exp(i*pos*theta^(-2i/d))."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    if theta <= 0:
        return x.copy()
    freq = np.power(float(theta), -np.arange(h, dtype=np.float64) * 2.0 / d)
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * float(pos) * freq)
    return np.concatenate([z.real, z.imag], axis=-1)


def gather_rows(pool, scales, block_table, b, L, page, kv_int8):
    """Rows 0..L of sequence b as float64 [L+1, Hk, d] via the block table."""
    t = np.arange(L + 1)
    pages = block_table[b, t // page]
    offs = t % page
    rows = pool[pages, :, offs, :]                       # [L+1, Hk, d]
    if kv_int8:
        return rows.astype(np.float64) * scales[pages, :, offs].astype(np.float64)[..., None]
    return bf16_bits_to_f64(rows)


def attend_reference(q_bits, k_rows, v_rows, pos, theta, scale, n_kvh):
    """out[h] = softmax(scale * rot(q_h) . K_{h//g}) @ V_{h//g}, float64."""
    n_qh, d = q_bits.shape
    g = n_qh // n_kvh
    qh = rope_complex(bf16_bits_to_f64(q_bits), pos, theta)      # [Hq, d]
    out = np.empty((n_qh, d))
    for h in range(n_qh):
        j = h // g
        s = scale * (k_rows[:, j, :] @ qh[h])
        out[h] = softmax(s) @ v_rows[:, j, :]
    return out


def store_key_f32(x_bits, pos, theta):
    """The appended key's fp32 storage recipe, replayed independently.

    c and s are the double cos/sin of the double angle pos * theta^(-2i/d)
    (Python's math module, scalar by scalar), each rounded to fp32; every
    product and every sum is then a separate numpy float32 operation, so
    nothing is fused.  theta <= 0 keeps the key as given.
    """
    x = bf16_bits_to_f64(x_bits).astype(np.float32)
    d = x.shape[-1]
    h = d // 2
    if theta <= 0:
        return x.copy()
    c = np.empty(h, np.float32)
    s = np.empty(h, np.float32)
    for i in range(h):
        phi = float(pos) * math.pow(float(theta), -(2.0 * i) / d)
        c[i] = np.float32(math.cos(phi))
        s[i] = np.float32(math.sin(phi))
    lo, hi = x[:h], x[h:]
    first = np.subtract(np.multiply(lo, c, dtype=np.float32),
                        np.multiply(hi, s, dtype=np.float32), dtype=np.float32)
    second = np.add(np.multiply(hi, c, dtype=np.float32),
                    np.multiply(lo, s, dtype=np.float32), dtype=np.float32)
    return np.concatenate([first, second])


def quant_row_int8(x):
    """Symmetric int8 codes and fp32 scale of one fp32 row: scale =
    fl32(max|x| / 127), code = clip(rint_half_even(fl32(x / scale)), -127, 127);
    a zero row gives scale 0 and zero codes."""
    x = np.asarray(x, np.float32)
    amax = np.float32(np.max(np.abs(x)))
    if amax == 0:
        return np.zeros(x.shape, np.int8), np.float32(0.0)
    sc = np.float32(amax / np.float32(127.0))
    t = np.divide(x, sc, dtype=np.float32)
    return np.clip(np.rint(t), -127, 127).astype(np.int8), sc
