"""Plain, slow fp64 CPU oracle for single-token MLA decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY.  This module exists to check the CUDA library.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline``
and ``--impl reference`` legs) may import it.  The product path never imports
it, and it imports nothing from the product: it shares no kernels, headers,
helpers, tables or constants with the CUDA path.

Everything is numpy in float64 unless a step is defined in another precision
(bf16 storage of the cache, the fp32 INT8 quantiser), in which case that
precision is emulated exactly.  Each function names the passage it follows:

  [P1] "Beyond the Attention Bottleneck: How Kimi and DeepSeek-V2 Architected
       Million-Token Context Windows"
  [P2] "KV Cache Optimization: Scaling to Million-Token Contexts"
  [P3] "DeepSeek's Config Says 16 KV Heads, Its Cache Holds a Ninth of That:
       Seven Ways LLMs Handle Attention, and Which Models Use Each"
  [P4] "The Architecture of Memory: KV Cache Dynamics, Optimization, and the
       Future of LLM Inference"

The oracle's definition of the decode is the UN-absorbed one: per head, the
content key and the value of every cached token are up-projected explicitly
from the latent ([P1] "Down-Projection and Up-Projection Mechanics"), the
decoupled RoPE key is concatenated ([P1] "The RoPE Compatibility Problem"),
and ordinary softmax attention is taken.  The absorbed form ([P4] "The Weight
Absorption Trick") is implemented separately and used only as a cross-check.

Pins (see tests/test_oracle.py): absorbed == un-absorbed, closed forms (one
token, equal rows, zero query), a library special case (torch SDPA in fp64 on
explicitly expanded K/V), softmax normalisation, split/combine invariance,
page-permutation invariance, RoPE invariants, INT8 error bound and worked
examples, the FP8 E4M3 format's closed forms, brute-force nearest encoding
and worked ties, the 1-byte caches' append -> read-back round trip within
each format's rounding bound (with planted layout mistakes it must catch),
multi-token decode against causal SDPA, sparse decode against masked SDPA
(out-of-range entries skipped), chunked prefill against causal SDPA and
chunk-split invariance, and the pages' own cache-size figures
(tests/golden/).

Readings where the pages are silent:
  * the 576-wide row is [latent 0..511 | RoPE key 512..575];
  * k_pe is rotated once, at append time, by the RoFormer pair rotation of
    (x[2i], x[2i+1]) with angle pos * theta**(-2i/64); the query's RoPE part
    arrives already rotated.  The pairing convention is a reading, not a
    value the pages fix: parity of the pairing is unpinned beyond the RoPE
    invariants;
  * INT8: per token, over all 576 values, asymmetric min/max with the range
    widened to include 0, fp32 arithmetic in a fixed order (see
    ``quantize_tokens_int8``).  The exact recipe is a reading: parity of the
    recipe is pinned only by the error bound and worked examples.
  * a prefill chunk is the last `chunk` tokens of each sequence, appended
    before its queries attend (the multi-token reading with chunk for q_len);
  * FP8: the E4M3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, subnormals, no infinities, S.1111.111 = NaN, largest finite 448),
    one fp32 scale per token from the row's largest magnitude, codes by
    round-to-nearest-even with saturation (see ``quantize_tokens_fp8``).  The
    pages name low-bit caches with per-token scaling but not this format: the
    format comes from its own definition, pinned by its closed-form values,
    brute-force nearest search and worked ties.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

LATENT_DIM = 512  # d_c: [P3] section 5 (kv_lora_rank: 512)
ROPE_DIM = 64     # d_rope: [P3] section 5 (qk_rope_head_dim: 64); [P4] "Decoupled RoPE"
ROW_DIM = LATENT_DIM + ROPE_DIM  # 576 numbers per token per layer: [P3] opening, section 5

# --------------------------------------------------------------------------- #
# bf16 storage (the cache and the weights are stored in a 16-bit format)      #
# --------------------------------------------------------------------------- #


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even, in one step.

    bf16 keeps 8 significant bits and fp32's exponent range.  For a finite x
    with frexp(x) = (m, e), the spacing of bf16 numbers around x is
    2**(e-8) (2**-133 below the normal range), so x is rounded to an integer
    multiple of that spacing with rint (which breaks ties to even).  Values
    that overflow the bf16 range become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)
    e_eff = np.maximum(e, -125)
    q = np.rint(np.ldexp(xf, 8 - e_eff))
    y = np.ldexp(q, e_eff - 8)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    y = np.where(np.abs(y) > bf16_max, np.copysign(np.inf, y), y)
    return np.where(finite, y, x)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of round_to_bf16(x)."""
    y = round_to_bf16(x).astype(np.float32)  # exact: bf16 values are fp32 values
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------- #
# Cache footprint ([P3] opening section; [P4] "DeepSeek's MLA")               #
# --------------------------------------------------------------------------- #


def latent_cache_bytes_per_token(layers: int, latent_dim: int = LATENT_DIM,
                                 rope_dim: int = ROPE_DIM, elem_bytes: int = 2,
                                 side_bytes_per_row: int = 0) -> int:
    """Bytes one token occupies in an MLA cache over ``layers`` layers.

    One row of latent_dim + rope_dim numbers per token per layer ([P3] opening:
    "one compressed 576-number vector per token per layer"), each of
    ``elem_bytes``; ``side_bytes_per_row`` adds per-row metadata such as the
    INT8 scale and zero point.
    """
    return layers * ((latent_dim + rope_dim) * elem_bytes + side_bytes_per_row)


def per_head_cache_bytes_per_token(layers: int, kv_heads: int, key_dim: int,
                                   value_dim: int, elem_bytes: int = 2) -> int:
    """Bytes per token if every head stored its own key and value ([P3] opening)."""
    return layers * kv_heads * (key_dim + value_dim) * elem_bytes


# --------------------------------------------------------------------------- #
# Decoupled RoPE ([P1] "The RoPE Compatibility Problem"; [P4] "Decoupled RoPE")#
# --------------------------------------------------------------------------- #


def rope_inv_freq(rope_dim: int = ROPE_DIM, theta: float = 10000.0) -> np.ndarray:
    """Angular frequency of each rotated pair i: theta ** (-2i / rope_dim)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -(2.0 * i) / rope_dim)


def rope_rotate(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each pair (x[2i], x[2i+1]) of the last axis by positions * inv_freq[i].

    The rotation depends on the position, which is why it cannot be folded into
    a fixed up-projection ([P4] "Decoupled RoPE").  theta <= 0 means "no
    rotation" (the caller stores k_pe as given).  fp64 throughout.
    """
    x = np.asarray(x, dtype=np.float64)
    if theta <= 0:
        return x.copy()
    d = x.shape[-1]
    pos = np.asarray(positions, dtype=np.float64)
    ang = pos[..., None] * rope_inv_freq(d, theta)   # positions have x's leading shape
    cos, sin = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * cos - x1 * sin
    out[..., 1::2] = x0 * sin + x1 * cos
    return out


# --------------------------------------------------------------------------- #
# INT8 per-token asymmetric quantisation ([P2] section 3; [P4] KIVI section)  #
# --------------------------------------------------------------------------- #


def quantize_tokens_int8(rows: np.ndarray):
    """Quantise each row (one token's 576 values) to int8 with its own scale and zero point.

    [P2] section 3 quantises with per-row min and max; [P4] ("The 2-Bit
    Quantization Barrier and KIVI") quantises per token the data that is mixed
    across tokens, which the latent row is.  Steps, all in IEEE fp32 with
    round-to-nearest-even and no fused multiply-add, in this order:

        lo = min(min(x), 0)            hi = max(max(x), 0)
        s  = (hi - lo) / 255           (s = 1 if that is 0)
        zp = clamp(rint(-128 - lo / s), -128, 127)
        q  = clamp(rint(x / s) + zp, -128, 127)

    Widening the range to include 0 makes 0 representable exactly.  Returns
    (codes int8 [N, D], scale fp32 [N], zero_point fp32 [N]).
    """
    x = np.asarray(rows, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    f = np.float32
    lo = np.minimum(x.min(axis=1), f(0)).astype(np.float32)
    hi = np.maximum(x.max(axis=1), f(0)).astype(np.float32)
    s = ((hi - lo) / f(255)).astype(np.float32)
    s = np.where(s == f(0), f(1), s).astype(np.float32)
    zp = np.rint((f(-128) - (lo / s).astype(np.float32)).astype(np.float32)).astype(np.float32)
    zp = np.clip(zp, f(-128), f(127)).astype(np.float32)
    q = np.rint((x / s[:, None]).astype(np.float32)).astype(np.float32)
    q = np.clip((q + zp[:, None]).astype(np.float32), f(-128), f(127))
    return q.astype(np.int8), s, zp


def dequantize_tokens_int8(codes: np.ndarray, scale: np.ndarray, zero_point: np.ndarray) -> np.ndarray:
    """x_hat = scale * (code - zero_point), evaluated in fp64."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scale, dtype=np.float64)[..., None]
    z = np.asarray(zero_point, dtype=np.float64)[..., None]
    return s * (c - z)


# --------------------------------------------------------------------------- #
# FP8 (E4M3) per-token scaled quantisation ([P2] section 3 and [P4] KIVI       #
# section: low-bit caches, scaled per token for the data mixed across tokens) #
# --------------------------------------------------------------------------- #

E4M3_MAX = 448.0  # largest finite E4M3 magnitude: (1 + 6/8) * 2**(15 - 7)


def e4m3_value(codes) -> np.ndarray:
    """Value of each FP8 E4M3 code (uint8), from the format's definition.

    Bit 7 is the sign, bits 6..3 the exponent e (bias 7), bits 2..0 the
    mantissa m.  e = 0 is subnormal: (m / 8) * 2**-6; otherwise
    (1 + m / 8) * 2**(e - 7).  The code with e = 15 and m = 7 is NaN (the
    format has no infinities), so the largest finite magnitude is
    1.75 * 2**8 = 448.  Returns fp64 (every E4M3 value is exact there).
    """
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


def e4m3_encode(x) -> np.ndarray:
    """Nearest finite E4M3 code to each value (uint8).

    Round to nearest, ties to the code with the even mantissa; magnitudes at
    or beyond 448 saturate to 448 (the format has no infinity, and the code
    above 448 is NaN); the sign is kept, so -0 and negative values that
    round to zero give 0x80.  The search runs over the table of the 127
    non-negative finite codes (their magnitudes rise with the code).
    """
    v = np.asarray(x, dtype=np.float64)
    table = e4m3_value(np.arange(0x7F))          # codes 0x00 .. 0x7E, ascending magnitudes
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, 0x7E)  # first code with magnitude >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = table[hi] - a
    d_lo = a - table[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.int64)
    code = np.where(np.signbit(v), code | 0x80, code)
    return code.astype(np.uint8)


def quantize_tokens_fp8(rows: np.ndarray):
    """Quantise each row (one token's 576 values) to E4M3 codes with one scale.

    Per token, as for the INT8 cache, but symmetric: E4M3 already spaces its
    values geometrically, so one scale that maps the row's largest magnitude
    onto the format's largest finite value suffices.  In IEEE fp32 with
    round-to-nearest-even, in this order:

        a = max |x|          s = a / 448          (s = 1 if that is 0)
        code = E4M3 nearest (ties to even, saturating) of  x / s

    Returns (codes uint8 [N, D], scale fp32 [N]).
    """
    x = np.asarray(rows, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    f = np.float32
    a = np.abs(x).max(axis=1).astype(np.float32)
    s = (a / f(E4M3_MAX)).astype(np.float32)
    s = np.where(s == f(0), f(1), s).astype(np.float32)
    y = (x / s[:, None]).astype(np.float32)
    return e4m3_encode(y), s


def dequantize_tokens_fp8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x_hat = scale * value(code), evaluated in fp64."""
    return np.asarray(scale, dtype=np.float64)[..., None] * e4m3_value(codes)


# --------------------------------------------------------------------------- #
# Paged cache ([P2] section 7 "Paged Attention"; [P4] "PagedAttention")       #
# --------------------------------------------------------------------------- #


def page_slot(block_table: np.ndarray, seq: int, pos: int, page_size: int):
    """Physical page and offset of token ``pos`` of sequence ``seq``.

    Logical page j of a sequence holds its tokens [j*P, (j+1)*P); the page
    table maps logical page -> physical page.
    """
    return int(block_table[seq, pos // page_size]), int(pos % page_size)


def append_tokens(cache: np.ndarray, scale_zero: np.ndarray | None, block_table: np.ndarray,
                  seq_ids: Sequence[int], positions: Sequence[int], c_kv_bits: np.ndarray,
                  k_pe_bits: np.ndarray, rope_theta: float, page_size: int, int8: bool, *,
                  fp8: bool = False) -> None:
    """Write new tokens into the paged cache, in place ([P4] decode phase: "the
    new Key and Value are appended").

    cache: bf16 bit patterns uint16 [num_pages, P, 576]; int8 codes with
    scale_zero fp32 [num_pages, P, 2] holding (scale, zero_point); or (fp8)
    E4M3 codes uint8 with scale_zero fp32 [num_pages, P] holding the scale.
    c_kv_bits / k_pe_bits: bf16 bit patterns of the new latent [N, 512] and
    RoPE key [N, 64].  The RoPE key is rotated by the token's position in fp64
    and rounded to bf16; the stored row is [latent | rotated key].
    """
    c = bf16_bits_to_f64(c_kv_bits)
    kp = bf16_bits_to_f64(k_pe_bits)
    for i, (b, pos) in enumerate(zip(seq_ids, positions)):
        page, off = page_slot(block_table, int(b), int(pos), page_size)
        k_rot = round_to_bf16(rope_rotate(kp[i][None, :], np.array([pos]), rope_theta))[0]
        row = np.concatenate([c[i], k_rot])
        if int8:
            q, s, z = quantize_tokens_int8(row.astype(np.float32))
            cache[page, off] = q[0]
            scale_zero[page, off, 0] = s[0]
            scale_zero[page, off, 1] = z[0]
        elif fp8:
            q, s = quantize_tokens_fp8(row.astype(np.float32))
            cache[page, off] = q[0]
            scale_zero[page, off] = s[0]
        else:
            cache[page, off] = f64_to_bf16_bits(row)


def gather_rows(cache: np.ndarray, scale_zero: np.ndarray | None, block_table: np.ndarray,
                seq: int, length: int, page_size: int, int8: bool, *, fp8: bool = False) -> np.ndarray:
    """The ``length`` cached rows of sequence ``seq`` in logical order, as fp64 [L, 576]."""
    t = np.arange(length)
    pages = block_table[seq, t // page_size].astype(np.int64)
    offs = t % page_size
    if fp8:
        return dequantize_tokens_fp8(cache[pages, offs], scale_zero[pages, offs])
    if int8:
        return dequantize_tokens_int8(cache[pages, offs], scale_zero[pages, offs, 0],
                                      scale_zero[pages, offs, 1])
    return bf16_bits_to_f64(cache[pages, offs])


# --------------------------------------------------------------------------- #
# Attention for one (sequence, head)                                          #
# --------------------------------------------------------------------------- #


def softmax_with_lse(s: np.ndarray):
    """p = exp(s - max) / sum, lse = max + ln(sum); empty input -> (empty, -inf)."""
    if s.size == 0:
        return s.copy(), -math.inf
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    return e / z, float(m + math.log(z))


def attend_unabsorbed(q_nope: np.ndarray, q_pe: np.ndarray, rows: np.ndarray,
                      W_UK: np.ndarray, W_UV: np.ndarray, scale: float):
    """One head's decode attention, written the un-absorbed way (the oracle's definition).

    For every cached token t ([P1] "Down-Projection and Up-Projection
    Mechanics"): content key K_t = W^UK c_t and value V_t = W^UV c_t, with
    this head's W^UK, W^UV in R^{128 x 512}.  The score adds the content and
    the positional dot products ([P1] "The RoPE Compatibility Problem"):
    s_t = scale * (q_nope . K_t + q_pe . k_pe_t).  Then p = softmax(s),
    o = sum_t p_t V_t and lse = ln sum_t exp(s_t).

    Returns (o [128], lse, p [L]).  L = 0 gives o = 0, lse = -inf.
    """
    c = rows[:, :LATENT_DIM]
    k_pe = rows[:, LATENT_DIM:]
    K = c @ np.asarray(W_UK, np.float64).T   # [L, 128]: K_t = W^UK c_t
    V = c @ np.asarray(W_UV, np.float64).T   # [L, 128]: V_t = W^UV c_t
    s = scale * (K @ np.asarray(q_nope, np.float64) + k_pe @ np.asarray(q_pe, np.float64))
    p, lse = softmax_with_lse(s)
    o = p @ V if rows.shape[0] else np.zeros(W_UV.shape[0])
    return o, lse, p


def attend_absorbed(q_nope: np.ndarray, q_pe: np.ndarray, rows: np.ndarray,
                    W_UK: np.ndarray, W_UV: np.ndarray, scale: float):
    """The same head computed in the absorbed form (cross-check only).

    [P4] "The Weight Absorption Trick" / [P3] section 5: by associativity the
    key up-projection moves onto the query, q_lat = W^UK^T q_nope, and the
    score is taken against the latent directly; the value up-projection moves
    after the weighted sum, o = W^UV (sum_t p_t c_t).
    Returns (o [128], lse, o_lat [512]).
    """
    c = rows[:, :LATENT_DIM]
    k_pe = rows[:, LATENT_DIM:]
    q_lat = np.asarray(W_UK, np.float64).T @ np.asarray(q_nope, np.float64)   # [512]
    s = scale * (c @ q_lat + k_pe @ np.asarray(q_pe, np.float64))
    p, lse = softmax_with_lse(s)
    o_lat = p @ c if rows.shape[0] else np.zeros(LATENT_DIM)
    return np.asarray(W_UV, np.float64) @ o_lat, lse, o_lat


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge partial results of disjoint token chunks by log-sum-exp ([P4]
    "Flash-Decoding and FlashInfer").

    Each part s holds its output normalised within the chunk and its chunk
    lse_s (natural log; -inf for an empty chunk).  lse = ln sum_s exp(lse_s),
    o = sum_s exp(lse_s - lse) o_s.  All parts empty -> (0, -inf).
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    if lse_parts.size == 0 or np.all(np.isneginf(lse_parts)):
        return np.zeros(o_parts.shape[1:]), -math.inf
    m = lse_parts.max()
    w = np.exp(lse_parts - m)
    z = w.sum()
    return np.tensordot(w / z, o_parts, axes=(0, 0)), float(m + math.log(z))


def attend_split(q_nope, q_pe, rows, W_UK, W_UV, scale, bounds: Iterable[int]):
    """Split the tokens at ``bounds`` into chunks, attend each chunk on its
    own, and merge the chunks' latent results with ``combine_partials``
    (Flash-Decoding, [P4]).  Returns (o [128], lse)."""
    edges = [0] + sorted(int(b) for b in bounds) + [rows.shape[0]]
    parts, lses = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        _, lse, o_lat = attend_absorbed(q_nope, q_pe, rows[a:b], W_UK, W_UV, scale)
        parts.append(o_lat)
        lses.append(lse)
    o_lat, lse = combine_partials(np.stack(parts), np.array(lses))
    return np.asarray(W_UV, np.float64) @ o_lat, lse


# --------------------------------------------------------------------------- #
# Whole decode step over a batch                                              #
# --------------------------------------------------------------------------- #


def decode(q_nope: np.ndarray, q_pe: np.ndarray, cache: np.ndarray, scale_zero: np.ndarray | None,
           block_table: np.ndarray, seq_lens: Sequence[int], W_UK: np.ndarray, W_UV: np.ndarray,
           scale: float, page_size: int, int8: bool, pairs=None, absorbed: bool = False, *,
           fp8: bool = False):
    """Decode attention for a batch: for each requested (b, h) pair, read the
    sequence's rows through its page table and attend.

    q_nope [B, H, 128], q_pe [B, H, 64] (already rotated), W_UK/W_UV
    [H, 128, 512] as float arrays (exact bf16 values).  ``pairs`` limits the
    work to a list of (b, h); others are left NaN.  ``absorbed`` selects the
    cross-check form.  Returns (out [B, H, 128], lse [B, H]) in fp64.
    """
    B, H = q_nope.shape[0], q_nope.shape[1]
    out = np.full((B, H, W_UV.shape[1]), np.nan)
    lse = np.full((B, H), np.nan)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    by_seq: dict[int, list[int]] = {}
    for b, h in pairs:
        by_seq.setdefault(int(b), []).append(int(h))
    fn = attend_absorbed if absorbed else attend_unabsorbed
    for b, heads in by_seq.items():
        rows = gather_rows(cache, scale_zero, block_table, b, int(seq_lens[b]), page_size, int8, fp8=fp8)
        for h in heads:
            o, l, _ = fn(q_nope[b, h], q_pe[b, h], rows, W_UK[h], W_UV[h], scale)
            out[b, h] = o
            lse[b, h] = l
    return out, lse


def decode_multi_token(q_nope: np.ndarray, q_pe: np.ndarray, cache: np.ndarray, scale_zero: np.ndarray | None,
                       block_table: np.ndarray, seq_lens: Sequence[int], W_UK: np.ndarray, W_UV: np.ndarray,
                       scale: float, page_size: int, int8: bool, triples=None, absorbed: bool = False, *,
                       fp8: bool = False):
    """Several new tokens of each sequence decoded in one pass: the
    verification read of speculative decoding ([P4] "Speculative Decoding:
    Amortizing the Memory Fetch": all drafted tokens are checked in one
    forward pass that reads the cache once), causal among the new tokens
    ([P4] "Tree Attention Verification": the history is attended densely and
    each new token sees only the new tokens before it -- a chain here).

    The T new tokens of sequence b are the last T of its L_b cached tokens
    (appended before the call): query token t sits at position L_b - T + t and
    attends to positions 0 .. L_b - T + t, itself included; a query whose
    position is below 0 attends to nothing (o = 0, lse = -inf).

    q_nope [B, T, H, 128], q_pe [B, T, H, 64] (each rotated for its own
    position).  ``triples`` limits the work to a list of (b, t, h); others are
    left NaN.  Returns (out [B, T, H, 128], lse [B, T, H]) in fp64.
    """
    B, T, H = q_nope.shape[0], q_nope.shape[1], q_nope.shape[2]
    out = np.full((B, T, H, W_UV.shape[1]), np.nan)
    lse = np.full((B, T, H), np.nan)
    if triples is None:
        triples = [(b, t, h) for b in range(B) for t in range(T) for h in range(H)]
    by_seq: dict[int, list[tuple[int, int]]] = {}
    for b, t, h in triples:
        by_seq.setdefault(int(b), []).append((int(t), int(h)))
    fn = attend_absorbed if absorbed else attend_unabsorbed
    for b, th in by_seq.items():
        L = int(seq_lens[b])
        rows = gather_rows(cache, scale_zero, block_table, b, L, page_size, int8, fp8=fp8)
        for t, h in th:
            visible = max(0, L - T + t + 1)
            o, l, _ = fn(q_nope[b, t, h], q_pe[b, t, h], rows[:visible], W_UK[h], W_UV[h], scale)
            out[b, t, h] = o
            lse[b, t, h] = l
    return out, lse


def prefill_chunk(cache: np.ndarray, scale_zero: np.ndarray | None, block_table: np.ndarray,
                  seq_lens: Sequence[int], c_kv_bits: np.ndarray, k_pe_bits: np.ndarray, rope_theta: float,
                  q_nope: np.ndarray, q_pe: np.ndarray, W_UK: np.ndarray, W_UV: np.ndarray, scale: float,
                  page_size: int, int8: bool, triples=None, absorbed: bool = False, *, fp8: bool = False):
    """One chunk of chunked prefill ([P4] "The Prefill Phase: Compute-Bound
    Parallelism": the prompt's tokens are processed together and their
    key/value state is written to the cache, which decode then reads; a long
    prompt goes in chunks, each attending to the cache the chunks before it
    wrote).

    Sequence b's chunk is the T tokens at positions L_b - T .. L_b - 1, L_b =
    seq_lens[b] counting the chunk.  First every chunk token's row is
    appended (``append_tokens``, in place on ``cache``; a position below 0,
    past the page table, or on a page-table entry below 0 is skipped), then
    query token t attends to positions 0 .. L_b - T + t
    (``decode_multi_token``: the history and the chunk's tokens up to itself).

    c_kv_bits [B, T, 512], k_pe_bits [B, T, 64] bf16 bit patterns; q_nope
    [B, T, H, 128], q_pe [B, T, H, 64].  Returns (out [B, T, H, 128],
    lse [B, T, H]); ``triples`` limits the attention to a list of (b, t, h).
    """
    B, T = q_nope.shape[0], q_nope.shape[1]
    for b in range(B):
        L = int(seq_lens[b])
        ts = [t for t in range(T) if 0 <= L - T + t < block_table.shape[1] * page_size
              and block_table[b, (L - T + t) // page_size] >= 0]
        if ts:
            append_tokens(cache, scale_zero, block_table, [b] * len(ts), [L - T + t for t in ts],
                          c_kv_bits[b, ts], k_pe_bits[b, ts], rope_theta, page_size, int8, fp8=fp8)
    return decode_multi_token(q_nope, q_pe, cache, scale_zero, block_table, seq_lens, W_UK, W_UV, scale,
                              page_size, int8, triples=triples, absorbed=absorbed, fp8=fp8)


def decode_sparse(q_nope: np.ndarray, q_pe: np.ndarray, cache: np.ndarray, scale_zero: np.ndarray | None,
                  block_table: np.ndarray, seq_lens: Sequence[int], token_indices: np.ndarray, W_UK: np.ndarray,
                  W_UV: np.ndarray, scale: float, page_size: int, int8: bool, pairs=None, absorbed: bool = False, *,
                  fp8: bool = False):
    """Sparse decode over a given selection of cached tokens ([P3] section 6,
    "Sparse attention: keep every token, read only some": the full cache is
    kept and each new token attends only to the top-k tokens an indexer
    picked; the indexer itself is not part of this path).

    token_indices [B, k] int: positions in sequence b's cache; -1 entries are
    padding and are skipped.  The attention of (b, h) runs over the rows at
    the listed positions, in list order, each listed entry once.  The page
    does not say what a position outside the sequence means; the reading
    taken is that such an entry (below -1, or at or past seq_lens[b]) selects
    nothing and is skipped like padding.
    Returns (out [B, H, 128], lse [B, H]) in fp64; ``pairs`` as for decode.
    """
    B, H = q_nope.shape[0], q_nope.shape[1]
    out = np.full((B, H, W_UV.shape[1]), np.nan)
    lse = np.full((B, H), np.nan)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    by_seq: dict[int, list[int]] = {}
    for b, h in pairs:
        by_seq.setdefault(int(b), []).append(int(h))
    fn = attend_absorbed if absorbed else attend_unabsorbed
    for b, heads in by_seq.items():
        L = int(seq_lens[b])
        rows = gather_rows(cache, scale_zero, block_table, b, L, page_size, int8, fp8=fp8)
        chosen = [int(i) for i in np.asarray(token_indices[b]).ravel() if 0 <= int(i) < L]
        sel = rows[chosen] if chosen else rows[:0]
        for h in heads:
            o, l, _ = fn(q_nope[b, h], q_pe[b, h], sel, W_UK[h], W_UV[h], scale)
            out[b, h] = o
            lse[b, h] = l
    return out, lse
