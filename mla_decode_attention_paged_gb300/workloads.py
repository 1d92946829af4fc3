"""Seeded synthetic inputs for paged MLA decode.

This module holds random draws, page tables and sequence lengths only -- none
of the method's arithmetic -- so that the oracle tests and the CUDA path can
draw identical inputs from it.  Shapes follow DeepSeek-V2-Lite / DeepSeek-V2
("Seven Ways LLMs Handle Attention", opening section and section 5: a
512-wide latent plus a 64-wide RoPE key per token, 16 or 128 heads, per-head
key 128+64 and value 128).  No trained weights or datasets are used:
weights are random normal draws of the right shape.

Draw order for a workload is fixed (lengths, page permutation, cache,
W_UK, W_UV, q_nope, q_pe, then append sources) so a seed names one input.
"""
from __future__ import annotations

import dataclasses
import math

import torch

LATENT_DIM = 512
ROPE_DIM = 64
NOPE_DIM = 128
V_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    context: int | tuple[int, int]  # fixed length, or (lo, hi) drawn uniformly per sequence
    page_size: int
    shuffled: bool                  # physical pages a seeded random permutation (else identity)
    cache_std: float
    w_std: float
    q_std: float
    seed: int
    int8: bool = False              # cache built from N(0,1) rows by the INT8 append
    min_splits_per_seq: int = 0     # the workload asks for at least this many KV chunks per sequence
    rope_theta: float = 10000.0     # used where the cache is built through the append
    q_len: int = 1                  # query tokens per sequence (multi-token decode: the last q_len cached)
    top_k: int = 0                  # sparse decode: attend to top_k drawn positions per sequence (0: all)
    fp8: bool = False               # cache built from N(0,1) rows by the FP8 (E4M3) append
    chunk: int = 0                  # chunked prefill: the last `chunk` tokens of each sequence are the
                                    # chunk, written and attended by one prefill call (0: decode)

    @property
    def quantised(self) -> bool:
        """1-byte cache (INT8 or FP8) with per-token scales, built through an append."""
        return self.int8 or self.fp8

    @property
    def cache_format(self) -> str:
        return "int8" if self.int8 else "fp8" if self.fp8 else "bf16"

    @property
    def softmax_scale(self) -> float:
        # 1/sqrt(per-head key width) = 1/sqrt(128 + 64)
        return 1.0 / math.sqrt(NOPE_DIM + ROPE_DIM)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny_b1_h16_l256_p16", 1, 16, 256, 16, False, 0.02, 0.02, 1.0, 0),
    "v2lite": Workload("v2lite_b32_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 1),
    "ragged": Workload("ragged_b64_h128_l1024-131072_p64", 64, 128, (1024, 131072), 64, True, 1.0, 0.02, 1.0, 2),
    "ctx1m": Workload("ctx1m_b2_h16_l1048576_p64", 2, 16, 1048576, 64, True, 1.0, 0.02, 1.0, 3,
                      min_splits_per_seq=148),
    "int8": Workload("int8_b128_h128_l8192_p64", 128, 128, 8192, 64, True, 1.0, 0.02, 1.0, 4, int8=True),
    # multi-token decode (speculative verification) on the V2-Lite shape: 2 or 4 new tokens per sequence
    "v2lite_mtp2": Workload("v2lite_mtp2_b32_t2_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 5,
                            q_len=2),
    "v2lite_mtp4": Workload("v2lite_mtp4_b32_t4_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 6,
                            q_len=4),
    # the V2-Lite batch over an INT8 cache (half the bytes per token)
    "int8_v2lite": Workload("int8_v2lite_b32_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 8, int8=True),
    # the V2-Lite batch over an FP8 (E4M3) cache with one scale per token
    "fp8_v2lite": Workload("fp8_v2lite_b32_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 9, fp8=True),
    # chunked prefill on the V2-Lite shape: 4 sequences, a 512-token chunk after 8,192 cached tokens
    "v2lite_prefill512": Workload("v2lite_prefill512_b4_h16_l8704_p64", 4, 16, 8704, 64, True, 1.0, 0.02, 1.0, 10,
                                  chunk=512),
    # sparse decode (DeepSeek Sparse Attention's top-2048 selection) over the V2-Lite cache
    "v2lite_topk2048": Workload("v2lite_topk2048_b32_h16_l32768_p64", 32, 16, 32768, 64, True, 1.0, 0.02, 1.0, 7,
                                top_k=2048),
}


def num_splits_for(w: Workload, auto_splits: int) -> int:
    """KV partitions to run ``w`` with: the automatic count, raised where the
    workload asks for a minimum number of chunks per sequence (equal-length
    sequences get num_splits / batch chunks each) -- to a multiple of the
    automatic count, so that every CTA pair (one partition each at the
    automatic count) walks the same number of equal partitions."""
    if w.min_splits_per_seq:
        need = max(auto_splits, w.min_splits_per_seq * w.batch)
        return -(-need // auto_splits) * auto_splits
    return 0


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_seq_lens(w: Workload, g: torch.Generator) -> torch.Tensor:
    """int32 [B] sequence lengths (including the token being decoded)."""
    if isinstance(w.context, tuple):
        lo, hi = w.context
        return torch.randint(lo, hi + 1, (w.batch,), generator=g, device=g.device, dtype=torch.int64).to(torch.int32)
    return torch.full((w.batch,), w.context, dtype=torch.int32, device=g.device)


def draw_page_table(seq_lens: torch.Tensor, page_size: int, shuffled: bool, g: torch.Generator,
                    spare_pages: int = 0):
    """Give each sequence ceil(len / page_size) physical pages from one pool.

    Returns (block_table int32 [B, max_pages], num_pages).  Physical pages are
    a seeded permutation of the pool when ``shuffled``; table entries past a
    sequence's last page are -1 (never read).
    """
    lens = seq_lens.to("cpu", torch.int64)
    need = (lens + page_size - 1) // page_size
    total = int(need.sum()) + spare_pages
    max_pages = max(int(need.max()) if len(need) else 1, 1)
    phys = torch.randperm(total, generator=g, device=g.device).cpu() if shuffled else torch.arange(total)
    table = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need.tolist()):
        table[b, :n] = phys[off:off + n].to(torch.int32)
        off += n
    return table, total


def draw_bf16(shape, std: float, g: torch.Generator) -> torch.Tensor:
    return (torch.randn(shape, generator=g, device=g.device, dtype=torch.float32) * std).to(torch.bfloat16)


def draw_int8_cache(num_pages: int, page_size: int, g: torch.Generator):
    """Random INT8 codes [num_pages, P, 576] and (scale, zero point) fp32
    [num_pages, P, 2] for decode-only tests of the quantised cache.

    Zero points are drawn from [-8, 8], as for rows whose range is roughly
    centred on 0 (per-token quantisation of zero-mean rows puts the zero
    point near 0); scales are uniform in [0.002, 0.032]."""
    codes = torch.randint(-128, 128, (num_pages, page_size, LATENT_DIM + ROPE_DIM), generator=g,
                          device=g.device, dtype=torch.int32).to(torch.int8)
    scale = torch.rand((num_pages, page_size), generator=g, device=g.device) * 0.03 + 0.002
    zp = torch.randint(-8, 9, (num_pages, page_size), generator=g, device=g.device).to(torch.float32)
    return codes, torch.stack([scale, zp], dim=-1).contiguous()


def draw_fp8_cache(num_pages: int, page_size: int, g: torch.Generator):
    """Random FP8 E4M3 codes uint8 [num_pages, P, 576] -- uniform over the 254
    finite codes (0x7F and 0xFF, the NaN patterns, are skipped) -- and scales
    fp32 [num_pages, P] uniform in [0.002, 0.01], for decode-only tests of the
    quantised cache."""
    v = torch.randint(0, 254, (num_pages, page_size, LATENT_DIM + ROPE_DIM), generator=g, device=g.device,
                      dtype=torch.int32)
    codes = (v + (v >= 0x7F).to(torch.int32)).to(torch.uint8)
    scale = torch.rand((num_pages, page_size), generator=g, device=g.device) * 0.008 + 0.002
    return codes, scale.contiguous()


def make_decode_inputs(w: Workload, device="cpu"):
    """All inputs of one decode step for workload ``w``, drawn on ``device``.

    bf16 workloads: the physical cache pool is filled directly with
    N(0, cache_std) values.  INT8 and FP8 workloads: the generator returns N(0, 1)
    source rows (latent and RoPE key) for every token of every sequence, to be
    written through the append of whichever side is under test; no cache is
    drawn.
    """
    g = generator(w.seed, device)
    seq_lens = draw_seq_lens(w, g)
    table, num_pages = draw_page_table(seq_lens, w.page_size, w.shuffled, g)
    d = dict(workload=w, seq_lens=seq_lens.to(device), block_table=table.to(device), num_pages=num_pages,
             page_size=w.page_size, scale=w.softmax_scale)
    if not w.quantised:
        d["cache"] = draw_bf16((num_pages, w.page_size, LATENT_DIM + ROPE_DIM), w.cache_std, g)
    d["W_UK"] = draw_bf16((w.heads, NOPE_DIM, LATENT_DIM), w.w_std, g)
    d["W_UV"] = draw_bf16((w.heads, V_DIM, LATENT_DIM), w.w_std, g)
    T = w.chunk or w.q_len
    qshape = (w.batch, w.heads) if T == 1 else (w.batch, T, w.heads)
    d["q_nope"] = draw_bf16(qshape + (NOPE_DIM,), w.q_std, g)
    d["q_pe"] = draw_bf16(qshape + (ROPE_DIM,), w.q_std, g)
    if w.chunk:  # the chunk's new rows (unrotated RoPE key), written by the prefill call
        d["chunk_c_kv"] = draw_bf16((w.batch, w.chunk, LATENT_DIM), 1.0, g)
        d["chunk_k_pe"] = draw_bf16((w.batch, w.chunk, ROPE_DIM), 1.0, g)
    if w.top_k:
        d["token_indices"] = draw_token_indices(seq_lens.cpu(), w.top_k, 1.0, g).to(device)
    if w.quantised:
        total = int(seq_lens.to(torch.int64).sum())
        d["src_c_kv"] = draw_bf16((total, LATENT_DIM), 1.0, g)
        d["src_k_pe"] = draw_bf16((total, ROPE_DIM), 1.0, g)
        lens = seq_lens.cpu().to(torch.int64)
        d["src_seq_ids"] = torch.repeat_interleave(torch.arange(w.batch, dtype=torch.int32), lens).to(device)
        d["src_positions"] = torch.cat([torch.arange(int(n), dtype=torch.int32) for n in lens]).to(device)
    return d


def draw_token_indices(seq_lens: torch.Tensor, top_k: int, fill: float, g: torch.Generator) -> torch.Tensor:
    """A sparse-attention selection per sequence (int32 [B, top_k]): about
    ``fill * top_k`` distinct positions below the sequence's length (all of
    them if it is shorter), in random order, then -1 padding."""
    B = seq_lens.numel()
    out = torch.full((B, top_k), -1, dtype=torch.int32)
    for b in range(B):
        L = int(seq_lens[b])
        n = min(L, max(1, int(round(fill * top_k)))) if L > 0 else 0
        if n:
            out[b, :n] = torch.randperm(L, generator=g, device=g.device)[:n].to(torch.int32).cpu()
    return out


def bf16_to_bits(t: torch.Tensor):
    """uint16 bit patterns of a bf16 tensor as a numpy array (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
