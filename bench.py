"""Benchmark of one decode step of paged MLA attention on GB300.

A step is the whole hot path for one layer: append the new token of every
sequence into the paged cache (mla_cache_append), then mla_decode (query
absorption, split-KV tensor-core attention, LSE combine + W^UV projection).
Inputs are seeded synthetic tensors of the workload's shapes, resident in HBM
before timing; the default workload's cache is larger than L2, so no flush is
needed between its steps (a workload whose cache fits in L2 gets a 256 MB
write between timed steps, outside their events).  Prints one JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload v2lite]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

IDX_SETS = 4  # sparse workloads: top-k selections the steps cycle through
METRIC = "MLA decode tokens/s and latent-cache HBM GB/s (fraction of 8 TB/s), 1×GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "MLA chunked-prefill tokens/s (chunk tokens written and attended), 1×GB300"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v2lite")
    ap.add_argument("--num-splits", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="run the workload with this many sequences instead (small cases for profiler captures)")
    return ap.parse_args()


def pick_workload(args):
    """The named workload, or (--batch) the same workload with another number of sequences."""
    from mla_decode_attention_paged_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if args.batch is not None and args.batch != w.batch:
        w = w.scaled(batch=args.batch, name=f"{w.name}@batch{args.batch}")
    return w


def dist_setup(n):
    import torch
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's value (the whole job ends when the last rank does)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time (weak scaling)."""
    return units_per_rank * world / (ms / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor-core TFLOP/s: the measured burst figure (a kernel timed alone), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_flops(seq_lens, chunk: int, heads: int) -> float:
    """Algorithmic FLOPs of the chunk's attention in the absorbed form: each
    (query token, head) scores every visible key over the 576-wide rows and
    sums 512-wide latent values, 2 * 576 + 2 * 512 FLOPs per key."""
    total = 0
    for L in seq_lens:
        first = int(L) - chunk            # position of the chunk's first token
        vis = [max(0, first + t + 1) for t in range(chunk)]
        total += sum(vis)
    return float(total) * heads * (2 * 576 + 2 * 512)


def attention_kernel(fmt: str, rows: int = 16):
    """(source file, kernel name) of the attention kernel the library runs for
    this cache format and number of query rows per sequence (heads x tokens)."""
    if rows % 128 == 0 or (rows > 32 and (fmt != "bf16" or rows > 64 or rows % 32)):
        return (os.path.join(ROOT, "mla_decode_attention_paged_gb300", "csrc", "decode_hm.cu"),
                f"decode_hm_kernel (128-row groups on CTA pairs, {fmt.upper()} cache)")
    name = "decode_pair.cu" if fmt == "bf16" else "decode_tc.cu"
    return (os.path.join(ROOT, "mla_decode_attention_paged_gb300", "csrc", name),
            "decode_pair_kernel (split-KV attention on CTA pairs)" if fmt == "bf16"
            else f"decode_tc_kernel (single-CTA split-KV attention, {fmt.upper()} cache)")


# bytes one cached token occupies: 576 values plus its quantisation parameters
BYTES_PER_TOKEN = {"bf16": 1152, "int8": 584, "fp8": 580}


def workload_config(w, cache_bytes: int, world: int) -> dict:
    """The `config` of a bench line: what the workload is, the same for both arms."""
    T = w.chunk or w.q_len
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "context": w.context, "page_size": w.page_size,
            "q_len": T, "top_k": w.top_k or None, "chunk": w.chunk or None, "cache_bytes": cache_bytes,
            "l2": ("inputs larger than L2 (no flush): each step reads one of "
                   f"{IDX_SETS} top-k selections, {IDX_SETS * cache_bytes / 1e6:.0f} MB of rows together"
                   if w.top_k else
                   "inputs larger than L2 (no flush): the cache read each step exceeds the 126 MB L2"
                   if cache_bytes > 200e6 else
                   "cache smaller than L2: a 256 MB buffer is written between timed steps, outside their "
                   "events (the end-to-end rate runs its steps back to back)"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def kernel_traffic(workload_name: str, tokens: int, fmt: str, rows: int = 16):
    """DRAM bytes per attention launch from the committed ncu summary, scaled
    to this launch's tokens; None if absent or taken on a different kernel."""
    path = os.path.join(ROOT, "profiles", "attention_dram_traffic.json")
    if not os.path.exists(path):
        return None
    e = json.load(open(path)).get("workloads", {}).get(workload_name)
    if not e:
        return None
    src, _ = attention_kernel(fmt, rows)
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != e.get("kernel_sha256"):
        return None
    return round(e["dram_bytes_per_token"] * tokens)


def staging(tensors: dict, dev):
    """One pinned host buffer and one device buffer that hold every tensor of
    ``tensors`` in 256-byte aligned slots, filled with the tensors' values.
    Returns (host buffer, device buffer, host views, device views)."""
    import torch
    slots, off = {}, 0
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        slots[k] = (off, n)
        off = (off + n + 255) // 256 * 256
    host = torch.empty(off, dtype=torch.uint8).pin_memory()
    devb = torch.empty(off, dtype=torch.uint8, device=dev)
    hv, dv = {}, {}
    for k, t in tensors.items():
        o, n = slots[k]
        hv[k] = host[o:o + n].view(t.dtype).view(t.shape)
        dv[k] = devb[o:o + n].view(t.dtype).view(t.shape)
        hv[k].copy_(t.detach().cpu())
    devb.copy_(host)
    return host, devb, hv, dv


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline_prefill(w, inp, seconds, gpu_out=None, gpu_lse=None, absorbed=False):
    """The oracle's chunked prefill on the host cores: per sampled sequence it
    appends the chunk to that sequence's pages itself and attends three of
    the chunk's tokens (first, middle, last) with every head, un-absorbed in
    fp64 (or in the oracle's absorbed form), until about `seconds` have
    passed.  Returns (baseline, parity) as cpu_baseline does, parity over the
    (token, head) rows computed."""
    import numpy as np
    import oracle as O
    import torch
    from mla_decode_attention_paged_gb300 import workloads as W
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 0) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    f64 = lambda t: O.bf16_bits_to_f64(W.bf16_to_bits(t))
    qn, qp, wk, wv = f64(inp["q_nope"]), f64(inp["q_pe"]), f64(inp["W_UK"]), f64(inp["W_UV"])
    c_bits, k_bits = W.bf16_to_bits(inp["chunk_c_kv"]), W.bf16_to_bits(inp["chunk_k_pe"])
    table = inp["block_table"].cpu().numpy()
    lens = inp["seq_lens"].cpu().numpy()
    T, H = w.chunk, w.heads
    toks = sorted({0, T // 2, T - 1})
    done, el = 0, 0.0
    worst = {"abs": 0.0, "rel": 0.0, "lse": 0.0, "rows": 0}
    while el < seconds:
        b = done % w.batch
        n = (int(lens[b]) + w.page_size - 1) // w.page_size
        tab = np.full_like(table, -1)
        tab[b, :n] = np.arange(n)
        # the sequence's pages: the history as cached; the oracle's own append rewrites the chunk's rows
        idx = torch.as_tensor(table[b, :n].astype(np.int64), device=inp["cache_dev"].device)
        cache = W.bf16_to_bits(inp["cache_dev"].index_select(0, idx))
        triples = [(b, t, h) for t in toks for h in range(H)]
        t_start = time.perf_counter()
        ref_o, ref_l = O.prefill_chunk(cache, None, tab, lens, c_bits, k_bits, w.rope_theta, qn, qp, wk, wv,
                                       inp["scale"], w.page_size, False, triples=triples, absorbed=absorbed)
        el += time.perf_counter() - t_start
        if gpu_out is not None and done < w.batch:
            for _, t, h in triples:
                g = np.asarray(gpu_out[b, t, h], np.float64)
                r = ref_o[b, t, h]
                err = float(np.abs(g - r).max())
                worst["abs"] = max(worst["abs"], err)
                worst["rel"] = max(worst["rel"], err / max(float(np.abs(r).max()), 1e-300))
                worst["lse"] = max(worst["lse"], abs(float(gpu_lse[b, t, h]) - float(ref_l[b, t, h])))
                worst["rows"] += 1
        done += 1
    form = "absorbed" if absorbed else "un-absorbed"
    base = {"value": done * len(toks) / el, "unit": "tokens/s", "cores": cores,
            "kind": "oracle (absorbed form)" if absorbed else "oracle",
            "sample": f"{done} sequence(s) of {w.name}: the oracle appends the {T}-token chunk and attends "
                      f"tokens {toks} with all {H} heads ({form} fp64 oracle), {el:.1f} s"}
    parity = None
    if gpu_out is not None:
        ok = worst["abs"] <= 2e-2 and worst["rel"] <= 1e-2 and worst["lse"] <= 2e-2
        parity = {"rows_checked": worst["rows"], "sequences": min(done, w.batch), "max_abs": worst["abs"],
                  "max_rel_row": worst["rel"], "max_lse_abs": worst["lse"],
                  "tolerance": {"abs": 2e-2, "rel_row": 1e-2, "lse_abs": 2e-2}, "pass": ok,
                  "against": "un-absorbed fp64 oracle on the step's own inputs"}
    return base, parity


def cpu_baseline(w, inp, seconds, gpu_out=None, gpu_lse=None, absorbed=False):
    """The fp64 oracle as it stands, on the host cores, over whole sequences
    (all heads) of this workload until about `seconds` have passed: its
    un-absorbed definition, or (absorbed=True) its absorbed cross-check form.
    Returns (baseline dict, parity dict or None): given the GPU's out / lse of
    the same step, the oracle's results for the sequences it ran are compared
    with them (max abs error, max per-row relative error, max lse error)."""
    if w.chunk:
        return cpu_baseline_prefill(w, inp, seconds, gpu_out, gpu_lse, absorbed)
    import numpy as np
    import oracle as O
    from mla_decode_attention_paged_gb300 import workloads as W
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 0) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    f64 = lambda t: O.bf16_bits_to_f64(W.bf16_to_bits(t))
    qn, qp, wk, wv = f64(inp["q_nope"]), f64(inp["q_pe"]), f64(inp["W_UK"]), f64(inp["W_UV"])
    table = inp["block_table"].cpu().numpy()
    lens = inp["seq_lens"].cpu().numpy()
    import torch
    done, el, tokens_attended = 0, 0.0, 0
    worst = {"abs": 0.0, "rel": 0.0, "lse": 0.0, "rows": 0, "bad": 0}

    def compare(b, ref_o, ref_l):
        g = np.asarray(gpu_out[b], np.float64).reshape(-1, ref_o.shape[-1])
        r = ref_o[b].reshape(-1, ref_o.shape[-1])
        gl = np.asarray(gpu_lse[b], np.float64).ravel()
        rl = ref_l[b].ravel()
        for i in range(r.shape[0]):
            err = float(np.abs(g[i] - r[i]).max())
            m = float(np.abs(r[i]).max())
            worst["abs"] = max(worst["abs"], err)
            if m > 0:
                worst["rel"] = max(worst["rel"], err / m)
            elif err > 0:
                worst["bad"] += 1
            if np.isinf(rl[i]):
                worst["bad"] += int(not (np.isinf(gl[i]) and gl[i] < 0))
            else:
                worst["lse"] = max(worst["lse"], abs(float(gl[i]) - float(rl[i])))
            worst["rows"] += 1

    while el < seconds:
        b = done % w.batch
        n = (int(lens[b]) + w.page_size - 1) // w.page_size
        tab = np.full_like(table, -1)
        tab[b, :n] = np.arange(n)
        if w.quantised and "src_c_kv" in inp:   # the oracle's own append builds this sequence's pages
            built = inp.setdefault("oracle_pages", {})   # once per sequence (input set-up, not timed)
            if b not in built:
                a = int(lens[:b].sum())
                cache = np.zeros((n, w.page_size, 576), np.int8 if w.int8 else np.uint8)
                sz = np.zeros((n, w.page_size, 2) if w.int8 else (n, w.page_size), np.float32)
                O.append_tokens(cache, sz, tab, [b] * int(lens[b]), list(range(int(lens[b]))),
                                W.bf16_to_bits(inp["src_c_kv"][a:a + int(lens[b])]),
                                W.bf16_to_bits(inp["src_k_pe"][a:a + int(lens[b])]), w.rope_theta, w.page_size,
                                w.int8, fp8=w.fp8)
                built[b] = (cache, sz)
            cache, sz = built[b]
        else:
            idx = torch.as_tensor(table[b, :n].astype(np.int64), device=inp["cache_dev"].device)
            sub = inp["cache_dev"].index_select(0, idx)
            if w.quantised:
                cache, sz = sub.cpu().numpy(), inp["sz_dev"].index_select(0, idx).cpu().numpy()
            else:
                cache, sz = W.bf16_to_bits(sub), None
        t_start = time.perf_counter()   # time the oracle itself, not the page gather
        if w.top_k:
            idx = inp["token_indices"].cpu().numpy()
            ref = O.decode_sparse(qn, qp, cache, sz, tab, lens, idx, wk, wv, inp["scale"], w.page_size, w.int8,
                                  pairs=[(b, h) for h in range(w.heads)], absorbed=absorbed, fp8=w.fp8)
        elif w.q_len == 1:
            ref = O.decode(qn, qp, cache, sz, tab, lens, wk, wv, inp["scale"], w.page_size, w.int8,
                           pairs=[(b, h) for h in range(w.heads)], absorbed=absorbed, fp8=w.fp8)
        else:
            ref = O.decode_multi_token(qn, qp, cache, sz, tab, lens, wk, wv, inp["scale"], w.page_size, w.int8,
                                       triples=[(b, t, h) for t in range(w.q_len) for h in range(w.heads)],
                                       absorbed=absorbed, fp8=w.fp8)
        el += time.perf_counter() - t_start
        if gpu_out is not None and done < w.batch:
            compare(b, *ref)
        done += 1
        tokens_attended += int((inp["token_indices"][b] >= 0).sum()) if w.top_k else int(lens[b])
    form = "absorbed" if absorbed else "un-absorbed"
    base = {"value": done * w.q_len / el, "unit": "tokens/s", "cores": cores,
            "kind": "oracle (absorbed form)" if absorbed else "oracle",
            "sample": f"{done} whole sequence(s) x {w.q_len} token(s) x {w.heads} heads of {w.name} "
                      f"({tokens_attended} cached tokens, "
                      f"{form} fp64 oracle), {el:.1f} s"}
    parity = None
    if gpu_out is not None:
        ok = worst["abs"] <= 2e-2 and worst["rel"] <= 1e-2 and worst["lse"] <= 2e-2 and worst["bad"] == 0
        parity = {"rows_checked": worst["rows"], "sequences": min(done, w.batch), "max_abs": worst["abs"],
                  "max_rel_row": worst["rel"], "max_lse_abs": worst["lse"],
                  "tolerance": {"abs": 2e-2, "rel_row": 1e-2, "lse_abs": 2e-2}, "pass": ok,
                  "against": "un-absorbed fp64 oracle on the step's own inputs"}
    return base, parity


def run_ours(args, rank, world):
    import torch
    import mla_decode_attention_paged_gb300 as mla
    from mla_decode_attention_paged_gb300 import workloads as W

    dev = torch.device("cuda", torch.cuda.current_device())
    mla.load_library(build_if_missing=True)
    w = pick_workload(args)
    inp = W.make_decode_inputs(w, device=dev)
    d = mla.dims(w.heads, w.page_size, int8=w.int8, fp8=w.fp8)
    B, H, T = w.batch, w.heads, (w.chunk or w.q_len)
    seq_lens = inp["seq_lens"]
    table = inp["block_table"].to(dev)
    npg = inp["num_pages"]
    # the cache: drawn directly (bf16) or written through the library's append (INT8, FP8)
    if w.quantised:
        cache = torch.zeros((npg, w.page_size, 576), dtype=torch.int8 if w.int8 else torch.uint8, device=dev)
        sz = torch.zeros((npg, w.page_size, 2) if w.int8 else (npg, w.page_size), dtype=torch.float32,
                         device=dev)
        mla.cache_append(d, cache, sz, table, inp["src_seq_ids"], inp["src_positions"], inp["src_c_kv"],
                         inp["src_k_pe"], w.rope_theta)
        del inp["src_c_kv"], inp["src_k_pe"]
    else:
        cache, sz = inp["cache"], None
    inp["cache_dev"], inp["sz_dev"] = cache, sz
    # the step's new tokens: the last T positions of each sequence
    g = W.generator(w.seed + 1000, dev)
    new_c = W.draw_bf16((B * T, 512), 1.0, g)
    new_k = W.draw_bf16((B * T, 64), 1.0, g)
    seq_ids = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(T)
    positions = (seq_lens.to(dev).repeat_interleave(T) - T +
                 torch.arange(T, dtype=torch.int32, device=dev).repeat(B)).clamp(min=0).to(torch.int32)
    # the kernels see T * H heads per sequence; the automatic split count is theirs
    d_rows = mla.dims(H * T, w.page_size, int8=w.int8, fp8=w.fp8)
    auto = mla.auto_num_splits(d_rows if mla.check_dims(d_rows) == mla.MLA_OK else d, B)
    splits = args.num_splits if args.num_splits is not None else (W.num_splits_for(w, auto) or auto)
    ws_bytes = (mla.decode_sparse_workspace_size(d, B, w.top_k, splits) if w.top_k
                else mla.prefill_workspace_size(d, B, T, splits) if w.chunk
                else mla.decode_multi_workspace_size(d, B, T, splits))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    qshape = (B, H) if T == 1 else (B, T, H)
    out = torch.empty(qshape + (128,), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(qshape, dtype=torch.float32, device=dev)
    q_nope, q_pe, W_UK, W_UV = inp["q_nope"], inp["q_pe"], inp["W_UK"], inp["W_UV"]
    seq_lens = seq_lens.to(dev)
    token_indices = inp.get("token_indices")
    # sparse: the selection changes every step, cycling through kIdxSets seeded
    # top-k sets (their rows together exceed L2, so no step finds its rows left
    # there by the step before)
    idx_sets = [token_indices]
    if w.top_k:
        idx_sets += [W.draw_token_indices(inp["seq_lens"].cpu(), w.top_k, 1.0, W.generator(w.seed + 2000 + r, dev)).to(dev)
                     for r in range(1, IDX_SETS)]

    def decode_fn(qn, qp, tab, lens, idx, o, l):
        """The workload's decode call: mla_decode, mla_decode_multi or mla_decode_sparse."""
        if w.top_k:
            mla.decode_sparse(d, qn, qp, cache, sz, tab, lens, idx, W_UK, W_UV, inp["scale"], num_splits=splits,
                              workspace=ws, out=o, lse_out=l)
        elif T == 1:
            mla.decode(d, qn, qp, cache, sz, tab, lens, W_UK, W_UV, inp["scale"], num_splits=splits, workspace=ws,
                       out=o, lse_out=l)
        else:
            mla.decode_multi(d, qn, qp, cache, sz, tab, lens, W_UK, W_UV, inp["scale"], num_splits=splits,
                             workspace=ws, out=o, lse_out=l)

    chunk_c, chunk_k = inp.get("chunk_c_kv"), inp.get("chunk_k_pe")

    def prefill_fn(qn, qp, tab, lens, c_kv, k_pe, o, l):
        """The prefill workload's call: mla_prefill writes the chunk and attends it."""
        mla.prefill(d, cache, sz, tab, lens, c_kv, k_pe, qn, qp, W_UK, W_UV, inp["scale"], rope_theta=w.rope_theta,
                    num_splits=splits, workspace=ws, out=o, lse_out=l)

    def step(i):
        if w.chunk:
            prefill_fn(q_nope, q_pe, table, seq_lens, chunk_c, chunk_k, out, lse)
            return
        mla.cache_append(d, cache, sz, table, seq_ids, positions, new_c, new_k, w.rope_theta)
        decode_fn(q_nope, q_pe, table, seq_lens, idx_sets[i % len(idx_sets)], out, lse)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert mla.read_device_status(ws) == mla.MLA_OK
    # attention-kernel timing through the library's event hook, one pair per step
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:  # create the underlying events
        a.record(); b.record()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a cache that fits in L2 would be found there by the next step: then a
    # buffer larger than L2 is written between timed steps, outside their events
    small = not w.top_k and int(seq_lens.to(torch.int64).sum()) * BYTES_PER_TOKEN[w.cache_format] <= 200e6
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        # untimed steps while the sampler starts (~0.3 s): after that long
        # idle the first steps ran slower, and a short timed run paid for it
        t_end = time.perf_counter() + 0.3
        i = 0
        while time.perf_counter() < t_end:
            step(i)
            i += 1
            if i % 16 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        # the step as a user runs it: no events between its kernels (an event
        # between two kernels would end the overlap of their launches)
        if flush is None:
            e0.record()
            for i in range(args.steps):
                step(i)
            e1.record()
        else:
            for i in range(args.steps):
                flush.zero_()
                sev[i][0].record()
                step(i)
                sev[i][1].record()
        torch.cuda.synchronize()
        # then K more steps with the library's event pair around the attention
        # launch: that kernel's own duration for the roofline
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            mla.set_timing_events(*kev[i])
            step(i)
        torch.cuda.synchronize()
        mla.set_timing_events(None, None)
        # the timed steps take milliseconds and nvidia-smi samples every 100 ms:
        # the same steps go on, untimed, for about half a second more so that
        # the clock record holds samples under this load
        t_end = time.perf_counter() + 0.5
        i = 0
        while time.perf_counter() < t_end:
            step(i)
            i += 1
            if i % 16 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = e0.elapsed_time(e1) if flush is None else sum(a.elapsed_time(b) for a, b in sev)
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    ms_total = max_over_ranks(ms_total, world)
    ms = ms_total / args.steps
    # tokens the attention reads: every cached one, or the selected ones (sparse)
    lens_sum = int((token_indices >= 0).sum()) if w.top_k else int(seq_lens.to(torch.int64).sum())
    bytes_per_token = BYTES_PER_TOKEN[w.cache_format]
    cache_bytes = lens_sum * bytes_per_token
    tokens_per_s = whole_job_rate(B * T, world, ms)
    step_cache_gbs = whole_job_rate(cache_bytes, world, ms) / 1e9

    # e2e: the same step through the public API from pinned host memory.  The
    # step's inputs sit in one pinned staging buffer and go over in one copy;
    # the library writes out and lse into one device buffer that comes back in
    # one copy (every byte of the step's inputs and results still crosses).
    # Two device copies of both, and a copy stream: step i + 2's inputs go in
    # and step i's results come out while the next steps compute, as a serving
    # loop would run it.  The timed region holds every copy of the K steps.
    step_inputs = (dict(q_nope=q_nope, q_pe=q_pe, c_kv=chunk_c, k_pe=chunk_k, table=table, seq_lens=seq_lens)
                   if w.chunk else
                   dict(q_nope=q_nope, q_pe=q_pe, new_c=new_c, new_k=new_k, seq_ids=seq_ids, positions=positions,
                        table=table, seq_lens=seq_lens))
    h_bufs = []
    for r in range(len(idx_sets)):
        if w.top_k:
            step_inputs["token_indices"] = idx_sets[r]
        h_bufs.append(staging(step_inputs, dev)[0])
    d_ins = [staging(step_inputs, dev) for _ in range(2)]      # (host, device, host views, device views)
    d_outs = [staging(dict(out=out, lse=lse), dev) for _ in range(2)]
    h_out_buf = d_outs[0][0]
    h2d = h_bufs[0].numel()
    d2h = h_out_buf.numel()
    main_s, copy_s = torch.cuda.current_stream(), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        k = i % 2
        if i >= 2:
            copy_s.wait_event(ev_done[k])   # step i - 2 has finished with this buffer
        with torch.cuda.stream(copy_s):
            d_ins[k][1].copy_(h_bufs[i % len(h_bufs)], non_blocking=True)
        ev_in[k].record(copy_s)

    def compute(i):
        k = i % 2
        main_s.wait_event(ev_in[k])
        d_in, d_out = d_ins[k][3], d_outs[k][3]
        if w.chunk:
            prefill_fn(d_in["q_nope"], d_in["q_pe"], d_in["table"], d_in["seq_lens"], d_in["c_kv"], d_in["k_pe"],
                       d_out["out"], d_out["lse"])
        else:
            mla.cache_append(d, cache, sz, d_in["table"], d_in["seq_ids"], d_in["positions"], d_in["new_c"],
                             d_in["new_k"], w.rope_theta)
            decode_fn(d_in["q_nope"], d_in["q_pe"], d_in["table"], d_in["seq_lens"], d_in.get("token_indices"),
                      d_out["out"], d_out["lse"])
        ev_done[k].record(main_s)
        copy_s.wait_event(ev_done[k])
        with torch.cuda.stream(copy_s):
            h_out_buf.copy_(d_outs[k][1], non_blocking=True)

    def e2e_run(n):
        if n == 0:
            return
        copy_in(0)
        if n > 1:
            copy_in(1)
        for i in range(n):
            compute(i)
            if i + 2 < n:
                copy_in(i + 2)
        main_s.wait_stream(copy_s)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(main_s)
    copy_s.wait_event(x0)
    e2e_run(args.steps)
    x1.record(main_s)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, world)

    peak, peak_src = peaks()
    tpeak, tpeak_src = tensor_peak()
    achieved = cache_bytes / (kern_ms / 1e3) / 1e9
    traffic = kernel_traffic(w.name, lens_sum, w.cache_format, H * T)
    kname = attention_kernel(w.cache_format, H * T)[1]
    # the attention's algorithmic FLOPs (absorbed form): every (query row,
    # visible token) pair scores a 576-wide row and adds a 512-wide one
    flops = (prefill_flops(seq_lens.cpu().tolist(), T, H) if T > 1 else
             float(lens_sum) * H * (2 * 576 + 2 * 512))
    tflops = flops / (kern_ms / 1e3) / 1e12
    hbm_frac, tensor_frac = achieved / peak, tflops / tpeak
    # the binding bound: whichever peak the launch's work needs longer on
    if flops / (tpeak * 1e12) > cache_bytes / (peak * 1e9):
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(tensor_frac, 4), "peak_source": tpeak_src, "traffic": traffic, "kernel": kname,
                    "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": cache_bytes,
                    "hbm_frac": round(hbm_frac, 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(hbm_frac, 4), "peak_source": peak_src, "traffic": traffic, "kernel": kname,
                    "algorithmic_bytes_per_launch": cache_bytes, "algorithmic_flops_per_launch": flops,
                    "tensor_frac": round(tensor_frac, 4)}
    if w.chunk:
        # prefill is compute-bound: FLOPs of the chunk's attention against the bf16 tensor peak
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(tflops / tpeak, 4), "peak_source": tpeak_src, "traffic": traffic,
                    "kernel": kname, "algorithmic_flops_per_launch": flops,
                    "history_bytes_per_launch": cache_bytes}
    res = {
        "metric": PREFILL_METRIC if w.chunk else METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "int8": "int8", "fp8": "fp8_e4m3"}[w.cache_format],
        "data": "synthetic (seeded; random-init weights of DeepSeek-V2 MLA shapes)",
        "config": workload_config(w, cache_bytes, world),
        "num_splits": splits,
        "cache_gbs": round(step_cache_gbs, 1),
        "frac_of_8tbs": round(step_cache_gbs / NOMINAL_HBM_GBS, 4),
        "attention_kernel_ms": round(kern_ms, 5),
        "roofline": roofline,
        "e2e": {"value": round(whole_job_rate(B * T, world, e2e_ms), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": (5 if w.top_k else 4) * args.steps,  # + the gather kernel for sparse decode
        "clocks": {**clk.summary(),
                   "window": "0.3 s of the same steps, the timed steps, then 0.5 s more (nvidia-smi every 100 ms)"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # one more step with the first selection (sparse), so that out / lse
        # are the results for the inputs the oracle reads
        step(0)
        torch.cuda.synchronize()
        res["cpu_baseline"], res["parity"] = cpu_baseline(w, inp, args.cpu_seconds, out.float().cpu().numpy(),
                                                          lse.cpu().numpy())
        # the oracle's absorbed form: the same fp64 arithmetic after the weight absorption
        res["cpu_baseline_absorbed"], _ = cpu_baseline(w, inp, max(2.0, args.cpu_seconds / 2), absorbed=True)
    return res


def run_reference(args, rank, world):
    """The oracle (the reference arm): bounded samples of the same workload on the host cores."""
    import torch
    import oracle as O  # noqa: F401
    from mla_decode_attention_paged_gb300 import workloads as W
    if rank != 0:
        return None
    w = pick_workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_decode_inputs(w.scaled(batch=min(w.batch, 4)) if w.quantised else w, device=dev)
    inp["cache_dev"], inp["sz_dev"] = inp.get("cache"), None
    # the bytes the attention of one full step reads, as the GPU arm counts them
    if w.top_k:
        attended = int((inp["token_indices"] >= 0).sum())
    else:
        attended = int(W.draw_seq_lens(w, W.generator(w.seed, dev)).to(torch.int64).sum())
    cache_bytes = attended * BYTES_PER_TOKEN[w.cache_format]
    per_step = max(1.0, min(6.0, 150.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        cpu_baseline(w, inp, per_step * 0.2)
    vals, samples = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r, _ = cpu_baseline(w, inp, per_step)
        vals.append(1.0 / r["value"])
        samples.append(r["sample"])
    el = time.perf_counter() - t0
    v = args.steps / sum(vals)
    cb = {"value": round(v, 5), "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
          "sample": f"per step: {samples[0]}"}
    return {"metric": PREFILL_METRIC if w.chunk else METRIC, "value": round(v, 5), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(w, cache_bytes, world), "impl": "reference",
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world = dist_setup(args.gpus)
    res = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
