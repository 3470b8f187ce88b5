"""Benchmark: paged decode attention on one or more GB300s (one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras]

One step of the default workload (Llama-2-7B-shaped dense bf16 decode: batch 4,
32 layers, 32 query heads = 32 kv heads, head_dim 128, context 2048, page 16)
is, for every layer, kv_append of one new token per sequence (position 2047,
so attention reads 2048 tokens) followed by paged_decode_attention. The 32
layers' calls are captured once in a CUDA graph and replayed. Inputs (4.3 GB of
KV) are larger than L2, so no flush is needed between steps.

The value is KV GB/s: the step's algorithmic bytes (K and V of every attended
token, INT8 scales, q, output, block-table entries, appended tokens) divided by
the device time of a step. Other workloads of the pages are timed the same way
and reported under "workloads". The reference arm (--impl reference) times the
fp64 CPU oracle on the host cores on a bounded sample of the same workload.

With --gpus N under torchrun, every rank runs its own replica of the workload
(independent sequences: weak scaling, no collective on the data path); the
step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time
from typing import Dict, List, Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

DEFAULT_WORKLOAD = "w2_llama7b_bf16"
# attention launches overlap the kernel before them (see Replica._layer)
EARLY_START = True
# the step's append is done by the attention kernel itself where the cache
# allows it (pkv_append_decode_attention)
FUSED_APPEND = True
FALLBACK_HBM_GBS = 6800.0
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


# --------------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base: int, rank: int) -> int:
    """Seed of rank r's replica (rank 0 runs the workload's own seed)."""
    return base + 1000003 * rank


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def algorithmic_bytes(w: synth.Workload, lens: np.ndarray, append_tokens: int = 1,
                      sparse_pages: Optional[int] = None, out_bytes: int = 2,
                      group_shared: bool = False) -> Dict[str, int]:
    """Bytes one layer's decode step must move (no padding, no re-reads).

    attention: K and V of every attended token (codes or fp16/bf16 values) plus
    INT8 scales/zero-points, the queries, the output and block-table entries;
    append: the new tokens read and written (codes + scales when INT8);
    score: the page bounding boxes read by the page scoring (sparse mode).
    group_shared: one page list per kv head, read once for its query-head group.
    """
    H, d, Hq = w.num_kv_heads, w.head_dim, w.num_q_heads
    ps = w.page_size
    if sparse_pages is None:
        toks = lens.astype(np.int64)
        units = H
    else:
        # each query head reads its own selected pages (or each group its list)
        toks = np.minimum(lens.astype(np.int64), sparse_pages * ps)
        units = H if group_shared else Hq
    if w.quant == "none":
        per_tok = 2 * d * 2
    elif w.quant == "per_token_u4":
        per_tok = 2 * (d // 2) + 16           # two 4-bit codes per byte, K and V, + scales
    else:
        per_tok = 2 * d + (16 if w.quant == "per_token" else 0)
    attn = int((toks * units).sum()) * per_tok
    if w.quant == "per_group64":
        attn += int(((toks + 63) // 64 * units).sum()) * 16
    attn += w.batch * Hq * d * (2 + out_bytes)                    # q in, out
    pages = (lens.astype(np.int64) + ps - 1) // ps
    attn += int(pages.sum()) * 4 * (1 if sparse_pages is None else 1)
    res = {"attention": attn}
    if append_tokens:
        src = w.batch * append_tokens * H * d * 2 * 2             # K and V read
        if w.quant == "none":
            dst = src
        elif w.quant == "per_token":
            dst = w.batch * append_tokens * H * 2 * (d + 8)
        elif w.quant == "per_token_u4":
            dst = w.batch * append_tokens * H * 2 * (d // 2 + 8)
        else:
            dst = w.batch * H * 2 * (64 * d + 8) + w.batch * H * 2 * 64 * d * 4  # open group + tail
        res["append"] = src + dst
    if sparse_pages is not None:
        rows = H if group_shared else Hq
        res["score"] = int(pages.sum()) * rows * 2 * d * 4 + w.batch * rows * sparse_pages * 4
    res["total"] = sum(res.values())
    return res


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in ("attention_kernel.cuh", "pkv_common.cuh", "quant.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_243_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str) -> Optional[float]:
    """DRAM bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"ncu_attention_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_tr.group(1))


def load_peaks() -> Dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            p = json.load(open(path))
            return {"hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during the timed region."""

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"pkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> Optional[Dict]:
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], 0.0, set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- GPU workloads
class Replica:
    """One workload's caches, inputs and captured CUDA graphs on this GPU."""

    def __init__(self, w: synth.Workload, seed: int, layers: Optional[int] = None,
                 with_meta: bool = False, top_k: Optional[int] = None, group_mode: int = 0):
        import torch
        from paged_kv_cache_243_gb300.cache import PagedKVCache
        self.torch = torch
        self.w = w
        self.layers = layers or w.layers
        self.top_k = top_k
        self.group_mode = group_mode   # 0: page lists per query head; 1/2: per kv head (sum / max)
        dev = torch.device("cuda")
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        self.lens = synth.seq_lens(w)
        extra = 1 if w.append_steps else 0
        kv_name, quant_name = synth.cache_kind(w)
        qdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        self.qdt = qdt
        B, H, d, Hq = w.batch, w.num_kv_heads, w.head_dim, w.num_q_heads
        T = int(self.lens.max())
        self.caches, self.bts, self.qs, self.outs, self.knews, self.vnews = [], [], [], [], [], []
        # every layer's per-step inputs (q, new K, new V) and outputs live in one
        # contiguous buffer each, so a host round trip is one copy each way
        n_q, n_kv = B * Hq * d, max(1, w.append_steps) * B * H * d
        per_layer = n_q + 2 * n_kv
        self.in_buf = torch.empty(self.layers * per_layer, dtype=qdt, device=dev)
        self.out_buf = torch.empty(self.layers * n_q, dtype=qdt, device=dev)
        self.pos_list = []
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        steps = max(1, w.append_steps)
        # decode positions: the new token overwrites the last slot (fixed-length
        # workloads) or extends the context (append workloads)
        for layer in range(self.layers):
            bt, pool = synth.block_tables(w, layer, extra)
            cache = PagedKVCache(pool, w.page_size, H, d, kv_dtype=kv_name, quant=quant_name,
                                 with_meta=with_meta, tail_rows=B)
            bt_d = torch.from_numpy(bt).to(dev)
            # prefill: T tokens per sequence drawn on the device, written by kv_append
            k0 = torch.randn((B, T, H, d), generator=gen, device=dev, dtype=torch.float32)
            v0 = torch.randn((B, T, H, d), generator=gen, device=dev, dtype=torch.float32)
            if w.outlier_channels:
                oc = torch.from_numpy(synth.outlier_channels(w)).to(dev)
                for g in range(H):
                    k0[:, :, g, oc[g]] *= w.outlier_scale
            if w.page_offset_std > 0:
                P = (T + w.page_size - 1) // w.page_size
                off = torch.randn((B, P, H, d), generator=gen, device=dev) * w.page_offset_std
                k0 += off.repeat_interleave(w.page_size, dim=1)[:, :T]
            pre_lens = self.lens if w.append_steps else self.lens - 1
            cache.append(k0.to(qdt), v0.to(qdt), bt_d, torch.zeros(B, dtype=torch.int32, device=dev),
                         torch.from_numpy(pre_lens.astype(np.int32)).to(dev), dev_status=self.status)
            del k0, v0
            self.caches.append(cache)
            self.bts.append(bt_d)
            o = layer * per_layer
            q_l = self.in_buf[o:o + n_q].view(B, Hq, d)
            k_l = self.in_buf[o + n_q:o + n_q + n_kv].view(steps, B, 1, H, d)
            v_l = self.in_buf[o + n_q + n_kv:o + per_layer].view(steps, B, 1, H, d)
            q_l.copy_(torch.randn((B, Hq, d), generator=gen, device=dev))
            k_l.copy_(torch.randn((steps, B, 1, H, d), generator=gen, device=dev))
            v_l.copy_(torch.randn((steps, B, 1, H, d), generator=gen, device=dev))
            self.qs.append(q_l)
            self.knews.append(k_l)
            self.vnews.append(v_l)
            self.outs.append(self.out_buf[layer * n_q:(layer + 1) * n_q].view(B, Hq, d))
        base = self.lens if w.append_steps else self.lens - 1
        self.pos_list = [torch.from_numpy((base + s).astype(np.int32)).to(dev) for s in range(steps)]
        self.len_list = [torch.from_numpy((base + s + 1).astype(np.int32)).to(dev) for s in range(steps)]
        if top_k is not None:
            R = Hq if group_mode == 0 else H
            self.sel = [torch.empty((B, R, top_k), dtype=torch.int32, device=dev) for _ in range(self.layers)]
            self.cnt = [torch.empty((B, R), dtype=torch.int32, device=dev) for _ in range(self.layers)]
        torch.cuda.synchronize()
        self.steps_per_replay = steps

    def fused(self, append: bool, attention: bool, sparse: bool) -> bool:
        """Whether a step's append + attention run as one call."""
        c = self.caches[0]
        return (FUSED_APPEND and append and attention and not sparse and c.page_meta is None
                and self.w.quant != "per_group64")

    def _layer(self, i: int, s: int, stream, append=True, attention=True, sparse=False):
        c = self.caches[i]
        if self.fused(append, attention, sparse):
            # the preceding kernel (another layer's combine) touches nothing
            # this call reads or the new rows: fresh_rows = 0
            c.append_attention(self.knews[i][s][:, 0], self.vnews[i][s][:, 0], self.qs[i], self.bts[i],
                               self.len_list[s], sm_scale=self.w.sm_scale, out=self.outs[i],
                               dev_status=self.status, stream=stream, fresh_rows=0 if EARLY_START else -1)
            return
        if append:
            c.append(self.knews[i][s], self.vnews[i][s], self.bts[i], self.pos_list[s],
                     dev_status=self.status, stream=stream)
        if sparse:
            # early start: the kernel before the scoring (another layer's
            # combine) writes nothing it reads; after this step's append (which
            # refreshes the boxes) it waits
            c.score_topk(self.qs[i], self.bts[i], self.len_list[s], self.top_k, dev_status=self.status,
                         sel=self.sel[i], count=self.cnt[i], stream=stream, group_mode=self.group_mode,
                         early_start=EARLY_START and not append)
        if attention:
            # early start: after this step's append, the kernel before the
            # attention writes only the new token's rows (fresh_rows = 1); after
            # another layer's attention it writes nothing the call reads (0);
            # after the page scoring it writes only the page lists (0).
            fresh = -1 if not EARLY_START else (1 if (append and not sparse) else 0)
            c.attention(self.qs[i], self.bts[i], self.len_list[s], sm_scale=self.w.sm_scale,
                        sel=self.sel[i] if sparse else None, sel_count=self.cnt[i] if sparse else None,
                        sel_shared=sparse and self.group_mode != 0,
                        out=self.outs[i], dev_status=self.status, stream=stream, fresh_rows=fresh)

    def capture(self, append=True, attention=True, sparse=False):
        """CUDA graph of one replay: every decode step of the workload over all layers."""
        torch = self.torch
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for s in range(self.steps_per_replay):          # warm (also sizes the workspaces)
                for i in range(self.layers):
                    self._layer(i, s, stream, append, attention, sparse)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(self.steps_per_replay):
                for i in range(self.layers):
                    self._layer(i, s, torch.cuda.current_stream(), append, attention, sparse)
        torch.cuda.synchronize()
        return g, self.launches_per_replay(append, attention, sparse)

    def launches_per_replay(self, append=True, attention=True, sparse=False) -> int:
        """Kernels of libpkv launched by one replay (append: one quantise/copy kernel,
        plus the bounding-box kernel when the cache keeps page metadata; attention:
        the attention kernel and its combine kernel)."""
        per_layer = 0
        if append and not self.fused(append, attention, sparse):
            per_layer += 1 + (1 if self.caches[0].page_meta is not None else 0)
        per_layer += (1 if sparse else 0) + (2 if attention else 0)
        return self.steps_per_replay * self.layers * per_layer


def time_graph(g, replays: int, warmup: int) -> float:
    """Average device ms of one graph replay (CUDA events on the replay stream)."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / replays


def prefill_append(w: synth.Workload, with_meta: bool, peak: float) -> Dict:
    """One kv_append of the whole context (T = L tokens per sequence) into an
    empty cache, timed in a CUDA graph; bytes = K/V input read + what is stored."""
    import torch
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    dev = torch.device("cuda")
    B, H, d, T = w.batch, w.num_kv_heads, w.head_dim, int(synth.seq_lens(w).max())
    kv_name, quant_name = synth.cache_kind(w)
    qdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    bt, pool = synth.block_tables(w, 0, 1 if w.append_steps else 0)
    cache = PagedKVCache(pool, w.page_size, H, d, kv_dtype=kv_name, quant=quant_name, with_meta=with_meta,
                         tail_rows=B)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed + 7)
    k = torch.randn((B, T, H, d), generator=gen, device=dev).to(qdt)
    v = torch.randn((B, T, H, d), generator=gen, device=dev).to(qdt)
    bt_d = torch.from_numpy(bt).to(dev)
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    lens = synth.seq_lens(w)
    new_lens = torch.from_numpy(lens.astype(np.int32)).to(dev)   # each sequence's own length
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cache.append(k, v, bt_d, pos, new_lens, dev_status=status, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cache.append(k, v, bt_d, pos, new_lens, dev_status=status, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    ms = time_graph(g, 10, 3)
    toks = int(lens.sum())
    src = toks * H * d * 2 * 2
    if w.quant == "none":
        dst = src
    elif w.quant == "per_token":
        dst = toks * H * 2 * (d + 8)
    elif w.quant == "per_token_u4":
        dst = toks * H * 2 * (d // 2 + 8)
    else:
        dst = toks * H * 2 * d + (toks // 64) * H * 2 * 8
    if with_meta:
        dst += int(((lens + w.page_size - 1) // w.page_size).sum()) * H * 2 * d * 4
    byts = src + dst
    gbs = byts / (ms * 1e-3) / 1e9
    out = {"tokens": toks, "ms": round(ms, 4), "bytes": int(byts), "gb_s": round(gbs, 1),
           "frac_of_hbm_peak": round(gbs / peak, 4), "with_meta": with_meta,
           "dev_status": int(status.item())}
    del cache, k, v
    return out


def extra_workloads(peak: float) -> Dict:
    """Other workloads of the pages, one line each (not the headline)."""
    import torch
    res = {}

    def entry(name, w, ms_step, byts, steps, att_ms=None, att_bytes=None, extra=None):
        e = {"description": w.description, "ms_per_step": round(ms_step, 6),
             "gb_s": round(byts / (ms_step * 1e-3) / 1e9, 1),
             "frac_of_hbm_peak": round(byts / (ms_step * 1e-3) / 1e9 / peak, 4),
             "steps_per_s": round(steps / (ms_step * 1e-3), 1), "bytes_per_step": int(byts)}
        if att_ms is not None:
            e["attention_us"] = round(att_ms * 1e3, 2)
            e["attention_gb_s"] = round(att_bytes / (att_ms * 1e-3) / 1e9, 1)
            e["attention_frac_of_hbm_peak"] = round(att_bytes / (att_ms * 1e-3) / 1e9 / peak, 4)
        if extra:
            e.update(extra)
        res[name] = e

    # 32K dense bf16 (the >= 70 % target), W3 per-token INT8, W4 per-group INT8 +
    # append, and the W3 shapes with per-token 4-bit codes
    for name in ("dense_32k_bf16", "w3_gqa_int8_token", "w4_long_int8_group", "w7_gqa_u4_token"):
        w = synth.WORKLOADS[name]
        rep = Replica(w, w.seed)
        g, _ = rep.capture(append=True, attention=True)
        ms = time_graph(g, 20 if name != "w4_long_int8_group" else 10, 3)
        ga, _ = rep.capture(append=False, attention=True)
        ms_a = time_graph(ga, 20 if name != "w4_long_int8_group" else 10, 3)
        steps = rep.steps_per_replay
        lens = rep.lens + (w.append_steps if w.append_steps else 0) // 2
        b = algorithmic_bytes(w, lens)
        entry(name, w, ms / steps, b["total"], 1, ms_a / steps, b["attention"])
        del rep, g, ga
        torch.cuda.empty_cache()
    # W5 sparse: score + top-K (30 %) + sparse attention; and dense for comparison
    w = synth.WORKLOADS["w5_sparse_f16"]
    P = w.seq_len // w.page_size
    K = int(math.ceil(w.top_k_ratio * P))
    rep = Replica(w, w.seed, with_meta=True, top_k=K)
    gs, _ = rep.capture(append=False, attention=True, sparse=True)
    ms_s = time_graph(gs, 50, 3)
    gd, _ = rep.capture(append=False, attention=True, sparse=False)
    ms_d = time_graph(gd, 50, 3)
    bs = algorithmic_bytes(w, rep.lens, append_tokens=0, sparse_pages=K)
    bd = algorithmic_bytes(w, rep.lens, append_tokens=0)
    entry("w5_sparse_f16", w, ms_s, bs["total"], 1,
          extra={"top_k": K, "dense_us": round(ms_d * 1e3, 2),
                 "dense_gb_s": round(bd["attention"] / (ms_d * 1e-3) / 1e9, 1),
                 "sparse_speedup_vs_dense": round(ms_d / ms_s, 3),
                 "context_pages_14.2_to_4.8ms_A100": "pages' figure, context only"})
    del rep
    torch.cuda.empty_cache()
    # Bulk prefill through kv_append: T tokens per sequence written at positions
    # 0 .. T-1 in one call (copy, per-token quantise with boxes, per-group
    # quantise), as GB/s of input read + codes, scales and boxes written
    for name, with_meta in (("w2_llama7b_bf16", False), ("w6_gqa_sparse_int8", True),
                            ("w4_long_int8_group", False)):
        w = synth.WORKLOADS[name]
        res["prefill_append_" + name] = prefill_append(w, with_meta, peak)
        torch.cuda.empty_cache()
    # W6: GQA per-token INT8 with one page list per kv head (sum of the group's
    # scores), so the group's K/V pages are read once
    w = synth.WORKLOADS["w6_gqa_sparse_int8"]
    P = w.seq_len // w.page_size
    K = int(math.ceil(w.top_k_ratio * P))
    rep = Replica(w, w.seed, with_meta=True, top_k=K, group_mode=1)
    gs, _ = rep.capture(append=False, attention=True, sparse=True)
    ms_s = time_graph(gs, 30, 3)
    gd, _ = rep.capture(append=False, attention=True, sparse=False)
    ms_d = time_graph(gd, 30, 3)
    bs = algorithmic_bytes(w, rep.lens, append_tokens=0, sparse_pages=K, group_shared=True)
    bd = algorithmic_bytes(w, rep.lens, append_tokens=0)
    entry("w6_gqa_sparse_int8", w, ms_s, bs["total"], 1,
          extra={"top_k": K, "selection": "group sum", "dense_us": round(ms_d * 1e3, 2),
                 "dense_gb_s": round(bd["attention"] / (ms_d * 1e-3) / 1e9, 1),
                 "sparse_speedup_vs_dense": round(ms_d / ms_s, 3)})
    del rep
    torch.cuda.empty_cache()
    return res


def sweep(peak: float) -> Dict:
    """Attention call time over batch x context for the Llama-2-7B head shapes (32 q
    heads over 32 or 8 kv heads, d = 128, page 16): bf16 caches, then per-token INT8
    caches with 8 kv heads (the GQA INT8 workload's quantisation and outliers). Each
    point is a chain of attention calls over distinct layers (early start, as in the
    bench's step), with enough layers that the chain's K/V exceed L2; points whose
    layer exceeds 4.3 GB (bf16) or 2.2 GB (INT8) are skipped."""
    import dataclasses as dc
    import torch
    res = []
    families = [("bf16", synth.WORKLOADS["w2_llama7b_bf16"], hkv, 2 * 128 * 2, 4.3e9, 1.0e9, 32)
                for hkv in (32, 8)]
    families.append(("int8 per-token", synth.WORKLOADS["w3_gqa_int8_token"], 8, (128 + 16) * 2, 2.2e9, 0.6e9, 16))
    for cache, base, hkv, bytes_per_token_head, max_layer, chain_bytes, max_layers in families:
        for B in (1, 4, 16, 64):
            for L in (1024, 4096, 16384, 32768):
                per_layer = B * L * hkv * bytes_per_token_head
                if per_layer > max_layer:
                    continue
                layers = int(min(max_layers, max(2, math.ceil(chain_bytes / per_layer))))
                w = dc.replace(base, name="sweep", batch=B, num_kv_heads=hkv, seq_len=L, seq_len_range=None,
                               layers=layers, pool_pages=None, description="")
                rep = Replica(w, w.seed, layers=layers)
                ga, _ = rep.capture(append=False, attention=True)
                ms = time_graph(ga, 20, 3) / layers
                byts = algorithmic_bytes(w, rep.lens, append_tokens=0)["attention"]
                res.append({"cache": cache, "kv_heads": hkv, "batch": B, "seq_len": L, "layers": layers,
                            "attention_us": round(ms * 1e3, 2),
                            "gb_s": round(byts / (ms * 1e-3) / 1e9, 1),
                            "frac_of_hbm_peak": round(byts / (ms * 1e-3) / 1e9 / peak, 4)})
                del rep, ga
                torch.cuda.empty_cache()
    return {"metric": "attention call GB/s over batch x context (32 q heads, d 128, page 16)",
            "peak_gbs": peak, "points": res}


def prefill_once() -> None:
    """One bulk kv_append of the whole context, no timing (a short command for
    profilers): per-token INT8 with page boxes at the sparse GQA INT8
    workload's shapes, then per-64-token-group INT8 at the long-context ones."""
    import torch
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    for name, meta in (("w6_gqa_sparse_int8", True), ("w4_long_int8_group", False)):
        w = synth.WORKLOADS[name]
        B, H, d, T = w.batch, w.num_kv_heads, w.head_dim, int(synth.seq_lens(w).max())
        kv_name, quant_name = synth.cache_kind(w)
        bt, pool = synth.block_tables(w, 0, 1 if w.append_steps else 0)
        cache = PagedKVCache(pool, w.page_size, H, d, kv_dtype=kv_name, quant=quant_name, with_meta=meta,
                             tail_rows=B)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(w.seed + 7)
        k = torch.randn((B, T, H, d), generator=gen, device="cuda").half()
        v = torch.randn((B, T, H, d), generator=gen, device="cuda").half()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        cache.append(k, v, torch.from_numpy(bt).cuda(), torch.zeros(B, dtype=torch.int32, device="cuda"),
                     dev_status=st)
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        del cache, k, v
        torch.cuda.empty_cache()


def sparse_breakdown(peak: float) -> List[Dict]:
    """Where a sparse decode step's time goes: the step (page scoring + top-K +
    sparse attention) with and without the attention's early start, the scoring
    alone, the sparse attention alone, and dense attention over all pages, for
    the fp16 per-head-list and the GQA INT8 group-sum workloads."""
    import torch
    global EARLY_START
    res = []
    saved = EARLY_START
    for name, gm in (("w5_sparse_f16", 0), ("w6_gqa_sparse_int8", 1)):
        w = synth.WORKLOADS[name]
        P = w.seq_len // w.page_size
        K = int(math.ceil(w.top_k_ratio * P))
        rep = Replica(w, w.seed, with_meta=True, top_k=K, group_mode=gm)
        r = {"workload": name}
        for early in (False, True):
            EARLY_START = early
            g, _ = rep.capture(append=False, attention=True, sparse=True)
            r[f"step_us_early{int(early)}"] = round(time_graph(g, 50, 5) * 1e3, 2)
        EARLY_START = saved
        c = rep.caches[0]

        def score_only():
            c.score_topk(rep.qs[0], rep.bts[0], rep.len_list[0], K, dev_status=rep.status, sel=rep.sel[0],
                         count=rep.cnt[0], stream=torch.cuda.current_stream(), group_mode=gm,
                         early_start=EARLY_START)

        def attention_only():
            c.attention(rep.qs[0], rep.bts[0], rep.len_list[0], sm_scale=w.sm_scale, sel=rep.sel[0],
                        sel_count=rep.cnt[0], sel_shared=gm != 0, out=rep.outs[0], dev_status=rep.status,
                        stream=torch.cuda.current_stream(), fresh_rows=0)

        for label, fn in (("score_us", score_only), ("attention_us", attention_only)):
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                fn()
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(10):
                    fn()
            torch.cuda.synchronize()
            r[label] = round(time_graph(g, 20, 3) / 10 * 1e3, 2)
        gd, _ = rep.capture(append=False, attention=True, sparse=False)
        r["dense_us"] = round(time_graph(gd, 50, 5) * 1e3, 2)
        b = algorithmic_bytes(w, rep.lens, append_tokens=0, sparse_pages=K, group_shared=gm != 0)
        r["step_frac_early1"] = round(b["total"] / (r["step_us_early1"] * 1e-6) / 1e9 / peak, 4)
        r["attention_frac"] = round(b["attention"] / (r["attention_us"] * 1e-6) / 1e9 / peak, 4)
        r["score_frac"] = round(b["score"] / (r["score_us"] * 1e-6) / 1e9 / peak, 4)
        r["gap_us"] = round(r["step_us_early1"] - r["score_us"] - r["attention_us"], 2)
        res.append(r)
        del rep
        torch.cuda.empty_cache()
    return res


# -------------------------------------------------------------- CPU baseline
# The oracle (fp64 NumPy, test infrastructure) timed on the host cores, per
# workload, on bounded samples. A unit is one (layer, sequence, query head):
# the oracle restores that query head's K/V from the stored form (INT8 codes,
# scales and zero-points precomputed with the oracle's quantiser, as the cache
# holds them), and runs its attention; for the sparse workload it also scores
# the pages from their boxes (precomputed, as the cache keeps them), selects
# the top-K and attends over them. Only that arithmetic is timed; seeded input
# generation and the stored-form preparation are not.
CPU_BASELINE_WORKLOADS = ("w1_tiny_f16", "w2_llama7b_bf16", "w3_gqa_int8_token",
                          "w4_long_int8_group", "w5_sparse_f16", "dense_32k_bf16")
_SEQ_CACHE: Dict = {}


def _stored_kv(name: str, layer: int, b: int, g: int):
    """(what the oracle restores from, K/V of kv head g of sequence b) kept per
    worker for the sequences it samples."""
    import oracle
    key = (name, layer, b, g)
    if key in _SEQ_CACHE:
        return _SEQ_CACHE[key]
    if len(_SEQ_CACHE) > 8:
        _SEQ_CACHE.clear()
    w = synth.WORKLOADS[name]
    L = int(synth.seq_lens(w)[b])
    sd = synth.seq_tokens(w, b, layer, L)
    k, v = sd.k[:, g:g + 1].copy(), sd.v[:, g:g + 1].copy()
    del sd
    if w.quant == "per_token":
        stored = (oracle.quantize_per_token(k), oracle.quantize_per_token(v))
    elif w.quant == "per_token_u4":
        stored = (oracle.quantize_per_token_u4(k), oracle.quantize_per_token_u4(v))
    elif w.quant == "per_group64":
        stored = (oracle.quantize_per_group(k), oracle.quantize_per_group(v))
    else:
        stored = (k, v)
    meta = oracle.page_bounding_boxes(k, w.page_size) if w.top_k_ratio else None
    _SEQ_CACHE[key] = (stored, meta, synth.queries(w, layer)[1])
    return _SEQ_CACHE[key]


def _oracle_units(args):
    """Oracle arithmetic of the given (layer, sequence, query head) units in this
    worker; returns (seconds of oracle arithmetic, units)."""
    name, units = args
    import oracle
    from oracle.quant import per_group_dequant, per_token_dequant
    w = synth.WORKLOADS[name]
    t_total = 0.0
    for layer, b, h in units:
        g = h // w.group
        stored, meta, qf = _stored_kv(name, layer, b, g)
        t0 = time.perf_counter()
        if w.quant == "per_token":
            k = per_token_dequant(*stored[0])[:, 0]
            v = per_token_dequant(*stored[1])[:, 0]
        elif w.quant == "per_token_u4":
            k = oracle.per_token_u4_dequant(*stored[0])[:, 0]
            v = oracle.per_token_u4_dequant(*stored[1])[:, 0]
        elif w.quant == "per_group64":
            k = per_group_dequant(*stored[0])[:, 0]
            v = per_group_dequant(*stored[1])[:, 0]
        else:
            k, v = stored[0][:, 0], stored[1][:, 0]
        if meta is None:
            oracle.decode_attention_tokens(qf[b, h], k, v, w.sm_scale)
        else:
            mn, mx = meta
            r = oracle.page_scores(qf[b, h:h + 1], mn, mx, 1)[0]
            K = oracle.top_k_count(w.top_k_ratio, r.shape[0])
            pages = oracle.select_top_k(r, K)
            oracle.sparse_decode_attention(qf[b, h:h + 1], k[:, None], v[:, None], w.sm_scale, [pages],
                                           w.page_size)
        t_total += time.perf_counter() - t0
    return t_total, len(units)


def _oracle_pool(workers: int):
    """Spawned single-threaded workers (BLAS threads pinned to one)."""
    import multiprocessing as mp
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        return mp.get_context("spawn").Pool(workers)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def step_bytes_of(w: synth.Workload) -> int:
    """Algorithmic bytes of one step of the workload (as the GPU arm counts them)."""
    lens = synth.seq_lens(w)
    if w.top_k_ratio:
        K = int(math.ceil(w.top_k_ratio * -(-int(lens.max()) // w.page_size)))
        return algorithmic_bytes(w, lens, append_tokens=0, sparse_pages=K)["total"] * w.layers
    return algorithmic_bytes(w, lens, append_tokens=1 if w.append_steps else 0)["total"] * w.layers


class OracleSampler:
    """Times oracle units of one workload on a pool of spawned single-threaded
    workers. Worker c takes units of one sequence (the first or the last of the
    batch, alternating) and of one kv head's query heads, so it restores one
    kv head's K/V (generated once per worker)."""

    def __init__(self, name: str, pool, workers: int):
        self.name, self.pool, self.workers = name, pool, workers
        w = synth.WORKLOADS[name]
        self.units_per_step = w.layers * w.batch * w.num_q_heads
        self.step_bytes = step_bytes_of(w)

    def run(self, units_per_worker: int, seed: int):
        """One sample; returns (units, seconds) where seconds is the slowest
        worker's oracle time (the workers run at once)."""
        w = synth.WORKLOADS[self.name]
        rng = np.random.default_rng(seed)
        seqs = [(0, 0), (w.layers - 1, w.batch - 1)]
        jobs = []
        for c in range(self.workers):
            layer, b = seqs[c % 2]
            g = (c // 2) % w.num_kv_heads
            hs = g * w.group + rng.integers(0, w.group, size=units_per_worker)
            jobs.append((self.name, [(layer, b, int(h)) for h in hs]))
        res = self.pool.map(_oracle_units, jobs, chunksize=1)
        return sum(r[1] for r in res), max(r[0] for r in res)

    def measure(self, budget_s: float) -> Dict:
        """About budget_s of oracle time per worker; GB/s of the workload's
        algorithmic bytes at the sampled rate of units."""
        self.run(1, 0)                                   # warm: imports, inputs
        n, t = self.run(1, 0)
        per_unit = max(t, 1e-6)
        upw = int(max(1, min(4000, budget_s / per_unit)))
        units, secs = self.run(upw, 2)
        rate = units / secs                               # units per second
        ms_step = self.units_per_step / rate * 1e3
        return {"gb_s": round(self.step_bytes / (ms_step * 1e-3) / 1e9, 4), "cores": self.workers,
                "est_ms_per_step": round(ms_step, 3), "units_timed": units, "seconds": round(secs, 3)}


def cpu_baseline(name: str, budget_s: float = 1.5) -> Dict:
    """The oracle on the host cores, single core and all cores, for the headline
    workload (top-level keys) and for every workload of the pages (per_config)."""
    cores = os.cpu_count() or 1
    single, multi = _oracle_pool(1), _oracle_pool(cores)
    per = {}
    try:
        for wname in CPU_BASELINE_WORKLOADS:
            per[wname] = {"single_core": OracleSampler(wname, single, 1).measure(budget_s),
                          "all_cores": OracleSampler(wname, multi, cores).measure(budget_s)}
    finally:
        for pool in (single, multi):
            pool.close()
            pool.join()
    head = per.get(name) or per["w2_llama7b_bf16"]
    return {"value": head["all_cores"]["gb_s"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_core": {"value": head["single_core"]["gb_s"], "cores": 1},
            "sample": f"per workload, about {budget_s} s of oracle arithmetic per worker on one "
                      f"single-threaded spawned worker (single_core) and on {cores} (all_cores); a unit "
                      f"is one (layer, sequence, query head): restore its K/V from the stored form and "
                      f"attend (sparse: score the page boxes, select the top-K, attend); GB/s = the "
                      f"workload's algorithmic bytes per step / (units per step / units per second); "
                      f"seeded input generation and the stored-form preparation are not timed",
            "per_config": per}


# ------------------------------------------------------------------- arms
def run_ours(args) -> None:
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_243_gb300 import _build
    _build.build()
    peaks = load_peaks()
    peak = peaks["hbm_gbs"]
    w = synth.WORKLOADS[args.workload]
    rep = Replica(w, rank_seed(w.seed, rank))
    g, launches_per_step = rep.capture(append=True, attention=True)
    lens = rep.lens
    byts = algorithmic_bytes(w, lens)
    step_bytes = byts["total"] * rep.layers
    K, W = args.steps, args.warmup

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(W):
        g.replay()
    barrier()
    with ClockSampler(dev.index) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        barrier()
    ms_local = e0.elapsed_time(e1) / K
    ms = reduce_max(ms_local, world, dev)
    total_bytes = reduce_sum(float(step_bytes), world, dev)
    value = total_bytes / (ms * 1e-3) / 1e9
    clocks = clk.summary()
    status = int(rep.status.item())

    # dominant kernel: the attention launch (graph of the 32 attention calls only)
    ga, _ = rep.capture(append=False, attention=True)
    ms_att = time_graph(ga, max(20, K // 10), 3) / rep.layers
    att_bytes = byts["attention"]
    achieved = att_bytes / (ms_att * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)

    # end to end through the C ABI with host buffers: per step, the pinned host
    # inputs of all layers (q, new K, new V) go host->device in one copy, the 32
    # layers run, the outputs of all layers come back in one copy, and the host
    # waits for them (the step is one captured graph)
    h_in = rep.in_buf.cpu().pin_memory()
    h_out = rep.out_buf.cpu().pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    ge = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(ge, stream=cap):
        st = torch.cuda.current_stream()
        rep.in_buf.copy_(h_in, non_blocking=True)
        for i in range(rep.layers):
            rep._layer(i, 0, st)
        h_out.copy_(rep.out_buf, non_blocking=True)
    torch.cuda.synchronize()
    for _ in range(3):
        ge.replay()
        torch.cuda.synchronize()
    n_e2e = max(10, min(K, 500))
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        ge.replay()
        torch.cuda.synchronize()
    ms_e2e = (time.perf_counter() - t0) * 1e3 / n_e2e
    ms_e2e = reduce_max(ms_e2e, world, dev)
    e2e = {"value": round(total_bytes / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
           "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
           "how": "per step: one graph replay (one copy of all layers' pinned-host q and new K/V "
                  "tokens in, the step's C-ABI calls for every layer (as in the timed step: one "
                  "append_decode_attention per layer, or kv_append + paged_decode_attention where "
                  "that path is off), one copy of all outputs to pinned host memory) then a host "
                  "wait for the outputs; host clock"}

    extras = None
    del ga, ge
    if rank == 0 and not args.no_extras:
        extras = extra_workloads(peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)

    if rank == 0:
        line = {
            "metric": "paged decode-attention KV GB/s", "value": round(value, 1), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f16",
            "data": "synthetic (seeded device RNG, N(0,1) rounded to the cache dtype)",
            "config": {"workload": w.name, "description": w.description, "batch": w.batch,
                       "layers": rep.layers, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                       "seq_len": int(lens.max()), "page_size": w.page_size,
                       "step": ("per layer: append of 1 token per sequence + dense attention, "
                                "as one append_decode_attention call" if rep.fused(True, True, False) else
                                "per layer: kv_append of 1 token per sequence + dense "
                                "paged_decode_attention") + "; all layers in one CUDA graph",
                       "l2": "inputs larger than L2 (KV per step >> 129 MB), no flush"},
            "steps_per_s": round(1e3 / ms * world, 2),
            "frac_of_hbm_peak": round(value / world / peak, 4),
            "bytes_per_step": int(step_bytes),
            "gpu_launches": int(launches_per_step * K),
            "gpu_launches_per_step": int(launches_per_step),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_source": peaks["source"],
                         "kernel": "paged_attention_kernel (one launch per layer)",
                         "early_start": EARLY_START,
                         "algorithmic_bytes_per_launch": int(att_bytes),
                         "avg_launch_us": round(ms_att * 1e3, 3)},
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "dev_status": status,
            "workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args) -> None:
    """The oracle as the reference arm: each step is a bounded sample of the
    workload (a few (layer, sequence, query head) units per host core), sized so
    the whole run takes minutes; ms_per_step is the measured time of one such
    sample step, and the value is the GB/s of the workload's algorithmic bytes
    at the sampled rate of units."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    pool = _oracle_pool(cores)
    smp = OracleSampler(args.workload, pool, cores)
    try:
        smp.run(1, 0)
        upw = 8
        units, secs = 0, 0.0
        for i in range(args.warmup + args.steps):
            n, t = smp.run(upw, 1 + i)
            if i >= args.warmup:
                units += n
                secs += t
    finally:
        pool.close()
        pool.join()
    rate = units / secs if secs > 0 else 0.0
    value = smp.step_bytes * rate / smp.units_per_step / 1e9 if rate > 0 else 0.0
    ms_sample = secs / max(1, args.steps) * 1e3
    cb = {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
          "sample": f"per step {upw} (layer, sequence, query head) units on each of {cores} single-threaded "
                    f"spawned workers ({upw * cores} units) of {args.workload}; fp64 numpy oracle; "
                    f"{args.steps} timed steps"}
    line = {"impl": "reference", "metric": "paged decode-attention KV GB/s", "value": round(value, 4),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_sample, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy generators)",
            "config": {"workload": w.name, "description": w.description,
                       "step": f"a sample of {upw * cores} units of the workload (its "
                               f"{smp.units_per_step} units take {smp.units_per_step / max(rate, 1e-9) * 1e3:.1f} ms "
                               f"at the sampled rate)"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv: Optional[List[str]] = None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-early-start", action="store_true",
                    help="attention waits for the preceding kernel before any read (fresh_rows = -1)")
    ap.add_argument("--no-fused-append", action="store_true",
                    help="the step's append is a separate kv_append launch")
    ap.add_argument("--sweep", action="store_true",
                    help="print attention call times over batch x context instead of the bench line")
    ap.add_argument("--sparse-breakdown", action="store_true",
                    help="print where the sparse decode steps' time goes instead of the bench line")
    ap.add_argument("--prefill-once", action="store_true",
                    help="run one bulk append of the INT8 GQA shapes, untimed (for profilers)")
    args = ap.parse_args(argv)
    global EARLY_START, FUSED_APPEND
    EARLY_START = not args.no_early_start
    FUSED_APPEND = not args.no_fused_append
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.sweep or args.sparse_breakdown or args.prefill_once:
        import torch
        from paged_kv_cache_243_gb300 import _build
        _build.build()
        torch.cuda.set_device(0)
        if args.sweep:
            print(json.dumps(sweep(load_peaks()["hbm_gbs"])), flush=True)
        elif args.sparse_breakdown:
            for r in sparse_breakdown(load_peaks()["hbm_gbs"]):
                print(json.dumps(r), flush=True)
        else:
            prefill_once()
            print("ok", flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
