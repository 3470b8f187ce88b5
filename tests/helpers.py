"""Test helpers: load seeded workloads into the CUDA path and into the oracle.

Inputs come from `synth` only; expected values come from `oracle` only. The
GPU pools are read back and gathered through the block table by plain numpy
indexing here, never fed to the oracle.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle
import synth
from oracle.quant import (per_group_bbox_values, per_group_dequant, per_token_bbox_values,
                          per_token_dequant)
from oracle.quant4 import per_token_u4_bbox_values, per_token_u4_dequant

# Tolerances on attention outputs (max-abs, fp32 outputs), per input precision.
TOL = {"bf16": 2e-3, "f16": 1e-3, "int8": 1e-3}


def set_knobs(monkeypatch, **env) -> None:
    """Set PKV_ATTN_* tuning variables for one test and make the library re-read
    them (it reads them once per process otherwise); the conftest fixture
    re-reads them after the test, once monkeypatch has restored the environment."""
    from paged_kv_cache_243_gb300 import binding as B
    for k, v in env.items():
        monkeypatch.setenv(k, str(v))
    B.tuning_reload()


def torch_dtype(name: str):
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


def bits_to_torch(bits: np.ndarray, name: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch_dtype(name))


@dataclasses.dataclass
class Loaded:
    w: synth.Workload
    cache: object
    bt: np.ndarray          # int32 [B][max_pages]
    lens: np.ndarray        # int32 [B]
    seqs: List[synth.SeqData]
    bt_dev: torch.Tensor
    lens_dev: torch.Tensor
    status: torch.Tensor


def load_workload(w: synth.Workload, layer: int = 0, lens: Optional[np.ndarray] = None,
                  with_meta: bool = False, extra_pages: int = 0, poison: bool = True,
                  chunks: Optional[Sequence[int]] = None) -> Loaded:
    """Generate a workload's tokens and write them into a fresh cache with kv_append.

    chunks: append in several calls of these token counts (default: one call).
    """
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    if lens is None:
        lens = synth.seq_lens(w)
        bt, pool = synth.block_tables(w, layer, extra_pages)
    else:
        lens = np.asarray(lens, dtype=np.int32)
        bt, pool = _block_tables(w, lens, layer, extra_pages)
    lens = np.asarray(lens, dtype=np.int32)
    kv_name, quant_name = synth.cache_kind(w)
    cache = PagedKVCache(pool, w.page_size, w.num_kv_heads, w.head_dim, kv_dtype=kv_name,
                         quant=quant_name, with_meta=with_meta, tail_rows=w.batch, poison=poison)
    seqs = [synth.seq_tokens(w, b, layer, int(lens[b])) for b in range(w.batch)]
    bt_dev = torch.from_numpy(bt).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    T = int(lens.max()) if len(lens) else 0
    if chunks is None:
        chunks = [T]
    pos = 0
    for n in chunks:
        if pos >= T:
            break
        n = min(n, T - pos)
        kb = np.zeros((w.batch, n, w.num_kv_heads, w.head_dim), dtype=np.uint16)
        vb = np.zeros_like(kb)
        nl = np.zeros(w.batch, dtype=np.int32)
        for b, sd in enumerate(seqs):
            m = max(0, min(n, int(lens[b]) - pos))
            kb[b, :m] = sd.k_bits[pos:pos + m]
            vb[b, :m] = sd.v_bits[pos:pos + m]
            nl[b] = m
        cache.append(bits_to_torch(kb, w.dtype).cuda(), bits_to_torch(vb, w.dtype).cuda(), bt_dev,
                     torch.from_numpy(np.minimum(lens, pos).astype(np.int32)).cuda(),
                     torch.from_numpy(nl).cuda(), dev_status=status)
        pos += n
    torch.cuda.synchronize()
    return Loaded(w, cache, bt, lens, seqs, bt_dev, torch.from_numpy(lens).cuda(), status)


def _block_tables(w, lens, layer, extra_pages):
    ps = w.page_size
    need = [-(-int(L) // ps) + extra_pages for L in lens]
    max_pages = max(1, max(need))
    rng = np.random.default_rng([w.seed, 5, layer, len(lens)])
    total = sum(need)
    pool = max(total + w.pool_spare, w.pool_pages or 0, 1)
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, pool


def gather(pool: np.ndarray, bt_row: np.ndarray, L: int, ps: int) -> np.ndarray:
    """Logical tokens [L][Hkv][...] of one sequence from a pool [pages][Hkv][ps][...]."""
    t = np.arange(L)
    return pool[bt_row[t // ps], :, t % ps]


def oracle_kv(ld: Loaded, b: int):
    """Oracle K, V (fp64, logical order) of sequence b as attention must see them."""
    w, sd = ld.w, ld.seqs[b]
    if w.quant == "none":
        return sd.k.astype(np.float64), sd.v.astype(np.float64)
    if w.quant == "per_token":
        kc, ks, kz = oracle.quantize_per_token(sd.k)
        vc, vs, vz = oracle.quantize_per_token(sd.v)
        return per_token_dequant(kc, ks, kz), per_token_dequant(vc, vs, vz)
    if w.quant == "per_token_u4":
        return (per_token_u4_dequant(*oracle.quantize_per_token_u4(sd.k)),
                per_token_u4_dequant(*oracle.quantize_per_token_u4(sd.v)))
    kc, ks, kz = oracle.quantize_per_group(sd.k)
    vc, vs, vz = oracle.quantize_per_group(sd.v)
    return per_group_dequant(kc, ks, kz), per_group_dequant(vc, vs, vz)


def oracle_bbox_keys(w, sd: synth.SeqData) -> np.ndarray:
    """fp32 key values the page bounding boxes are built from."""
    if w.quant == "none":
        return sd.k
    if w.quant == "per_token":
        kc, ks, kz = oracle.quantize_per_token(sd.k)
        return per_token_bbox_values(kc, ks, kz)
    if w.quant == "per_token_u4":
        return per_token_u4_bbox_values(*oracle.quantize_per_token_u4(sd.k))
    kc, ks, kz = oracle.quantize_per_group(sd.k)
    return per_group_bbox_values(kc, ks, kz)


def queries_dev(w, layer=0, step=0):
    qb, qf = synth.queries(w, layer, step)
    return bits_to_torch(qb, w.dtype).cuda(), qf


def oracle_dense(ld: Loaded, qf: np.ndarray, units=None) -> dict:
    """Oracle outputs {(b, h): [d]} for the listed (b, h) (default: all)."""
    w = ld.w
    G = w.group
    res = {}
    want = units if units is not None else [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    by_b = {}
    for b, h in want:
        by_b.setdefault(b, []).append(h)
    for b, hs in by_b.items():
        k, v = oracle_kv(ld, b)
        for h in hs:
            g = h // G
            res[(b, h)] = oracle.decode_attention_tokens(qf[b, h], k[:, g, :], v[:, g, :], w.sm_scale)
    return res


def max_abs_err(gpu_out: np.ndarray, ref: dict) -> float:
    return max(float(np.abs(gpu_out[b, h].astype(np.float64) - o).max()) for (b, h), o in ref.items())


def int8_codes(pool_bytes: np.ndarray) -> np.ndarray:
    """INT8 codes (the oracle's c in [-128, 127]) from stored bytes u = c + 128."""
    return (pool_bytes.astype(np.int16) - 128).astype(np.int8)


def pools(ld):
    c = ld.cache
    return (c.k_pages.cpu().numpy(), c.v_pages.cpu().numpy(), c.kv_sz.cpu().numpy())


def check_per_token_codes(ld):
    kp, vp, sz = pools(ld)
    ps = ld.w.page_size
    for b in range(ld.w.batch):
        L = int(ld.lens[b])
        for x, pool, col in ((ld.seqs[b].k, kp, 0), (ld.seqs[b].v, vp, 2)):
            c, s, z = oracle.quantize_per_token(x)
            assert np.array_equal(int8_codes(gather(pool, ld.bt[b], L, ps)), c)
            g = gather(sz, ld.bt[b], L, ps)             # [L][Hkv][4]
            assert np.array_equal(g[:, :, col].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(g[:, :, col + 1].view(np.uint32), z.view(np.uint32))


def check_per_group_codes(ld):
    kp, vp, sz = pools(ld)
    ps = ld.w.page_size
    for b in range(ld.w.batch):
        L = int(ld.lens[b])
        for x, pool, col in ((ld.seqs[b].k, kp, 0), (ld.seqs[b].v, vp, 2)):
            c, s, z = oracle.quantize_per_group(x)
            assert np.array_equal(int8_codes(gather(pool, ld.bt[b], L, ps)), c)
            ng = s.shape[0]
            t0 = np.arange(ng) * 64
            gs = sz[ld.bt[b][t0 // ps], :, (t0 % ps) // 64]   # [ng][Hkv][4]
            assert np.array_equal(gs[:, :, col].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(gs[:, :, col + 1].view(np.uint32), z.view(np.uint32))


def check_per_token_u4_codes(ld):
    """Packed 4-bit codes, scales and zero-points bit-exact against the oracle's
    quantiser, gathered through the block table."""
    kp, vp, sz = pools(ld)
    ps = ld.w.page_size
    for b in range(ld.w.batch):
        L = int(ld.lens[b])
        for x, pool, col in ((ld.seqs[b].k, kp, 0), (ld.seqs[b].v, vp, 2)):
            c, s, z = oracle.quantize_per_token_u4(x)
            assert np.array_equal(gather(pool, ld.bt[b], L, ps), oracle.pack_u4(c))
            g = gather(sz, ld.bt[b], L, ps)
            assert np.array_equal(g[:, :, col].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(g[:, :, col + 1].view(np.uint32), z.view(np.uint32))
