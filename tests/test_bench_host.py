"""Host-side logic of bench.py without a GPU: byte accounting and the
multi-rank reductions (two gloo ranks on CPU)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as tmp

import bench
import oracle
import synth


def test_step_bytes_match_the_pages_arithmetic():
    w = synth.WORKLOADS["w2_llama7b_bf16"]
    b = bench.algorithmic_bytes(w, synth.seq_lens(w), append_tokens=0)
    kv = oracle.kv_cache_bytes(1, w.batch, w.num_kv_heads, 2048, w.head_dim, 2)
    # K/V of every token plus q, output and block-table entries
    assert b["attention"] == kv + w.batch * w.num_q_heads * w.head_dim * 4 + w.batch * 128 * 4
    assert kv * 32 == oracle.kv_cache_bytes(32, 4, 32, 2048, 128, 2) == 4294967296


def test_int8_per_token_bytes_per_token():
    w = synth.WORKLOADS["w3_gqa_int8_token"]
    lens = np.array([1000], dtype=np.int32)
    w1 = synth.scaled(w, batch=1)
    b = bench.algorithmic_bytes(w1, lens, append_tokens=0)
    fixed = 1 * w.num_q_heads * w.head_dim * 4 + (1000 + 15) // 16 * 4
    assert b["attention"] - fixed == 1000 * 2176          # 2 x 128 codes + 16 B scales, 8 kv heads


def test_sparse_bytes():
    w = synth.WORKLOADS["w5_sparse_f16"]
    b = bench.algorithmic_bytes(w, synth.seq_lens(w), append_tokens=0, sparse_pages=308)
    assert b["score"] >= 64 * 2**20                       # page boxes: 8 x 16 x 1024 x 512 B
    kv = 8 * 16 * 308 * 16 * 64 * 2 * 2
    assert b["attention"] >= kv


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsz, lr = bench.dist_env()
    t = bench.reduce_max(1.5 + rank, wsz)          # per-rank step time; the max wins
    s = bench.reduce_sum(100.0 * (rank + 1), wsz)  # per-rank bytes; the sum is the job's
    q.put((r, wsz, lr, t, s, bench.rank_seed(7, r)))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == 2.5 for r in res)            # max over ranks
    assert all(r[4] == 300.0 for r in res)          # whole-job bytes
    assert res[0][5] == 7 and res[1][5] != 7        # ranks draw different replicas
