"""The N-GPU layout on CPU: two gloo ranks each verify their own shard of the
global batch (no collective in the data path); the shards' results equal the
single-process result over the whole batch, and the timing reduction takes the
slowest rank."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
import oracle
import specgen as sg


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, B, out_q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = sg.CONFIGS["cfg2_v32000_bf16"].with_(B=B, V=700)
        d = sg.sample_inputs(cfg, seq_offset=bench.shard_offset(rank, B))
        toks, acc, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                            cfg.temperature, cfg.top_p)
        g = sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=B, V=300)
        gd = sg.greedy_inputs(g, seq_offset=bench.shard_offset(rank, B))
        gt, ga, _ = oracle.verify_greedy(gd["logits"], gd["cand"])
        la = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"].with_(B=B, V=400, temperature=0.5)
        ld = sg.lookahead_sample_inputs(la, seq_offset=bench.shard_offset(rank, B))
        lt, lacc, _, _ = oracle.verify_lookahead_sample(ld["logits"], ld["cand"], ld["uniforms"], la.temperature)
        slowest = bench.max_over_ranks(10.0 + rank)
        parts = [None] * world
        dist.all_gather_object(parts, (rank, toks, acc, gt, ga, slowest, lt, lacc))
        if rank == 0:
            out_q.put(parts)
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_equal_the_global_batch():
    world, B = 2, 6
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, B, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    parts.sort(key=lambda x: x[0])
    assert all(x[5] == 11.0 for x in parts)  # max over ranks
    cfg = sg.CONFIGS["cfg2_v32000_bf16"].with_(B=world * B, V=700)
    d = sg.sample_inputs(cfg)
    toks, acc, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                        cfg.temperature, cfg.top_p)
    np.testing.assert_array_equal(np.concatenate([x[1] for x in parts]), toks)
    np.testing.assert_array_equal(np.concatenate([x[2] for x in parts]), acc)
    g = sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=world * B, V=300)
    gd = sg.greedy_inputs(g)
    gt, ga, _ = oracle.verify_greedy(gd["logits"], gd["cand"])
    np.testing.assert_array_equal(np.concatenate([x[3] for x in parts]), gt)
    np.testing.assert_array_equal(np.concatenate([x[4] for x in parts]), ga)
    la = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"].with_(B=world * B, V=400, temperature=0.5)
    ld = sg.lookahead_sample_inputs(la)
    lt, lacc, _, _ = oracle.verify_lookahead_sample(ld["logits"], ld["cand"], ld["uniforms"], la.temperature)
    np.testing.assert_array_equal(np.concatenate([x[6] for x in parts]), lt)
    np.testing.assert_array_equal(np.concatenate([x[7] for x in parts]), lacc)
