"""World-size-2 tests of the multi-rank host logic on CPU (gloo).

* Data parallel over tokens (what `bench.py --gpus N` runs): each rank
  processes its own tokens; the forward needs no collective, and the
  concatenation of the ranks' outputs equals the single-process forward.
* Expert parallel (the pages' ep4 runs; `group_offset` / `E_local`): each rank
  computes gmm for its shard of experts, rows of other experts come out zero,
  and the sum over ranks equals the whole grouped matmul.
* Timing: the bench reports the max over ranks (all_reduce MAX)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # ---- data parallel forward: tokens split across ranks
        cfg = synth.scaled(synth.CONFIGS["tiny"], T=64)
        x = oracle.bf16_bits(synth.activations(cfg, 0))
        ids, w = synth.routing(cfg, 0)
        w_in, w_out = synth.expert_weights(cfg, 0)
        wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode)
        sl = slice(rank * cfg.T // world, (rank + 1) * cfg.T // world)
        y_local = oracle.ffn_forward(np.ascontiguousarray(x[sl]), np.ascontiguousarray(ids[sl]),
                                     np.ascontiguousarray(w[sl]), wq, cfg.E, cfg.act_mode)["y"]
        t = torch.from_numpy(y_local.astype(np.int32))
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        y_dp = torch.cat(parts).numpy().astype(np.uint16)

        # ---- expert parallel gmm: experts split across ranks, outputs summed
        rng = np.random.default_rng(3)
        E, M, K, N = 6, 300, 256, 128
        sizes = np.array([40, 0, 90, 70, 50, 50], np.int32)
        a = (rng.integers(0, 0x7F, (M, K)).astype(np.uint8)) | (rng.integers(0, 2, (M, K)).astype(np.uint8) << 7)
        wts = rng.integers(0, 0x7F, (E, N, K)).astype(np.uint8)
        sa = rng.uniform(0.5, 2, M).astype(np.float32) / 448
        sw = rng.uniform(0.5, 2, (E, N)).astype(np.float32) / 448
        per = E // world
        g0 = rank * per
        part = oracle.gmm(a, sa, 0, wts[g0:g0 + per], sw[g0:g0 + per], 0, sizes, group_offset=g0, E_local=per,
                          want="f64")
        summed = torch.from_numpy(part)
        dist.all_reduce(summed, op=dist.ReduceOp.SUM)

        # ---- max-over-ranks timing
        ms = torch.tensor([1.0 + rank])
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
        if rank == 0:
            np.save(os.path.join(out_dir, "y_dp.npy"), y_dp)
            np.save(os.path.join(out_dir, "ep.npy"), summed.numpy())
            np.save(os.path.join(out_dir, "ms.npy"), ms.numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_data_and_expert_parallel(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    # single-process references
    cfg = synth.scaled(synth.CONFIGS["tiny"], T=64)
    x = oracle.bf16_bits(synth.activations(cfg, 0))
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode)
    y = oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode)["y"]
    assert np.array_equal(np.load(tmp_path / "y_dp.npy"), y)

    rng = np.random.default_rng(3)
    E, M, K, N = 6, 300, 256, 128
    sizes = np.array([40, 0, 90, 70, 50, 50], np.int32)
    a = (rng.integers(0, 0x7F, (M, K)).astype(np.uint8)) | (rng.integers(0, 2, (M, K)).astype(np.uint8) << 7)
    wts = rng.integers(0, 0x7F, (E, N, K)).astype(np.uint8)
    sa = rng.uniform(0.5, 2, M).astype(np.float32) / 448
    sw = rng.uniform(0.5, 2, (E, N)).astype(np.float32) / 448
    full = oracle.gmm(a, sa, 0, wts, sw, 0, sizes, want="f64")
    assert np.array_equal(np.load(tmp_path / "ep.npy"), full)
    assert float(np.load(tmp_path / "ms.npy")[0]) == 2.0
