"""Record sharding across ranks (world size 2, gloo, CPU only).

Each rank runs the head (the CPU oracle stands in for the GPU path here) on its
own contiguous, row-balanced record range; the ranks gather their outputs and
rank 0 reassembles them in batch order.  Because records are independent, the
reassembled outputs must equal the single-process batch outputs exactly.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from structured_decision_model_gb300.sharding import assemble, shard_records, sub_batch

SHAPE = synth.HeadShape(H=64, D=32, heads=2, F=64, vocab=300)
SPEC = synth.BatchSpec(name="shard", B=5, H=64, vocab=300, length_law="uniform", length_range=(150, 420),
                       questions=(1, 4), options=(2, 5), instr_len=(3, 8), option_len=(2, 5))


def _run_shard(bt, w, sb):
    return oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden[sb.records], sb.lengths,
                               sb.q_rec, sb.q_type, sb.q_span, sb.q_opt_off, sb.o_span, bt.token_ids[sb.records],
                               bt.lexical)


def _worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bt = synth.make_batch(SPEC, seed=3)
    w = synth.make_weights(SHAPE, seed=1)
    shards = shard_records(bt.lengths, world)
    sb = sub_batch(shards[rank], bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    res = _run_shard(bt, w, sb)
    gathered = [None] * world
    dist.all_gather_object(gathered, (rank, res))
    if rank == 0:
        parts = []
        for r, res_r in sorted(gathered, key=lambda x: x[0]):
            sbr = sub_batch(shards[r], bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
            parts.append((sbr, res_r))
        full = assemble(parts, bt.Q, bt.O)
        np.savez(result_path, **full)
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shards_cover_records_and_balance_rows():
    lengths = np.array([16384, 100, 200, 16000, 300, 500, 7000, 9000])
    for world in (1, 2, 3, 4, 8, 10):
        sh = shard_records(lengths, world)
        assert len(sh) == world
        assert np.array_equal(np.concatenate(sh), np.arange(len(lengths)))
        if world <= len(lengths):
            assert all(len(s) > 0 for s in sh)
    sh = shard_records(np.full(8, 16384), 4)
    assert [len(s) for s in sh] == [2, 2, 2, 2]


def test_two_rank_gloo_sharding_matches_single_process(tmp_path):
    result = str(tmp_path / "sharded.npz")
    mp.start_processes(_worker, args=(2, _free_port(), result), nprocs=2, join=True, start_method="spawn")
    got = np.load(result)
    bt = synth.make_batch(SPEC, seed=3)
    w = synth.make_weights(SHAPE, seed=1)
    ref = oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden, bt.lengths, bt.q_rec,
                              bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical)
    for k in ("logits", "probs", "value", "conf", "argmax"):
        np.testing.assert_array_equal(got[k], ref[k])
