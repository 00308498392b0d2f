"""Record sharding across ranks (gloo, CPU only).

The ranks run ``ShardedRunner`` -- the code a multi-GPU job runs -- with the CPU
oracle standing in for the per-rank CUDA head: each rank computes its own
contiguous, row-balanced record range, the outputs are gathered once and every rank
reassembles them in batch order.  Because records are independent, the reassembled
outputs must equal the single-process batch outputs exactly.
"""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from structured_decision_model_gb300.sharding import ShardedRunner, shard_records

SHAPE = synth.HeadShape(H=64, D=32, heads=2, F=64, vocab=300)
SPEC = synth.BatchSpec(name="shard", B=5, H=64, vocab=300, length_law="uniform", length_range=(150, 420),
                       questions=(1, 4), options=(2, 5), instr_len=(3, 8), option_len=(2, 5))


def _oracle_shard_fn(bt, w):
    """Per-rank compute stand-in: the oracle on the shard's records."""
    def run(sb):
        r = oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden[sb.records], sb.lengths,
                                sb.q_rec, sb.q_type, sb.q_span, sb.q_opt_off, sb.o_span, bt.token_ids[sb.records],
                                bt.lexical)
        return {k: r[k] for k in ("logits", "probs", "value", "conf", "argmax")}
    return run


def _worker(rank, world, port, result_path, n_records):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bt = synth.make_batch(dataclasses.replace(SPEC, B=n_records), seed=3)
    w = synth.make_weights(SHAPE, seed=1)
    runner = ShardedRunner(_oracle_shard_fn(bt, w))
    assert runner.world_rank() == (world, rank)
    mine = runner.local(bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    assert np.array_equal(mine.records, shard_records(bt.lengths, world)[rank])
    full = runner.forward(bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    np.savez(f"{result_path}.{rank}.npz", **full)
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


@pytest.mark.parametrize("world,n_records", [(2, 5), (3, 2)])
def test_gloo_sharded_runner_matches_single_process(tmp_path, world, n_records):
    """world 3 over 2 records leaves one rank without a record."""
    result = str(tmp_path / "sharded")
    mp.start_processes(_worker, args=(world, _free_port(), result, n_records), nprocs=world, join=True,
                       start_method="spawn")
    bt = synth.make_batch(dataclasses.replace(SPEC, B=n_records), seed=3)
    w = synth.make_weights(SHAPE, seed=1)
    ref = oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden, bt.lengths, bt.q_rec,
                              bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical)
    for r in range(world):  # every rank returns the whole batch
        got = np.load(f"{result}.{r}.npz")
        for k in ("logits", "probs", "value", "conf", "argmax"):
            np.testing.assert_array_equal(got[k], ref[k])


def test_single_process_runner_is_one_rank():
    bt = synth.make_batch(dataclasses.replace(SPEC, B=3), seed=4)
    w = synth.make_weights(SHAPE, seed=1)
    runner = ShardedRunner(_oracle_shard_fn(bt, w))
    assert runner.world_rank() == (1, 0)
    got = runner.forward(bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    ref = oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden, bt.lengths, bt.q_rec,
                              bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical)
    np.testing.assert_array_equal(got["logits"], ref["logits"])
