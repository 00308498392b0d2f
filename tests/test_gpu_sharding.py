"""The per-GPU compute of the record-sharded runner, on one GPU.

``ClefHead.shard_fn`` is what each rank of a multi-GPU job runs on its own records.
Here the shards of a 2- and a 3-way split run one after the other on one GPU (no
rank waits on another) and are reassembled; since no reduction crosses records, the
result must equal one whole-batch forward bit for bit, and the oracle within the
parity bar.
"""
import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library
from structured_decision_model_gb300.sharding import ShardedRunner, assemble, shard_records, sub_batch

from gpu_support import compare, device_inputs, head_for, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FULL = synth.HeadShape()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()


@pytest.mark.parametrize("world", [2, 3])
def test_shards_reassemble_to_the_whole_batch_bitwise(world):
    spec = synth.BatchSpec(name="shard", B=5, length_law="uniform", length_range=(400, 2200), questions=(2, 5),
                           options=(2, 6))
    bt = synth.make_batch(spec, seed=31)
    head, w = head_for(FULL)
    hidden, ids, lex = device_inputs(bt, FULL.vocab)
    whole = run_gpu(head, bt, inputs=(hidden, ids, lex))
    tables = (bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    run = head.shard_fn(bt.hidden, bt.token_ids, lex)  # host arrays: each shard copies its own records
    parts = []
    for recs in shard_records(bt.lengths, world):
        sb = sub_batch(recs, *tables)
        parts.append((sb, run(sb)))
    got = assemble(parts, bt.Q, bt.O)
    np.testing.assert_array_equal(got["logits"], whole["logits"])
    np.testing.assert_array_equal(got["probs"], whole["probs"])
    np.testing.assert_array_equal(got["argmax"], whole["q_argmax"])
    gpu = {"logits": got["logits"], "probs": got["probs"], "q_value": got["value"], "q_conf": got["conf"],
           "q_argmax": got["argmax"]}
    compare(gpu, run_oracle(w, FULL, bt), bt)


def test_single_rank_runner_with_device_tensors():
    spec = synth.BatchSpec(name="shard1", B=2, length_law="uniform", length_range=(300, 900), questions=(1, 3),
                           options=(2, 4))
    bt = synth.make_batch(spec, seed=32)
    head, _ = head_for(FULL)
    hidden, ids, lex = device_inputs(bt, FULL.vocab)
    runner = ShardedRunner(head.shard_fn(hidden, ids, lex))
    got = runner.forward(bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    whole = run_gpu(head, bt, inputs=(hidden, ids, lex))
    np.testing.assert_array_equal(got["logits"], whole["logits"])
    torch.cuda.synchronize()
