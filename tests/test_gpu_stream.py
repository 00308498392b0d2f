"""Streaming memory ingestion: the memory rows of each record arrive in chunks (64 rows,
the chunk of the CoreAI readout, or irregular sizes in any order) and the head finishes
after the last one.  The outputs must equal the one-shot forward's on the same inputs,
bit for bit (every K/V element is the same dot product in the same order), and match
the oracle within the acceptance bar.
"""
import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library

from gpu_support import compare, device_inputs, head_for, run_oracle, schema_of

pytestmark = pytest.mark.gpu

FULL = synth.HeadShape()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()


def _spec():
    return synth.BatchSpec(name="stream", B=3, length_law="uniform", length_range=(700, 2600), questions=(3, 6),
                           options=(2, 7))


def _outputs(out):
    return {k: getattr(out, k).cpu().numpy() for k in ("logits", "probs", "q_value", "q_conf", "q_argmax")}


def _streamed(head, bt, inputs, chunks):
    hidden, ids, lex = inputs
    sch = schema_of(bt)
    head.stream_begin(sch)
    for (b, r0, n) in chunks:
        head.stream_rows(sch, hidden, b, r0, n)
    out = head.stream_finish(sch, hidden, ids, lex)
    torch.cuda.synchronize()
    assert head.device_status() == 0
    return _outputs(out)


def _one_shot(head, bt, inputs):
    hidden, ids, lex = inputs
    out = head.forward(schema_of(bt), hidden, ids, lex)
    torch.cuda.synchronize()
    assert head.device_status() == 0
    return _outputs(out)


def test_stream_64_row_chunks_equals_forward():
    bt = synth.make_batch(_spec(), seed=31)
    head, w = head_for(FULL)
    inputs = device_inputs(bt, FULL.vocab)
    ref = _one_shot(head, bt, inputs)
    # records interleaved round-robin, 64 rows at a time (the last chunk of a record is shorter)
    chunks, pos = [], [0] * bt.B
    while any(pos[b] < bt.lengths[b] for b in range(bt.B)):
        for b in range(bt.B):
            if pos[b] < bt.lengths[b]:
                n = min(64, int(bt.lengths[b]) - pos[b])
                chunks.append((b, pos[b], n))
                pos[b] += n
    got = _streamed(head, bt, inputs, chunks)
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k])
    compare(got, run_oracle(w, FULL, bt), bt)


def test_stream_irregular_chunks_any_order():
    bt = synth.make_batch(_spec(), seed=32)
    head, w = head_for(FULL)
    inputs = device_inputs(bt, FULL.vocab)
    ref = _one_shot(head, bt, inputs)
    rng = np.random.default_rng(5)
    chunks = []
    for b in range(bt.B):
        r = 0
        while r < bt.lengths[b]:
            n = int(min(rng.integers(1, 300), bt.lengths[b] - r))
            chunks.append((b, r, n))
            r += n
    chunks = [chunks[i] for i in rng.permutation(len(chunks))]
    got = _streamed(head, bt, inputs, chunks)
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k])
