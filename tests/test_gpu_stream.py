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


def test_stream_fp16_rows_equal_rounded_bf16_and_match_oracle():
    """fp16 hidden rows (the dtype of the CoreAI chunked readout).  The head rounds each
    fp16 value to bf16 where it reads it, so streaming the fp16 rows must give exactly the
    outputs of streaming the host-rounded bf16 rows; and the oracle, fed the fp16 values
    widened exactly, must agree within the acceptance bar.  Record 0 arrives as one chunk
    longer than the 1024-row staging pass; the others in 64-row chunks."""
    import dataclasses

    import oracle

    bt = synth.make_batch(_spec(), seed=33, with_hidden=False)
    rng = np.random.default_rng(33)
    h16 = (rng.standard_normal((bt.B, bt.Lpad, bt.H), dtype=np.float32) * 1.5).astype(np.float16)
    bt = dataclasses.replace(bt, hidden=synth.f32_to_bf16(h16.astype(np.float32)))
    assert bt.lengths[0] > 1024
    head, w = head_for(FULL)
    hidden_b, ids, lex = device_inputs(bt, FULL.vocab)
    hidden16 = torch.from_numpy(h16).cuda()
    chunks = [(0, 0, int(bt.lengths[0]))]
    chunks += [(b, r0, min(64, int(bt.lengths[b]) - r0)) for r0 in range(0, int(bt.lengths.max()), 64)
               for b in range(1, bt.B) if r0 < bt.lengths[b]]
    got = _streamed(head, bt, (hidden16, ids, lex), chunks)
    ref_b = _streamed(head, bt, (hidden_b, ids, lex), chunks)
    for k in got:
        np.testing.assert_array_equal(got[k], ref_b[k])
    ref = oracle.head_forward(w, FULL.heads, FULL.n_route, FULL.n_joint, lambda b: h16[b].astype(np.float64),
                              bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids,
                              bt.lexical)
    print("fp16 stream", compare(got, ref, bt))
