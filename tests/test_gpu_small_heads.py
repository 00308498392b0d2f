"""Parity of small head shapes against the oracle, one-shot and streamed.

The shapes have narrow widths, one or two attention heads, few layers, and hidden sizes
whose K range is an odd number of 64-wide slices.  With the pages' width (D = 1024) the
memory K/V projection always runs as CTA pairs or on 64-wide tiles with at least 16
output-column tiles.  These shapes run it on the single-CTA kernels with two to eight
column tiles and a part-filled last K stage.  That exercises the in-kernel memory
LayerNorm statistics in other launch geometries: jobs of 16 rows dealt over every CTA of
the launch, paced by each CTA's producer, published through per-row flags.  The rows
carry per-row offsets far from zero mean and a few outlier channels, as final-norm
hidden states do ("clef-flash-CoreAI metadata.json" decision.head.reads: the head reads
the backbone's final-norm states).  Records of 127, 129 and 130 rows put real and
padding rows in one 128-row tile.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library

from gpu_support import compare, device_inputs, head_for, run_gpu, run_oracle, schema_of

pytestmark = pytest.mark.gpu

SHAPES = [
    synth.HeadShape(H=192, D=64, heads=1, F=128, n_route=1, n_joint=1, vocab=3000),
    synth.HeadShape(H=320, D=128, heads=2, F=192, n_route=2, n_joint=2, vocab=3000),
]
# one 128-wide column tile per row tile and more row tiles (157) than CTAs: each CTA
# walks two tiles and the statistics jobs of a tile belong to other CTAs
NARROW = synth.HeadShape(H=64, D=64, heads=1, F=64, n_route=1, n_joint=1, vocab=3000)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()


def _batch(shape, seed, lengths=(130, 127, 129, 300)):
    spec = synth.BatchSpec(name="small", B=len(lengths), H=shape.H, vocab=shape.vocab, lengths=list(lengths),
                           questions=(2, 3), options=(2, 4), instr_len=(4, 12), option_len=(2, 8))
    bt = synth.make_batch(spec, seed=seed)
    rng = np.random.default_rng(seed)
    h = synth.bf16_to_f32(bt.hidden)
    h += rng.uniform(-20, 20, size=(bt.B, bt.Lpad, 1)).astype(np.float32)
    ch = rng.choice(bt.H, size=2, replace=False)
    h[:, :, ch] *= 20.0
    return dataclasses.replace(bt, hidden=synth.f32_to_bf16(h))


def _stream(head, bt, inputs):
    hidden, ids, lex = inputs
    sch = schema_of(bt)
    head.stream_begin(sch)
    pos = [0] * bt.B
    while any(pos[b] < bt.lengths[b] for b in range(bt.B)):  # 64-row chunks, records interleaved
        for b in range(bt.B):
            if pos[b] < bt.lengths[b]:
                n = min(64, int(bt.lengths[b]) - pos[b])
                head.stream_rows(sch, hidden, b, pos[b], n)
                pos[b] += n
    out = head.stream_finish(sch, hidden, ids, lex)
    torch.cuda.synchronize()
    assert head.device_status() == 0
    return {k: getattr(out, k).cpu().numpy() for k in ("logits", "probs", "q_value", "q_conf", "q_argmax")}


@pytest.mark.parametrize("shape", SHAPES, ids=["h192_d64", "h320_d128"])
def test_small_head_forward_and_stream(shape):
    bt = _batch(shape, seed=41 + shape.H)
    head, w = head_for(shape)
    inputs = device_inputs(bt, shape.vocab)
    gpu = run_gpu(head, bt, inputs=inputs)
    compare(gpu, run_oracle(w, shape, bt), bt)
    streamed = _stream(head, bt, inputs)
    for k in gpu:
        np.testing.assert_array_equal(streamed[k], gpu[k])


def test_narrow_head_long_records_one_column_tile():
    bt = _batch(NARROW, seed=47, lengths=(9000, 11000))
    head, w = head_for(NARROW)
    inputs = device_inputs(bt, NARROW.vocab)
    gpu = run_gpu(head, bt, inputs=inputs)
    compare(gpu, run_oracle(w, NARROW, bt), bt)
    streamed = _stream(head, bt, inputs)
    for k in gpu:
        np.testing.assert_array_equal(streamed[k], gpu[k])
