"""Degenerate and stressed cases of the routing cross-attention ("clef-4bit
JointSchemaHead walkthrough" section 3 step 2), through the whole head on the GPU.

- Zero key projection (weights and bias): every score is equal, so each option's
  attention is the plain mean of V over its record's rows t < L_b. The head then matches
  the oracle, and permuting the memory rows that no span reads (and that are not the
  global last row) changes nothing beyond fp32 summation order.
- Key projection scaled by 8: scores spread over tens of units in the exp2 domain, so
  most probabilities underflow and the running maximum moves across tiles and chunks.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library
from structured_decision_model_gb300.head import ClefHead
from synth.bf16 import bf16_to_f32, f32_to_bf16

from gpu_support import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FULL = synth.HeadShape()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()
    torch.cuda.init()


def _head(w):
    s = FULL
    return ClefHead(w, s.H, s.D, s.heads, s.F, s.n_route, s.n_joint, s.vocab)


def _with_keys(scale):
    """Base weights with every routing layer's key projection (weight and bias) times `scale`."""
    w = dict(synth.make_weights(FULL, 0))
    for l in range(FULL.n_route):
        for name in (f"route.{l}.k.weight", f"route.{l}.k.bias"):
            w[name] = f32_to_bf16(bf16_to_f32(w[name]) * np.float32(scale))  # exact: power of two or zero
    return w


def _batch(seed):
    spec = synth.BatchSpec(name="attn", B=2, length_law="uniform", length_range=(1100, 2300), questions=(2, 4),
                           options=(2, 6))
    bt = synth.make_batch(spec, seed=seed)
    assert (bt.lengths % 64 != 0).all() and bt.lengths.max() > 1024  # ragged last tile, several chunks
    return bt


def test_zero_keys_give_uniform_attention():
    w = _with_keys(0.0)
    head = _head(w)
    bt = _batch(31)
    gpu = run_gpu(head, bt)
    compare(gpu, run_oracle(w, FULL, bt), bt)

    # rows no span reads and that are not the last row only enter through the uniform mean
    used = np.zeros((bt.B, bt.Lpad), bool)
    for q in range(bt.Q):
        b = bt.q_rec[q]
        used[b, bt.q_span[q, 0]:bt.q_span[q, 1]] = True
        for j in range(bt.q_opt_off[q], bt.q_opt_off[q + 1]):
            used[b, bt.o_span[j, 0]:bt.o_span[j, 1]] = True
    hidden = bt.hidden.copy()
    ids = bt.token_ids.copy()
    rng = np.random.default_rng(32)
    for b in range(bt.B):
        used[b, bt.lengths[b] - 1] = True
        free = np.nonzero(~used[b, :bt.lengths[b]])[0]
        perm = rng.permutation(free)
        hidden[b, free] = bt.hidden[b, perm]
        ids[b, free] = bt.token_ids[b, perm]
    moved = run_gpu(head, dataclasses.replace(bt, hidden=hidden, token_ids=ids))
    np.testing.assert_allclose(moved["logits"], gpu["logits"], atol=1e-3)
    np.testing.assert_allclose(moved["probs"], gpu["probs"], atol=1e-4)


def test_sharp_scores_match_oracle():
    w = _with_keys(8.0)
    head = _head(w)
    bt = _batch(33)
    compare(run_gpu(head, bt), run_oracle(w, FULL, bt), bt)
