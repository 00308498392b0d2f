"""Shared pieces of the GPU parity tests: device inputs from a synthetic batch,
oracle runs on chosen records, and the acceptance checks.

Acceptance (the head's parity bar): logits within 3e-2 max-abs, probabilities
within 1e-2 max-abs, and the same argmax on every question whose top-two
probability margin in the oracle is at least 0.05.
"""
import numpy as np
import torch

import oracle
import synth
from structured_decision_model_gb300 import binding
from structured_decision_model_gb300.head import ClefHead, to_device_bf16

LOGIT_TOL = 3e-2
PROB_TOL = 1e-2
ARGMAX_MARGIN = 0.05

_HEADS = {}


def head_for(shape: synth.HeadShape, seed=0):
    key = (shape, seed)
    if key not in _HEADS:
        w = synth.make_weights(shape, seed)
        _HEADS[key] = (ClefHead(w, shape.H, shape.D, shape.heads, shape.F, shape.n_route, shape.n_joint,
                                shape.vocab), w)
    return _HEADS[key]


def schema_of(bt, row_stride=None):
    return binding.Schema(bt.B, bt.Lpad, row_stride or bt.H, bt.lengths, bt.q_rec, bt.q_type, bt.q_span,
                          bt.q_opt_off, bt.o_span)


def device_lexical(bt, vocab, fill_seed=0):
    """Full [vocab, H] table on the device: rows the batch reads come from the seeded
    generator; the others are filled on the device (they are never read)."""
    g = torch.Generator(device="cuda").manual_seed(fill_seed)
    lex = torch.empty((vocab, bt.H), dtype=torch.bfloat16, device="cuda")
    lex.normal_(0.0, 0.02, generator=g)
    used = bt.lexical_ids()
    used = used[(used >= 0) & (used < vocab)]
    if len(used):
        lex[torch.from_numpy(used.astype(np.int64)).cuda()] = to_device_bf16(bt.lexical[used])
    return lex


def device_inputs(bt, vocab, row_stride=None):
    if row_stride is None or row_stride == bt.H:
        hidden = to_device_bf16(bt.hidden)
    else:
        hidden = torch.zeros((bt.B, bt.Lpad, row_stride), dtype=torch.bfloat16, device="cuda")
        hidden[:, :, :bt.H] = to_device_bf16(bt.hidden)
    ids = torch.from_numpy(bt.token_ids).cuda()
    return hidden, ids, device_lexical(bt, vocab)


def run_gpu(head, bt, debug=None, row_stride=None, inputs=None):
    hidden, ids, lex = inputs if inputs is not None else device_inputs(bt, head.vocab, row_stride)
    out = head.forward(schema_of(bt, row_stride), hidden, ids, lex, debug=debug)
    torch.cuda.synchronize()
    st = head.device_status()
    assert st == 0, binding.STATUS.get(st, st)
    return {k: getattr(out, k).cpu().numpy() for k in ("logits", "probs", "q_value", "q_conf", "q_argmax")}


def run_oracle(w, shape, bt, records=None, keep=False):
    return oracle.head_forward(w, shape.heads, shape.n_route, shape.n_joint,
                               bt.hidden if bt.hidden is not None else bt.record_hidden, bt.lengths, bt.q_rec,
                               bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical,
                               records=records, keep=keep)


def rel_rms(got, ref):
    """Root-mean-square error relative to the reference's RMS: a systematic slip in a
    stage (a wrong bias, a skipped norm, a shifted row) moves it by O(1), where
    per-element rounding of bf16 activations stays near 1e-3."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.sqrt(((got - ref) ** 2).mean() / max((ref ** 2).mean(), 1e-30)))


def compare(gpu, ref, bt, records=None):
    """Acceptance check on the options / questions of ``records`` (all by default)."""
    if records is None:
        qsel = np.arange(bt.Q)
    else:
        qsel = np.nonzero(np.isin(bt.q_rec, records))[0]
    osel = np.concatenate([np.arange(bt.q_opt_off[q], bt.q_opt_off[q + 1]) for q in qsel])
    dl = np.abs(gpu["logits"][osel] - ref["logits"][osel]).max()
    dp = np.abs(gpu["probs"][osel] - ref["probs"][osel]).max()
    dv = np.abs(gpu["q_value"][qsel] - ref["value"][qsel]).max()
    assert np.isfinite(gpu["logits"][osel]).all()
    bad = []
    for q in qsel:
        p = np.sort(ref["probs"][bt.q_opt_off[q]:bt.q_opt_off[q + 1]])[::-1]
        margin = p[0] - (p[1] if len(p) > 1 else 0.0)
        if margin >= ARGMAX_MARGIN and gpu["q_argmax"][q] != ref["argmax"][q]:
            bad.append(int(q))
    assert dl <= LOGIT_TOL, f"max |dlogit| {dl:.3e}"
    assert dp <= PROB_TOL, f"max |dprob| {dp:.3e}"
    assert dv <= 5 * PROB_TOL, f"max |dvalue| {dv:.3e}"  # score values scale by up to the level count
    assert not bad, f"argmax disagrees on questions {bad}"
    return dict(max_dlogit=float(dl), max_dprob=float(dp), n_opts=int(len(osel)))
