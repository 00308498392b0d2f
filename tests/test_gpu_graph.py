"""clef_head_forward captured into a CUDA graph and replayed on new inputs.

After one ordinary call (which sets up the kernels' attributes and caches the plan), a
forward pass without debug outputs can be captured: every step of it is a kernel launch
on the caller's stream.  Each replay uploads the captured plan, clears the status word
and the memory statistics' publication flags, and recomputes everything.  Replaying
after copying a different batch's hidden states into the captured input buffer must
give that batch's outputs bit for bit.  The flags are what would go wrong here: a replay
that found the previous replay's flags still set would fold stale row statistics into
the K/V projection.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library

from gpu_support import device_inputs, head_for, schema_of

pytestmark = pytest.mark.gpu

FULL = synth.HeadShape()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()


def _outputs(out):
    return {k: getattr(out, k).cpu().numpy() for k in ("logits", "probs", "q_value", "q_conf", "q_argmax")}


def test_forward_replays_from_a_cuda_graph_on_new_inputs():
    spec = synth.BatchSpec(name="graph", B=2, lengths=[1500, 2200], questions=(3, 5), options=(2, 6))
    first = synth.make_batch(spec, seed=51)
    # the first batch's schema tables and token ids with another batch's hidden rows
    second = dataclasses.replace(first, hidden=synth.make_batch(spec, seed=52).hidden)
    head, _ = head_for(FULL)
    sch = schema_of(first)
    hidden, ids, lex = device_inputs(first, FULL.vocab)
    hidden_second = device_inputs(second, FULL.vocab)[0]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        out = head.forward(sch, hidden, ids, lex)  # the ordinary first call
        direct_first = _outputs(out)
        direct_second = _outputs(head.forward(sch, hidden_second, ids, lex))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            head.forward(sch, hidden, ids, lex, out=out)
        for src, ref in ((hidden_second, direct_second), (hidden_second, direct_second),
                         (None, direct_first)):
            hidden.copy_(src if src is not None else device_inputs(first, FULL.vocab)[0])
            graph.replay()
            torch.cuda.synchronize()
            assert head.device_status() == 0
            got = _outputs(out)
            for k in ref:
                np.testing.assert_array_equal(got[k], ref[k])
    assert not np.array_equal(direct_first["logits"], direct_second["logits"])
