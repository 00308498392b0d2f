"""Answers built from the GPU head's outputs against answers built from the oracle's."""
import numpy as np
import pytest

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.answers import batch_responses, option_order
from structured_decision_model_gb300.build import build_library

from gpu_support import head_for, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_answers_from_gpu_match_oracle():
    build_library()
    B.load()
    shape = synth.HeadShape()
    spec = synth.BatchSpec(name="ans", B=3, length_law="uniform", length_range=(600, 1500), questions=(3, 6),
                           options=(2, 6))
    bt = synth.make_batch(spec, seed=41)
    head, w = head_for(shape)
    gpu = run_gpu(head, bt)
    ref = run_oracle(w, shape, bt)
    qids, types, options, legends = [], [], [], []
    for q in range(bt.Q):
        n = int(bt.q_opt_off[q + 1] - bt.q_opt_off[q])
        t = int(bt.q_type[q])
        qids.append(f"q{q}")
        types.append(t)
        crit = {f"o{k}": "" for k in range(n)} if t == 1 else {str(k): f"l{k}" for k in range(n)}
        options.append(option_order(["noul", "choice", "score"][t], crit))
        legends.append(crit if t == 2 else None)
    args = (bt.q_rec, bt.q_opt_off, qids, types, options, legends, bt.lengths)
    rg = batch_responses("clef", *args, gpu["probs"], gpu["q_value"], gpu["q_conf"], gpu["q_argmax"])
    ro = batch_responses("clef", *args, ref["probs"], ref["value"], ref["conf"], ref["argmax"])
    for b in range(bt.B):
        for q in np.nonzero(bt.q_rec == b)[0]:
            a, e = rg[b]["answers"][f"q{q}"], ro[b]["answers"][f"q{q}"]
            assert a["type"] == e["type"]
            p = np.sort(ref["probs"][bt.q_opt_off[q]:bt.q_opt_off[q + 1]])[::-1]
            if a["type"] == "choice" and p[0] - p[1] >= 0.05:
                assert a["choice"] == e["choice"]
            for key in ("noul", "score", "confidence"):
                if key in e:
                    assert abs(a[key] - e[key]) <= 5e-2 if key == "score" else abs(a[key] - e[key]) <= 1e-2
            for o in e.get("probabilities", {}):
                assert abs(a["probabilities"][o] - e["probabilities"][o]) <= 1e-2
