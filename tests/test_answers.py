"""The answer layer on CPU: response shape, option order, rounding, usage.

The numbers come from the oracle here (the layer only names, orders and rounds the
head's outputs); the GPU side is covered by test_gpu_answers in the GPU suite.
"""
import numpy as np

import oracle
import synth
from structured_decision_model_gb300.answers import batch_responses, option_order

SHAPE = synth.HeadShape(H=64, D=32, heads=2, F=64, vocab=300)


def test_option_order_rules():
    assert option_order("noul") == ["true", "false"]
    assert option_order("choice", {"paid": "x", "overdue": "y", "draft": "z"}) == ["draft", "overdue", "paid"]
    assert option_order("choice", {"10": "a", "2": "b", "1": "c"}) == ["1", "10", "2"]  # sorted as strings
    assert option_order("score", {"0": "low", "1": "mid", "2": "high"}) == ["0", "1", "2"]


def _batch():
    spec = synth.BatchSpec(name="ans", B=2, H=64, vocab=300, length_law="uniform", length_range=(250, 400),
                           questions=(3, 4), options=(2, 5), instr_len=(3, 8), option_len=(2, 5))
    bt = synth.make_batch(spec, seed=9)
    w = synth.make_weights(SHAPE, seed=2)
    res = oracle.head_forward(w, SHAPE.heads, SHAPE.n_route, SHAPE.n_joint, bt.hidden, bt.lengths, bt.q_rec,
                              bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical)
    qids, types, options, legends = [], [], [], []
    for q in range(bt.Q):
        n = int(bt.q_opt_off[q + 1] - bt.q_opt_off[q])
        t = int(bt.q_type[q])
        qids.append(f"q{q}")
        types.append(t)
        if t == 0:
            options.append(option_order("noul"))
            legends.append(None)
        elif t == 1:
            options.append(option_order("choice", {f"opt{k}": "" for k in range(n)}))
            legends.append(None)
        else:
            lg = {str(k): f"level {k}" for k in range(n)}
            options.append(option_order("score", lg))
            legends.append(lg)
    return bt, res, qids, types, options, legends


def test_responses_shape_and_values():
    bt, res, qids, types, options, legends = _batch()
    resp = batch_responses("clef", bt.q_rec, bt.q_opt_off, qids, types, options, legends, bt.lengths,
                           res["probs"], res["value"], res["conf"], res["argmax"])
    assert len(resp) == bt.B
    for b, r in enumerate(resp):
        assert r["model"] == "clef"
        assert r["usage"] == {"input_tokens": int(bt.lengths[b]), "output_tokens": 0}
        for q in np.nonzero(bt.q_rec == b)[0]:
            a = r["answers"][f"q{q}"]
            p = res["probs"][bt.q_opt_off[q]:bt.q_opt_off[q + 1]]
            if types[q] == 0:
                assert a == {"type": "noul", "noul": round(float(p[0]), 4)}
            elif types[q] == 1:
                assert a["choice"] == options[q][int(np.argmax(p))]
                assert a["confidence"] == round(float(p.max()), 4)
                assert list(a["probabilities"]) == options[q]
                assert abs(sum(a["probabilities"].values()) - 1.0) <= 5e-5 * len(p)
            else:
                ev = float(np.dot(np.arange(len(p)), p))
                assert a["score"] == round(ev, 4) and 0 <= a["score"] <= len(p) - 1
                assert a["confidence"] == round(float(p.max()), 4)
                assert list(a["legend"]) == [str(k) for k in range(len(p))]
                assert a["legend"]["0"] == "level 0"
            for v in (a.get("probabilities") or {}).values():
                assert v == round(v, 4)
