"""The answer layer: per-question answers in the SystemOne-compatible response shape.

Host code around the head's outputs, following "clef-flash-CoreAI metadata.json"
decision.option_order, decision.question_types and decision.response:
  - option order: noul [true, false]; choice: option ids sorted as strings; score:
    levels 0..n-1 (``option_order``, used when the schema's option spans are laid out);
  - noul: {type, noul: p(true)}; choice: {type, choice: argmax id, confidence, probabilities};
    score: {type, score: sum(level * p), confidence: max p, legend, probabilities};
  - probabilities and values rounded to 4 decimals;
  - usage: {input_tokens: prompt tokens of the record, output_tokens: 0} (no decoding).
The numbers come from the head (``q_value``, ``q_conf``, ``q_argmax``, ``probs``); this
module only orders, names and rounds them.
"""
from typing import Dict, List, Sequence

import numpy as np

TYPE_IDS = {"noul": 0, "choice": 1, "score": 2}
TYPE_NAMES = {v: k for k, v in TYPE_IDS.items()}
NOUL_OPTIONS = ["true", "false"]


def option_order(qtype: str, criteria=None) -> List[str]:
    """Option ids of a question in the order the head scores them."""
    if qtype == "noul":
        return list(NOUL_OPTIONS)
    if qtype == "choice":
        return sorted(str(k) for k in (criteria or {}))
    if qtype == "score":
        n = len(criteria) if criteria else 0
        return [str(i) for i in range(n)]
    raise ValueError(f"unknown question type {qtype!r}")


def _r4(x) -> float:
    return round(float(x), 4)


def record_answers(question_ids: Sequence[str], question_types: Sequence[int], options: Sequence[List[str]],
                   legends: Sequence[dict], probs: Sequence[np.ndarray], q_value, q_conf, q_argmax) -> Dict[str, dict]:
    """Answers of one record, keyed by question id.

    ``options[k]`` are question k's option ids in head order, ``probs[k]`` its option
    probabilities, ``legends[k]`` the score legend (level -> criterion) or None.
    """
    out = {}
    for k, qid in enumerate(question_ids):
        t = int(question_types[k])
        p = np.asarray(probs[k], np.float64)
        if len(p) != len(options[k]):
            raise ValueError(f"question {qid!r}: {len(p)} probabilities for {len(options[k])} options")
        if t == 0:
            out[qid] = {"type": "noul", "noul": _r4(q_value[k])}
        elif t == 1:
            out[qid] = {"type": "choice", "choice": options[k][int(q_argmax[k])], "confidence": _r4(q_conf[k]),
                        "probabilities": {o: _r4(x) for o, x in zip(options[k], p)}}
        elif t == 2:
            legend = legends[k] or {}
            out[qid] = {"type": "score", "score": _r4(q_value[k]), "confidence": _r4(q_conf[k]),
                        "legend": {str(lv): legend.get(str(lv), legend.get(lv)) for lv in range(len(p))},
                        "probabilities": {str(i): _r4(x) for i, x in enumerate(p)}}
        else:
            raise ValueError(f"question {qid!r}: unknown type id {t}")
    return out


def batch_responses(model: str, q_rec, q_opt_off, question_ids, question_types, options, legends, input_tokens,
                    probs, q_value, q_conf, q_argmax) -> List[dict]:
    """One response per record: {model, answers, usage}.

    ``question_ids`` / ``question_types`` / ``options`` / ``legends`` are per question of
    the batch (in the schema's order), ``input_tokens`` per record, and the numeric
    arrays are the head's outputs for the batch.
    """
    q_rec = np.asarray(q_rec)
    q_opt_off = np.asarray(q_opt_off)
    probs = np.asarray(probs)
    responses = []
    for b in range(len(input_tokens)):
        qs = np.nonzero(q_rec == b)[0]
        ans = record_answers([question_ids[q] for q in qs], [question_types[q] for q in qs],
                             [options[q] for q in qs], [legends[q] for q in qs],
                             [probs[q_opt_off[q]:q_opt_off[q + 1]] for q in qs],
                             np.asarray(q_value)[qs], np.asarray(q_conf)[qs], np.asarray(q_argmax)[qs])
        responses.append({"model": model, "answers": ans,
                          "usage": {"input_tokens": int(input_tokens[b]), "output_tokens": 0}})
    return responses
