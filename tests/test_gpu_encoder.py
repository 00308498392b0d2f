"""Record -> encode -> collate -> head on the GPU -> answers, against the oracle.

The backbone is out of scope, so the hidden states of the encoded rows are seeded
random rows; everything the encoder produces (ids, lengths, span tables, option order)
drives the head and the answer layer as it would after a real backbone.
"""
import numpy as np
import pytest
import torch

import synth
from synth.records import draw_hidden_record
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.answers import batch_responses
from structured_decision_model_gb300.build import build_library
from structured_decision_model_gb300.encoder import ByteTokenizer, collate_records, encode_record

from gpu_support import compare, head_for, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

RECORDS = [
    {"state": {"invoice": {"vendor": "Acme", "total": 1250.0, "currency": "USD", "status": "overdue"}},
     "questions": {
         "status": {"type": "choice", "instructions": "What is the invoice status?",
                    "criteria": {"paid": "Invoice is paid.", "overdue": "Invoice is past due.", "draft": "Not sent."}},
         "large": {"type": "noul", "instructions": "Is the total above 1000 USD?"},
         "risk": {"type": "score", "instructions": "How risky is this account?",
                  "criteria": {"0": "low", "1": "medium", "2": "high", "3": "critical"}}}},
    {"state": "Our checkout started returning errors and orders are blocked. " * 20,
     "questions": {"outage": {"type": "noul", "instructions": "Is a service down?"},
                   "team": {"type": "choice", "instructions": "Which team owns it?",
                            "criteria": {"payments": "Payments", "web": "Web front end", "infra": "Infrastructure"}}}},
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()
    torch.cuda.init()


def test_encoded_records_through_the_head_and_answers():
    tok = ByteTokenizer()
    shape = synth.HeadShape(H=256, vocab=512)
    enc = [encode_record(tok, r, max_length=1024) for r in RECORDS]
    cb = collate_records(enc, tok.pad_token_id)
    spec = synth.BatchSpec(name="encoded", B=cb.B, H=shape.H, vocab=shape.vocab, lengths=list(cb.lengths))
    hidden = np.stack([draw_hidden_record(31, b, cb.Lpad, shape.H) for b in range(cb.B)])
    bt = synth.Batch(spec=spec, seed=31, H=shape.H, B=cb.B, Lpad=cb.Lpad, lengths=cb.lengths, q_rec=cb.q_rec,
                     q_type=cb.q_type, q_span=cb.q_span, q_opt_off=cb.q_opt_off, o_span=cb.o_span,
                     token_ids=cb.token_ids, lexical=synth.SparseLexical(31, shape.vocab, shape.H), hidden=hidden)
    head, w = head_for(shape)
    got = run_gpu(head, bt)
    ref = run_oracle(w, shape, bt)
    compare(got, ref, bt)
    resp = batch_responses("clef", cb.q_rec, cb.q_opt_off, cb.question_ids, cb.question_types, cb.options,
                           cb.legends, cb.lengths, got["probs"], got["q_value"], got["q_conf"], got["q_argmax"])
    assert [sorted(r["answers"]) for r in resp] == [["large", "risk", "status"], ["outage", "team"]]
    assert resp[0]["answers"]["status"]["choice"] in ("draft", "overdue", "paid")
    assert set(resp[0]["answers"]["risk"]["legend"]) == {"0", "1", "2", "3"}
    assert resp[1]["usage"] == {"input_tokens": int(cb.lengths[1]), "output_tokens": 0}
