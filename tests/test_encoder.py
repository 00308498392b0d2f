"""Host record encoding and batching (prompt layout, spans, truncation) with the stand-in tokenizer."""
import numpy as np
import pytest

from structured_decision_model_gb300.encoder import (PREFIX, SUFFIX, ByteTokenizer, collate_records, encode_record,
                                                      render)

TOK = ByteTokenizer()

INVOICE = {
    "state": {"invoice": {"vendor": "Acme", "total": 1250.0, "currency": "USD", "status": "overdue"}},
    "questions": {
        "status": {"type": "choice", "instructions": "What is the invoice status?",
                   "criteria": {"paid": "Invoice is paid.", "overdue": "Invoice is past due.", "draft": "Not sent."}},
        "large": {"type": "noul", "instructions": "Is the total above 1000 USD?"},
        "risk": {"type": "score", "instructions": "How risky is this account?",
                 "criteria": {"0": "low", "1": "medium", "2": "high"}},
    },
}


def test_render_rules():
    assert render("as is") == "as is"
    assert render({"b": 1, "a": "é"}) == '{"a":"é","b":1}'  # sorted keys, compact, non-ASCII kept


def test_layout_and_spans_decode_to_their_texts():
    e = encode_record(TOK, INVOICE)
    text = TOK.decode(e.ids)
    assert text.startswith(PREFIX + render(INVOICE["state"]))
    assert text.endswith(SUFFIX) and TOK.decode(e.ids[-1:]) == ":"
    assert e.question_ids == ["status", "large", "risk"] and e.question_types == [1, 0, 2]
    assert e.options[0] == ["draft", "overdue", "paid"]      # choice: option ids sorted as strings
    assert e.options[1] == ["true", "false"]                 # noul order
    assert e.options[2] == ["0", "1", "2"]                   # score levels
    for k, (qid, q) in enumerate(INVOICE["questions"].items()):
        s, t = e.q_span[k]
        assert TOK.decode(e.ids[s:t]) == q["instructions"]
        crit = q.get("criteria") or {"true": "The proposition is true or the answer is yes.",
                                     "false": "The proposition is false or the answer is no."}
        for j, oid in enumerate(e.options[k]):
            s, t = e.o_span[k][j]
            assert TOK.decode(e.ids[s:t]) == render({oid: crit[oid]})
            assert TOK.decode(e.ids[s - len("OPTION 1: "):s]) == f"OPTION {j + 1}: "
    assert e.legends[2] == {"0": "low", "1": "medium", "2": "high"} and e.legends[0] is None
    # spans are disjoint and increasing
    flat = [sp for k in range(3) for sp in [e.q_span[k]] + e.o_span[k]]
    assert all(a[1] <= b[0] for a, b in zip(flat, flat[1:]))


def test_instruction_defaults_to_the_id():
    e = encode_record(TOK, {"state": "x", "questions": {"outage": {"type": "noul"}}})
    s, t = e.q_span[0]
    assert TOK.decode(e.ids[s:t]) == "outage"


def test_truncation_keeps_the_schema_and_cuts_the_state():
    full = encode_record(TOK, INVOICE)
    fixed = len(full.ids) - full.state_tokens
    cut = encode_record(TOK, INVOICE, max_length=fixed + 10)
    assert cut.state_tokens == 10 and cut.state_truncated and len(cut.ids) == fixed + 10
    cap = encode_record(TOK, INVOICE, max_state_tokens=5)
    assert cap.state_tokens == 5 and len(cap.ids) == fixed + 5
    # spans move with the shorter state but still decode to the same text
    for e in (cut, cap):
        s, t = e.q_span[1]
        assert TOK.decode(e.ids[s:t]) == "Is the total above 1000 USD?"
    with pytest.raises(ValueError):
        encode_record(TOK, INVOICE, max_length=fixed - 1)


def test_bad_questions_are_rejected():
    with pytest.raises(ValueError):
        encode_record(TOK, {"state": "s", "questions": {}})
    with pytest.raises(ValueError):
        encode_record(TOK, {"state": "s", "questions": {"q": {"type": "rank"}}})
    with pytest.raises(ValueError):
        encode_record(TOK, {"state": "s", "questions": {"q": {"type": "choice"}}})
    with pytest.raises(ValueError):
        encode_record(TOK, {"state": "s", "questions": {"q": {"type": "score", "criteria": {"1": "a", "2": "b"}}}})


def test_collate_pads_right_and_builds_the_tables():
    recs = [INVOICE, {"state": "Our checkout started returning errors.",
                      "questions": {"outage": {"type": "noul", "instructions": "Is a service down?"}}}]
    enc = [encode_record(TOK, r) for r in recs]
    bt = collate_records(enc, TOK.pad_token_id)
    assert bt.B == 2 and bt.Lpad == max(len(e.ids) for e in enc)
    assert list(bt.lengths) == [len(e.ids) for e in enc]
    assert (bt.token_ids[1, len(enc[1].ids):] == TOK.pad_token_id).all()
    assert list(bt.q_rec) == [0, 0, 0, 1] and list(bt.q_type) == [1, 0, 2, 0]
    assert list(np.diff(bt.q_opt_off)) == [3, 2, 3, 2]
    assert bt.o_span.shape == (10, 2) and (bt.o_span[:, 1] <= bt.lengths[np.repeat(bt.q_rec, np.diff(bt.q_opt_off))]).all()
