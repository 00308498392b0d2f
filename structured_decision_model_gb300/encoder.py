"""Host-side record encoding and batching: prompt layout, span tables, truncation.

Follows the readout contract of "clef_flash_decode_fp16_pf64 metadata.json" (prompt,
spans, option_order, question_types, noul_default_criteria) and the batching rules of
"making Clef-Flash inference faster: collate, max_length, max_state_tokens":

  prompt = prefix + state + schema + suffix, every piece tokenized on its own and the
  ids concatenated (no image block: media input is out of scope here);
  schema = a header, then per question i (1-based) its FIELD / ID / TYPE / INSTRUCTION
  lines, the instruction text, an ALLOWED OPTIONS line and one OPTION j line per option
  in the head's option order, then END FIELD;
  question span = the tokens of render(instructions or id);
  option span   = the tokens of render({option_id: description});
  the last token of the row is the suffix's final ':' (the head's global row);
  truncation: the schema is kept whole; the state is cut to what is left of max_length
  (and to max_state_tokens); a schema that alone exceeds max_length is an error.

The tokenizer is any object with ``encode(text) -> list[int]``.  The release tokenizer
is not available here, so ``ByteTokenizer`` stands in: it maps the chat-template
markers to single reserved ids and every other UTF-8 byte to one id.  Spans, layout and
truncation do not depend on which tokenizer is used.
"""
import json
import re
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

from .answers import TYPE_IDS, option_order

SYSTEM_PROMPT = ("Read the complete state and schema. Decide every field jointly. "
                 "Each answer must be exactly one of that field's allowed options.")
PREFIX = "<|im_start|>system\n" + SYSTEM_PROMPT + "<|im_end|>\n<|im_start|>user\nSTATE:\n"
SCHEMA_HEADER = "\n\nSCHEMA FIELDS:\n"
SUFFIX = "\n<|im_end|>\n<|im_start|>assistant\n<think>\n\n</think>\n\nJOINT SCHEMA DECISIONS:"
NOUL_CRITERIA = {"true": "The proposition is true or the answer is yes.",
                 "false": "The proposition is false or the answer is no."}


def render(x) -> str:
    """A string as it is; anything else as compact JSON with sorted keys, non-ASCII kept."""
    if isinstance(x, str):
        return x
    return json.dumps(x, sort_keys=True, ensure_ascii=False, separators=(",", ":"))


class ByteTokenizer:
    """Stand-in tokenizer: chat-template markers are single ids, other text one id per
    UTF-8 byte (ids 0..255).  ``pad_token_id`` pads collated rows."""

    SPECIAL = ["<|im_start|>", "<|im_end|>", "<think>", "</think>", "<|endoftext|>"]

    def __init__(self):
        self.special_ids = {s: 256 + k for k, s in enumerate(self.SPECIAL)}
        self._split = re.compile("(" + "|".join(re.escape(s) for s in self.SPECIAL) + ")")
        self.pad_token_id = self.special_ids["<|endoftext|>"]
        self.vocab_size = 256 + len(self.SPECIAL)

    def encode(self, text: str) -> List[int]:
        ids: List[int] = []
        for piece in self._split.split(text):
            if not piece:
                continue
            sid = self.special_ids.get(piece)
            if sid is not None:
                ids.append(sid)
            else:
                ids.extend(piece.encode("utf-8"))
        return ids

    def decode(self, ids: Sequence[int]) -> str:
        inv = {v: k for k, v in self.special_ids.items()}
        out, buf = [], bytearray()
        for t in ids:
            if t in inv:
                out.append(buf.decode("utf-8", errors="replace"))
                buf = bytearray()
                out.append(inv[t])
            else:
                buf.append(int(t))
        out.append(buf.decode("utf-8", errors="replace"))
        return "".join(out)


@dataclass
class EncodedRecord:
    ids: List[int]
    question_ids: List[str]
    question_types: List[int]              # 0 noul, 1 choice, 2 score
    q_span: List[tuple]                    # [start, end) of each instruction
    options: List[List[str]]               # option ids in head order, per question
    o_span: List[List[tuple]]              # [start, end) of each option, per question
    legends: List[Optional[dict]]          # score questions: level -> criterion
    state_tokens: int                      # state tokens kept after truncation
    state_truncated: bool = False
    meta: dict = field(default_factory=dict)


def _question_options(q: dict):
    """(option ids in head order, {option id: description}) of one question."""
    qtype = q.get("type")
    if qtype not in TYPE_IDS:
        raise ValueError(f"unknown question type {qtype!r}")
    criteria = q.get("criteria")
    if qtype == "noul":
        criteria = dict(NOUL_CRITERIA) if not criteria else {str(k): v for k, v in criteria.items()}
        order = option_order("noul")
        if set(criteria) != set(order):
            raise ValueError("a noul question's criteria must be exactly 'true' and 'false'")
    else:
        if not criteria:
            raise ValueError(f"a {qtype} question needs criteria")
        criteria = {str(k): v for k, v in criteria.items()}
        order = option_order(qtype, criteria)
        if qtype == "score" and set(criteria) != set(order):
            raise ValueError("a score question's criteria must be keyed by the levels 0..n-1")
    return order, criteria


def encode_record(tokenizer, record: dict, max_length: int = 16384,
                  max_state_tokens: Optional[int] = None) -> EncodedRecord:
    """Token ids and span tables of one record ({"state": ..., "questions": {id: {...}}})."""
    questions = record.get("questions") or {}
    if not questions:
        raise ValueError("a record needs at least one question")
    prefix = tokenizer.encode(PREFIX)
    suffix = tokenizer.encode(SUFFIX)
    # the schema, with spans relative to its start
    schema: List[int] = list(tokenizer.encode(SCHEMA_HEADER))
    qids, qtypes, qspans, opts, ospans, legends = [], [], [], [], [], []
    for i, (qid, q) in enumerate(questions.items(), start=1):
        order, criteria = _question_options(q)
        schema += tokenizer.encode(f"\nFIELD {i}\nID: {qid}\nTYPE: {q['type']}\nINSTRUCTION: ")
        instr = tokenizer.encode(render(q.get("instructions") or qid))
        if not instr:
            raise ValueError(f"question {qid!r}: empty instruction")
        qspans.append((len(schema), len(schema) + len(instr)))
        schema += instr
        schema += tokenizer.encode("\nALLOWED OPTIONS:\n")
        spans = []
        for j, oid in enumerate(order, start=1):
            schema += tokenizer.encode(f"OPTION {j}: ")
            body = tokenizer.encode(render({oid: criteria[oid]}))
            spans.append((len(schema), len(schema) + len(body)))
            schema += body
            schema += tokenizer.encode("\n")
        schema += tokenizer.encode("END FIELD\n")
        qids.append(str(qid))
        qtypes.append(TYPE_IDS[q["type"]])
        opts.append(order)
        ospans.append(spans)
        legends.append({lv: criteria[lv] for lv in order} if q["type"] == "score" else None)
    fixed = len(prefix) + len(schema) + len(suffix)
    if fixed > max_length:
        raise ValueError(f"the schema and the fixed prompt take {fixed} tokens, more than "
                         f"max_length={max_length} leaves before any state")
    state = tokenizer.encode(render(record.get("state", "")))
    budget = max_length - fixed
    if max_state_tokens is not None:
        budget = min(budget, max_state_tokens)
    truncated = len(state) > budget
    state = state[:budget]
    base = len(prefix) + len(state)
    ids = prefix + state + schema + suffix
    return EncodedRecord(
        ids=ids, question_ids=qids, question_types=qtypes,
        q_span=[(s + base, e + base) for s, e in qspans], options=opts,
        o_span=[[(s + base, e + base) for s, e in sp] for sp in ospans], legends=legends,
        state_tokens=len(state), state_truncated=truncated)


@dataclass
class CollatedBatch:
    """The head's inputs for a batch, right-padded to the longest record."""
    token_ids: np.ndarray     # int32 [B, Lpad]
    lengths: np.ndarray       # int32 [B]
    q_rec: np.ndarray         # int32 [Q]
    q_type: np.ndarray        # int32 [Q]
    q_span: np.ndarray        # int32 [Q, 2]
    q_opt_off: np.ndarray     # int32 [Q + 1]
    o_span: np.ndarray        # int32 [O, 2]
    question_ids: List[str]
    question_types: List[int]
    options: List[List[str]]
    legends: List[Optional[dict]]

    @property
    def B(self):
        return int(self.lengths.shape[0])

    @property
    def Lpad(self):
        return int(self.token_ids.shape[1])


def collate_records(encoded: Sequence[EncodedRecord], pad_token_id: int) -> CollatedBatch:
    """Stacks encoded records into padded id rows and the batch's span tables (spans
    index each record's own row; records keep their order)."""
    if not encoded:
        raise ValueError("nothing to collate")
    lengths = np.array([len(e.ids) for e in encoded], np.int32)
    ids = np.full((len(encoded), int(lengths.max())), pad_token_id, np.int32)
    q_rec, q_type, q_span, o_span, off = [], [], [], [], [0]
    qids, qtypes, options, legends = [], [], [], []
    for b, e in enumerate(encoded):
        ids[b, :len(e.ids)] = e.ids
        for k in range(len(e.question_ids)):
            q_rec.append(b)
            q_type.append(e.question_types[k])
            q_span.append(e.q_span[k])
            o_span.extend(e.o_span[k])
            off.append(len(o_span))
            qids.append(e.question_ids[k])
            qtypes.append(e.question_types[k])
            options.append(e.options[k])
            legends.append(e.legends[k])
    return CollatedBatch(token_ids=ids, lengths=lengths, q_rec=np.array(q_rec, np.int32),
                         q_type=np.array(q_type, np.int32), q_span=np.array(q_span, np.int32).reshape(-1, 2),
                         q_opt_off=np.array(off, np.int32), o_span=np.array(o_span, np.int32).reshape(-1, 2),
                         question_ids=qids, question_types=qtypes, options=options, legends=legends)
