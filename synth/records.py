"""Seeded synthetic record batches: hidden states, lengths, span tables, token ids.

The layout of one record follows the prompt layout the CoreAI metadata page
("clef-flash-CoreAI metadata.json", keys decision.prompt.layout / prefix_tokens /
suffix_tokens / schema) describes: a 36-row prefix, the state, the schema and an
18-row suffix whose last row is the ':' token the head reads as the global vector.
Inside the schema every question has a template gap (FIELD / ID / TYPE /
INSTRUCTION:), the instruction span, a gap (ALLOWED OPTIONS:), then per option a
gap ("OPTION j: "), the option span and one newline row, then "END FIELD".

Schema fitting mirrors the schema-first budget of the inference-tuning page
("Clef-Flash inference tuning checklist", tip 2): the state is cut, the schema is
kept; when even the schema does not fit, trailing questions are dropped here
(the real encoder raises instead; a synthetic batch must still be valid).
"""
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

from .bf16 import f32_to_bf16

PREFIX_ROWS = 36
SUFFIX_ROWS = 18
MIN_STATE_ROWS = 16
SCHEMA_HEADER_ROWS = 5
QUESTION_GAP_ROWS = 12
INSTRUCTION_GAP_ROWS = 4
OPTION_GAP_ROWS = 3
OPTION_TAIL_ROWS = 1
END_FIELD_ROWS = 3

NOUL, CHOICE, SCORE = 0, 1, 2
VOCAB = 248320

# salts keep the independent random streams apart
_SALT_LENGTHS, _SALT_SCHEMA, _SALT_HIDDEN, _SALT_IDS, _SALT_LEXICAL, _SALT_SCALE = 11, 12, 13, 14, 15, 16


@dataclass
class BatchSpec:
    """How to draw one batch (all ranges inclusive)."""
    name: str
    B: int
    H: int = 4096
    vocab: int = VOCAB
    lengths: Optional[Sequence[int]] = None        # fixed lengths, or None to draw
    length_law: str = "fixed"                      # fixed | uniform | lognormal
    length_range: tuple = (1024, 4096)             # uniform law bounds, lognormal clip
    lognormal: tuple = (1500.0, 0.8)               # median, sigma
    questions: tuple = (4, 8)                      # questions per record
    options: tuple = (2, 6)                        # options per choice / score question
    type_probs: tuple = (1 / 3, 1 / 3, 1 / 3)      # noul, choice, score
    fixed_types: Optional[Sequence[tuple]] = None  # [(type, n_options)] for every record
    instr_len: tuple = (8, 40)
    option_len: tuple = (3, 20)
    row_scale: Optional[tuple] = None              # per-row RMS scale U(lo, hi)
    lpad: Optional[int] = None                     # pad beyond max length


WORKLOADS = {
    "pr1_ref_b1_l512": BatchSpec(
        name="pr1_ref_b1_l512", B=1, lengths=[512],
        fixed_types=[(NOUL, 2), (CHOICE, 3), (SCORE, 5)], instr_len=(4, 16), option_len=(4, 16)),
    "batch32_l1k_4k": BatchSpec(
        name="batch32_l1k_4k", B=32, length_law="uniform", length_range=(1024, 4096),
        questions=(4, 8), options=(2, 6)),
    "batch8_l16k": BatchSpec(
        name="batch8_l16k", B=8, lengths=[16384] * 8, questions=(16, 16), options=(2, 8),
        row_scale=(0.5, 2.0)),
    "wide_h5120_b16_l8k": BatchSpec(
        name="wide_h5120_b16_l8k", B=16, H=5120, lengths=[8192] * 16, questions=(8, 8),
        options=(2, 10)),
    "serving_mix_b64": BatchSpec(
        name="serving_mix_b64", B=64, length_law="lognormal", length_range=(256, 16384),
        questions=(1, 32), options=(2, 10), type_probs=(0.4, 0.4, 0.2)),
    "short_b256": BatchSpec(
        name="short_b256", B=256, length_law="lognormal", length_range=(256, 512),
        questions=(1, 32), options=(2, 10), type_probs=(0.4, 0.4, 0.2)),
}


def workload_spec(name: str) -> BatchSpec:
    return WORKLOADS[name]


class SparseLexical:
    """The output-embedding (lexical) table [vocab, H] with row r drawn on demand.

    Row r is N(0, 0.02) from a generator seeded by (seed, r), so any subset of rows
    can be materialised without drawing the whole 248320-row table.
    """

    def __init__(self, seed: int, vocab: int, H: int):
        self.seed, self.vocab, self.H = seed, vocab, H
        self._cache = {}

    def row(self, r: int) -> np.ndarray:
        r = int(r)
        if not 0 <= r < self.vocab:
            raise IndexError(f"lexical row {r} outside [0, {self.vocab})")
        got = self._cache.get(r)
        if got is None:
            g = np.random.default_rng([self.seed, _SALT_LEXICAL, r])
            got = f32_to_bf16(g.standard_normal(self.H, dtype=np.float32) * np.float32(0.02))
            self._cache[r] = got
        return got

    def __getitem__(self, ids) -> np.ndarray:
        ids = np.asarray(ids)
        flat = [self.row(r) for r in ids.reshape(-1)]
        out = np.stack(flat) if flat else np.zeros((0, self.H), np.uint16)
        return out.reshape(ids.shape + (self.H,))

    def dense(self) -> np.ndarray:
        """The whole table (only sensible for small test vocabularies)."""
        return self[np.arange(self.vocab)]


@dataclass
class Batch:
    spec: BatchSpec
    seed: int
    H: int
    B: int
    Lpad: int
    lengths: np.ndarray      # int32 [B]
    q_rec: np.ndarray        # int32 [Q], non-decreasing
    q_type: np.ndarray       # int32 [Q]
    q_span: np.ndarray       # int32 [Q, 2] instruction [start, end)
    q_opt_off: np.ndarray    # int32 [Q + 1] CSR into the option table
    o_span: np.ndarray       # int32 [O, 2] option [start, end)
    token_ids: np.ndarray    # int32 [B, Lpad]
    lexical: SparseLexical
    hidden: Optional[np.ndarray] = field(default=None, repr=False)  # uint16 bf16 [B, Lpad, H]

    @property
    def Q(self):
        return int(self.q_type.shape[0])

    @property
    def O(self):
        return int(self.o_span.shape[0])

    @property
    def T(self):
        return int(self.lengths.sum())

    def lexical_ids(self) -> np.ndarray:
        """Sorted unique token ids read by the option spans (the lexical rows in use)."""
        o_rec = np.repeat(self.q_rec, np.diff(self.q_opt_off))
        ids = [self.token_ids[o_rec[j], self.o_span[j, 0]:self.o_span[j, 1]] for j in range(self.O)]
        return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int32)

    def record_hidden(self, b: int) -> np.ndarray:
        """Hidden rows [Lpad, H] of record b (drawn on demand when not held)."""
        if self.hidden is not None:
            return self.hidden[b]
        return draw_hidden_record(self.seed, b, self.Lpad, self.H, self.spec.row_scale)

    def real_rows(self, b: int) -> np.ndarray:
        """The real rows [L_b, H] of record b: the same values as the first L_b rows of
        ``record_hidden(b)``, without drawing the padding."""
        if self.hidden is not None:
            return self.hidden[b, :self.lengths[b]]
        return draw_hidden_record(self.seed, b, int(self.lengths[b]), self.H, self.spec.row_scale)


def _draw_lengths(spec: BatchSpec, rng) -> np.ndarray:
    if spec.lengths is not None:
        return np.asarray(spec.lengths, np.int64)
    lo, hi = spec.length_range
    if spec.length_law == "uniform":
        return rng.integers(lo, hi + 1, size=spec.B)
    if spec.length_law == "lognormal":
        med, sigma = spec.lognormal
        out = np.empty(spec.B, np.int64)
        for b in range(spec.B):
            while True:  # rejection-sample inside the clip range
                v = int(round(med * np.exp(sigma * rng.standard_normal())))
                if hi >= 16384:
                    out[b] = min(max(v, lo), hi)
                    break
                if v <= hi:
                    out[b] = max(v, lo)
                    break
        return out
    raise ValueError(spec.length_law)


def _schema_rows(qs):
    rows = SCHEMA_HEADER_ROWS
    for (_t, instr, opts) in qs:
        rows += QUESTION_GAP_ROWS + instr + INSTRUCTION_GAP_ROWS + END_FIELD_ROWS
        rows += sum(OPTION_GAP_ROWS + s + OPTION_TAIL_ROWS for s in opts)
    return rows


def _draw_schema(spec: BatchSpec, rng, L: int):
    """Questions for one record as [(type, instr_len, [option lens])], fitted to L."""
    if spec.fixed_types is not None:
        plan = list(spec.fixed_types)
    else:
        nq = int(rng.integers(spec.questions[0], spec.questions[1] + 1))
        types = rng.choice(3, size=nq, p=np.asarray(spec.type_probs) / np.sum(spec.type_probs))
        plan = []
        for t in types:
            n = 2 if t == NOUL else int(rng.integers(spec.options[0], spec.options[1] + 1))
            plan.append((int(t), n))
    qs = []
    for (t, n) in plan:
        instr = int(rng.integers(spec.instr_len[0], spec.instr_len[1] + 1))
        opts = [int(v) for v in rng.integers(spec.option_len[0], spec.option_len[1] + 1, size=n)]
        qs.append((t, instr, opts))
    budget = L - PREFIX_ROWS - SUFFIX_ROWS - MIN_STATE_ROWS
    while len(qs) > 1 and _schema_rows(qs) > budget:
        qs.pop()
    if _schema_rows(qs) > budget:  # one question left: shrink it to the minimum
        t = qs[0][0]
        qs = [(t, min(qs[0][1], 3), [3, 3])]
        if _schema_rows(qs) > budget:
            raise ValueError(f"record length {L} cannot hold a one-question schema")
    return qs


def draw_hidden_record(seed: int, b: int, Lpad: int, H: int, row_scale=None) -> np.ndarray:
    """Hidden rows of record b: bf16 N(0,1), times a per-row U(lo,hi) scale if given.

    Padding rows (t >= L_b) are drawn the same way: the head must ignore them.
    """
    g = np.random.default_rng([seed, _SALT_HIDDEN, b])
    x = g.standard_normal((Lpad, H), dtype=np.float32)
    if row_scale is not None:
        gs = np.random.default_rng([seed, _SALT_SCALE, b])
        s = gs.uniform(row_scale[0], row_scale[1], size=(Lpad, 1)).astype(np.float32)
        x *= s
    return f32_to_bf16(x)


def make_batch(spec: BatchSpec, seed: int = 1, with_hidden: bool = True, lpad: Optional[int] = None) -> Batch:
    """Draw one batch.  Everything is a pure function of (spec, seed)."""
    rng_len = np.random.default_rng([seed, _SALT_LENGTHS])
    lengths = _draw_lengths(spec, rng_len).astype(np.int64)
    if len(lengths) != spec.B:
        raise ValueError("lengths do not match B")
    Lpad = int(max(lengths.max(), lpad or 0, spec.lpad or 0))

    q_rec, q_type, q_span, q_opt_off, o_span = [], [], [], [0], []
    for b in range(spec.B):
        rng = np.random.default_rng([seed, _SALT_SCHEMA, b])
        L = int(lengths[b])
        qs = _draw_schema(spec, rng, L)
        pos = L - SUFFIX_ROWS - _schema_rows(qs) + SCHEMA_HEADER_ROWS
        for (t, instr, opts) in qs:
            pos += QUESTION_GAP_ROWS
            q_rec.append(b)
            q_type.append(t)
            q_span.append((pos, pos + instr))
            pos += instr + INSTRUCTION_GAP_ROWS
            for s in opts:
                pos += OPTION_GAP_ROWS
                o_span.append((pos, pos + s))
                pos += s + OPTION_TAIL_ROWS
            q_opt_off.append(len(o_span))
            pos += END_FIELD_ROWS
        assert pos == L - SUFFIX_ROWS, (pos, L)

    ids = np.empty((spec.B, Lpad), np.int32)
    for b in range(spec.B):
        g = np.random.default_rng([seed, _SALT_IDS, b])
        ids[b] = g.integers(0, spec.vocab, size=Lpad, dtype=np.int64).astype(np.int32)

    batch = Batch(
        spec=spec, seed=seed, H=spec.H, B=spec.B, Lpad=Lpad,
        lengths=lengths.astype(np.int32),
        q_rec=np.asarray(q_rec, np.int32), q_type=np.asarray(q_type, np.int32),
        q_span=np.asarray(q_span, np.int32).reshape(-1, 2),
        q_opt_off=np.asarray(q_opt_off, np.int32),
        o_span=np.asarray(o_span, np.int32).reshape(-1, 2),
        token_ids=ids, lexical=SparseLexical(seed, spec.vocab, spec.H))
    if with_hidden:
        hid = np.empty((spec.B, Lpad, spec.H), np.uint16)
        for b in range(spec.B):
            hid[b] = draw_hidden_record(seed, b, Lpad, spec.H, spec.row_scale)
        batch.hidden = hid
    return batch
