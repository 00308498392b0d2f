"""Plain fp64 oracle of the Clef JointSchemaHead forward pass.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg; never by the library or its binding.

Sources (web pages, cited by title and section):
  [walkthrough]  "clef-4bit: JointSchemaHead walkthrough" (2kiu.com), section 3
                 steps 1-4 — pooling, evidence routing, field aggregation, scoring.
  [dissect]      "Dissecting the Clef-Flash architecture" (lshu.cn), section 3.2
                 head config table and its four-step summary.
  [overview]     "Clef-Flash overview" (lmnt.cn), section 3 "joint schema head".
  [coreai]       "clef-flash-CoreAI metadata.json", keys decision.spans,
                 decision.option_order, decision.question_types, decision.head.reads,
                 decision.head.lexical, decision.softmax, decision.response.
  [tuning]       "Clef-Flash inference tuning checklist" (gsyq.cn), tip 1 (batches
                 are padded to the longest record).

Where the pages leave a step open, each function states the reading it follows:
pre-LN layers, exact GELU, biases on every Linear (one summed bias for the three
option-query and for the three field projections), eps 1e-5, the option summary as a
learned attention pooling, the prior cosine in the backbone space on the raw pooled
vectors, right padding, a 4D -> D -> 1 scorer MLP, one learned gate and one learned
joint scale.

All arithmetic is fp64; bf16 inputs and weights are widened exactly.
"""
from dataclasses import dataclass

import numpy as np
from scipy.special import erf, expit

EPS_LN = 1e-5   # reading: LayerNorm eps (pages silent)
EPS_COS = 1e-8  # reading: cosine denominators clamp each norm at 1e-8 (pages silent)


def _f64(a):
    """bf16 bit patterns (uint16) or floats -> float64, exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------- primitives

def layer_norm(x, w, b, eps=EPS_LN):
    """Affine LayerNorm over the last axis, biased variance.

    [coreai] decision.head.reads: the hidden rows pass a LayerNorm(4096) before
    they become memory; the same affine form is used for the head's inner norms.
    """
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * w + b


def gelu(x):
    """Exact GELU 0.5 x (1 + erf(x / sqrt 2)) (reading: pages name no activation)."""
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def linear(x, W, b=None):
    """torch-style Linear: x W^T + b, W is [out, in]."""
    y = x @ W.T
    return y if b is None else y + b


def cosine(a, b, eps=EPS_COS):
    """Row-wise cosine a.b / (max(|a|, eps) max(|b|, eps))."""
    na = np.maximum(np.linalg.norm(a, axis=-1), eps)
    nb = np.maximum(np.linalg.norm(b, axis=-1), eps)
    return (a * b).sum(axis=-1) / (na * nb)


def softmax(z, axis=-1):
    z = z - z.max(axis=axis, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=axis, keepdims=True)


# ------------------------------------------------------------------ weights

@dataclass
class HeadParams:
    """The head's tensors widened to fp64, addressed by their state-dict names."""
    t: dict
    heads: int
    n_route: int
    n_joint: int

    @classmethod
    def from_bf16(cls, weights: dict, heads: int, n_route: int, n_joint: int):
        return cls({k: _f64(v) for k, v in weights.items()}, heads, n_route, n_joint)

    def __getitem__(self, k):
        return self.t[k]


# ----------------------------------------------------------- step 1: pooling

def memory_rows(hidden_b, L_b, p: HeadParams):
    """Memory of one record: LayerNorm of its real hidden rows 0..L_b-1.

    [coreai] decision.head.reads ("LayerNorm(4096) -> memory"); right padding is the
    reading for "padded to the longest" of [tuning] tip 1, so rows >= L_b are pad.
    """
    return layer_norm(_f64(hidden_b[:L_b]), p["mem_ln.weight"], p["mem_ln.bias"])


def pool_record(mem, L_b, q_span, o_span, o_ids, lexical):
    """Pooled vectors of one record.

    [walkthrough] section 3 step 1 and [coreai] decision.spans / head.reads / lexical:
      u_q = mean of memory rows over the question's instruction span [start, end)
      c_j = mean of memory rows over option j's span
      x_j = mean of output-embedding (lm_head) rows of the token ids in option j's span
      g   = memory row of the last token (row L_b - 1)
    ``o_ids`` holds the token ids of each option span; ``lexical`` maps ids to bf16 rows.
    """
    u = np.stack([mem[s:e].mean(axis=0) for (s, e) in q_span])
    c = np.stack([mem[s:e].mean(axis=0) for (s, e) in o_span])
    x = np.stack([_f64(lexical[np.asarray(ids)]).mean(axis=0) for ids in o_ids])
    g = mem[L_b - 1]
    return u, c, x, g


def span_raw_sums(hidden_b, q_span, o_span, o_ids, lexical):
    """Un-normalised span sums of raw hidden rows and lexical rows (index checks).

    Same spans as ``pool_record`` but summed before the LayerNorm and without the
    division: with small-integer inputs these sums are exact in any precision, so
    they check span / offset / gather indexing bit for bit.
    """
    h = _f64(hidden_b)
    sq = np.stack([h[s:e].sum(axis=0) for (s, e) in q_span])
    so = np.stack([h[s:e].sum(axis=0) for (s, e) in o_span])
    sx = np.stack([_f64(lexical[np.asarray(ids)]).sum(axis=0) for ids in o_ids])
    return sq, so, sx


def option_query(c, x, u_of_opt, p: HeadParams):
    """Option query = context projection + lexical projection + question projection.

    [walkthrough] section 3 step 1 (the three-part sum).  Reading: the three
    projections share one summed bias.
    """
    return (linear(c, p["query.ctx.weight"]) + linear(x, p["query.lex.weight"])
            + linear(u_of_opt, p["query.question.weight"]) + p["query.bias"])


# ------------------------------------------------------ step 2: evidence routing

def cross_attention(qx, mem, Wq, bq, Wk, bk, Wv, bv, heads):
    """Multi-head attention of the rows of ``qx`` over every memory row.

    [walkthrough] section 3 step 2: every option is a query attending the whole
    memory.  Readings: K and V are projections of the H-wide memory, head dim
    D/heads, scale 1/sqrt(head dim), no mask besides the record's own rows (the
    caller passes only rows 0..L_b-1).  Returns the concatenated heads [n, D].
    """
    Qm, Km, Vm = linear(qx, Wq, bq), linear(mem, Wk, bk), linear(mem, Wv, bv)
    n, D = Qm.shape
    dh = D // heads
    out = np.empty((n, D))
    for h in range(heads):
        sl = slice(h * dh, (h + 1) * dh)
        s = Qm[:, sl] @ Km[:, sl].T / np.sqrt(dh)
        out[:, sl] = softmax(s, axis=1) @ Vm[:, sl]
    return out


def routing_layer(o, mem, l, p: HeadParams):
    """One EvidenceRoutingLayer: cross-attention to memory, then FFN, with residuals.

    [walkthrough] section 3 step 2 ("cross-attention" then "FFN + residual");
    [dissect] section 3.2 (2 routing layers, 16 heads, feedforward 4096).
    Readings: pre-LN on the option stream before attention and before the FFN,
    exact GELU, no self-attention among options.
    """
    q = f"route.{l}."
    a = layer_norm(o, p[q + "attn_ln.weight"], p[q + "attn_ln.bias"])
    att = cross_attention(a, mem, p[q + "q.weight"], p[q + "q.bias"], p[q + "k.weight"],
                          p[q + "k.bias"], p[q + "v.weight"], p[q + "v.bias"], p.heads)
    o = o + linear(att, p[q + "o.weight"], p[q + "o.bias"])
    hdn = gelu(linear(layer_norm(o, p[q + "ffn_ln.weight"], p[q + "ffn_ln.bias"]),
                      p[q + "ffn1.weight"], p[q + "ffn1.bias"]))
    return o + linear(hdn, p[q + "ffn2.weight"], p[q + "ffn2.bias"])


# ------------------------------------------- step 3: fields and joint layers

def field_aggregate(u_q, o_hat_q, g, qtype, p: HeadParams):
    """Field vector of one question.

    [walkthrough] section 3 step 3: question base vector + option-weighted summary
    + global vector (the last hidden state) + type embedding.  Readings: the summary
    is a learned attention pooling alpha = softmax_j(w_a . o_j + b_a) over the
    question's final option vectors; base, summary and global vectors are each
    projected to the width, and the three projections share one summed bias.
    """
    a = softmax(linear(o_hat_q, p["field.pool.weight"], p["field.pool.bias"])[:, 0])
    summary = a @ o_hat_q
    return (linear(u_q, p["field.question.weight"]) + linear(summary, p["field.summary.weight"])
            + linear(g, p["field.global.weight"]) + p["field.bias"]
            + p["field.type_embedding"][qtype])


def self_attention(f, Wqkv, bqkv, heads):
    """Multi-head self-attention among the rows of ``f`` (all mutually visible)."""
    n, D = f.shape
    qkv = linear(f, Wqkv, bqkv)
    Qm, Km, Vm = qkv[:, :D], qkv[:, D:2 * D], qkv[:, 2 * D:]
    dh = D // heads
    out = np.empty((n, D))
    for h in range(heads):
        sl = slice(h * dh, (h + 1) * dh)
        out[:, sl] = softmax(Qm[:, sl] @ Km[:, sl].T / np.sqrt(dh), axis=1) @ Vm[:, sl]
    return out


def joint_layer(f, i, p: HeadParams):
    """One joint transformer layer over one record's fields.

    [walkthrough] section 3 step 3 (4 standard layers, fields mutually visible);
    [dissect] section 3.2 (layers 4, width 1024, 16 heads, feedforward 4096).
    Readings: pre-LN self-attention + FFN, no causal mask, no field positions.
    """
    q = f"joint.{i}."
    a = layer_norm(f, p[q + "attn_ln.weight"], p[q + "attn_ln.bias"])
    f = f + linear(self_attention(a, p[q + "qkv.weight"], p[q + "qkv.bias"], p.heads),
                   p[q + "o.weight"], p[q + "o.bias"])
    hdn = gelu(linear(layer_norm(f, p[q + "ffn_ln.weight"], p[q + "ffn_ln.bias"]),
                      p[q + "ffn1.weight"], p[q + "ffn1.bias"]))
    return f + linear(hdn, p[q + "ffn2.weight"], p[q + "ffn2.bias"])


# --------------------------------------------------------- step 4: the scorer

def scorer_logits(x_q, u_q, g, f_hat, o_hat_q, p: HeadParams):
    """Logits of one question's options.

    [walkthrough] section 3 step 4:
      logit = prior + gate * (joint_scale * cos(field, option) + MLP([f, o, f*o, |f-o|]))
    with prior = cos(option lexical vector, question + global anchor) and a sigmoid
    gate.  Readings: the prior lives in the backbone space on the raw pooled vectors;
    gate = sigmoid of one learned scalar; joint_scale is one learned scalar; the MLP
    is 4D -> D -> GELU -> 1.
    """
    prior = cosine(x_q, (u_q + g)[None, :])
    f = np.broadcast_to(f_hat, o_hat_q.shape)
    joint = cosine(f, o_hat_q)
    z = np.concatenate([f, o_hat_q, f * o_hat_q, np.abs(f - o_hat_q)], axis=1)
    mlp = linear(gelu(linear(z, p["scorer.mlp1.weight"], p["scorer.mlp1.bias"])),
                 p["scorer.mlp2.weight"], p["scorer.mlp2.bias"])[:, 0]
    gate = expit(p["scorer.gate"][0])  # logistic sigmoid
    return prior + gate * (p["scorer.joint_scale"][0] * joint + mlp)


def question_softmax(logits):
    """Per-question softmax, temperature 1 ([coreai] decision.softmax)."""
    return softmax(np.asarray(logits, np.float64))


def answers(qtype, probs):
    """(value, confidence, argmax) of one question ([coreai] decision.response).

    noul: value = p(true), the first option; choice: value = confidence = max p;
    score: value = sum(level * p) over levels 0..n-1, confidence = max p.  argmax is
    the first maximum in option order.
    """
    k = int(np.argmax(probs))
    conf = float(probs[k])
    if qtype == 0:
        value = float(probs[0])
    elif qtype == 1:
        value = conf
    else:
        value = float(np.dot(np.arange(len(probs)), probs))
    return value, conf, k


# ---------------------------------------------------------------- the head

def head_forward(weights, heads, n_route, n_joint, hidden, lengths, q_rec, q_type, q_span,
                 q_opt_off, o_span, token_ids, lexical, records=None, keep=False):
    """Whole head on a batch; records are independent, so ``records`` may pick a subset.

    ``hidden`` is a bf16 array [B, Lpad, H] or a callable b -> [Lpad, H].  Returns a
    dict of per-option ``logits`` / ``probs`` and per-question ``value`` / ``conf`` /
    ``argmax``; entries of records that were not computed are NaN (-1 for argmax).
    """
    p = weights if isinstance(weights, HeadParams) else HeadParams.from_bf16(weights, heads, n_route, n_joint)
    q_rec = np.asarray(q_rec)
    Q, O = len(q_type), int(q_opt_off[-1])
    out = {"logits": np.full(O, np.nan), "probs": np.full(O, np.nan), "value": np.full(Q, np.nan),
           "conf": np.full(Q, np.nan), "argmax": np.full(Q, -1, np.int64)}
    if keep:
        out["inter"] = {}
    B = len(lengths)
    for b in (range(B) if records is None else records):
        qs = np.nonzero(q_rec == b)[0]
        if len(qs) == 0:
            continue
        L_b = int(lengths[b])
        hb = hidden(b) if callable(hidden) else hidden[b]
        mem = memory_rows(hb, L_b, p)
        o_lo, o_hi = int(q_opt_off[qs[0]]), int(q_opt_off[qs[-1] + 1])
        o_sp = np.asarray(o_span[o_lo:o_hi])
        o_ids = [token_ids[b][s:e] for (s, e) in o_sp]
        u, c, x, g = pool_record(mem, L_b, np.asarray(q_span)[qs], o_sp, o_ids, lexical)
        o_q = np.repeat(np.arange(len(qs)), np.diff(np.asarray(q_opt_off)[qs[0]:qs[-1] + 2]))
        o = option_query(c, x, u[o_q], p)
        for l in range(n_route):
            o = routing_layer(o, mem, l, p)
        o_hat = layer_norm(o, p["option_ln.weight"], p["option_ln.bias"])
        f = np.stack([field_aggregate(u[k], o_hat[o_q == k], g, int(q_type[q]), p)
                      for k, q in enumerate(qs)])
        for i in range(n_joint):
            f = joint_layer(f, i, p)
        f_hat = layer_norm(f, p["field_ln.weight"], p["field_ln.bias"])
        for k, q in enumerate(qs):
            sel = o_q == k
            lg = scorer_logits(x[sel], u[k], g, f_hat[k], o_hat[sel], p)
            pr = question_softmax(lg)
            a, b_ = int(q_opt_off[q]), int(q_opt_off[q + 1])
            out["logits"][a:b_] = lg
            out["probs"][a:b_] = pr
            out["value"][q], out["conf"][q], out["argmax"][q] = answers(int(q_type[q]), pr)
        if keep:
            out["inter"][b] = dict(u=u, c=c, x=x, g=g, o_hat=o_hat, f_hat=f_hat)
    return out
