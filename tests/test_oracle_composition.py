"""Pins of the oracle's option query and of its whole-head composition (CPU only).

The option query ("clef-4bit JointSchemaHead walkthrough" section 3 step 1: context
projection + lexical projection + question projection) is checked against three
separate torch Linear modules.  The whole head (section 3 steps 1-4, in that order)
is rebuilt from torch modules -- LayerNorm, MultiheadAttention, TransformerEncoderLayer,
Linear, Embedding, cosine_similarity, softmax -- composed in the order the pages give
and the readings fix, and compared with the oracle on a tiny batch.  Each input
stream gets its own distribution, so that swapping two projections, dropping a term
or skipping a norm changes the result far beyond the tolerance.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.clef_head import HeadParams
from synth import BatchSpec, HeadShape

F64 = dict(dtype=torch.float64)
TINY = HeadShape(H=48, D=32, heads=4, F=64, vocab=500)


def T(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def params(seed, shape=TINY):
    return HeadParams.from_bf16(synth.make_weights(shape, seed), shape.heads, shape.n_route, shape.n_joint)


def _linear(w, b=None):
    lin = torch.nn.Linear(w.shape[1], w.shape[0], bias=b is not None, **F64)
    with torch.no_grad():
        lin.weight.copy_(T(w))
        if b is not None:
            lin.bias.copy_(T(b))
    return lin


def _layer_norm(p, name, n):
    ln = torch.nn.LayerNorm(n, eps=1e-5, **F64)
    with torch.no_grad():
        ln.weight.copy_(T(p[name + ".weight"]))
        ln.bias.copy_(T(p[name + ".bias"]))
    return ln


# ------------------------------------------------------------- option query

def test_option_query_matches_three_torch_linears():
    p = params(seed=31)
    rng = np.random.default_rng(40)
    n_opt, n_q = 7, 3
    # three streams with clearly different statistics: a ctx/lex swap or a missing
    # question term moves the result by O(1)
    c = rng.normal(loc=1.5, scale=2.0, size=(n_opt, TINY.H))
    x = rng.uniform(-0.05, 0.05, size=(n_opt, TINY.H))
    u = rng.normal(loc=-0.7, scale=0.5, size=(n_q, TINY.H))
    o_q = np.array([0, 0, 1, 1, 1, 2, 2])
    got = oracle.option_query(c, x, u[o_q], p)
    ctx, lex, qst = (_linear(p[k]) for k in ("query.ctx.weight", "query.lex.weight", "query.question.weight"))
    with torch.no_grad():
        ref = (ctx(T(c)) + lex(T(x)) + qst(T(u))[torch.from_numpy(o_q)] + T(p["query.bias"])).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # the plausible slips all miss by far more than the tolerance
    with torch.no_grad():
        swapped = (lex(T(c)) + ctx(T(x)) + qst(T(u))[torch.from_numpy(o_q)] + T(p["query.bias"])).numpy()
        no_question = (ctx(T(c)) + lex(T(x)) + T(p["query.bias"])).numpy()
    assert np.abs(swapped - ref).max() > 0.1
    assert np.abs(no_question - ref).max() > 0.1


def test_option_query_zero_context_and_lexical_is_question_projection():
    t = dict(params(seed=32).t)
    t["query.ctx.weight"] = np.zeros_like(t["query.ctx.weight"])
    t["query.lex.weight"] = np.zeros_like(t["query.lex.weight"])
    p = HeadParams(t, TINY.heads, TINY.n_route, TINY.n_joint)
    rng = np.random.default_rng(41)
    c, x, u = rng.normal(size=(4, TINY.H)), rng.normal(size=(4, TINY.H)), rng.normal(size=(4, TINY.H))
    closed = u @ t["query.question.weight"].T + t["query.bias"]
    np.testing.assert_allclose(oracle.option_query(c, x, u, p), closed, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- whole-head composition

class TorchHead:
    """The head rebuilt from torch modules, one record at a time, in the pages' order:
    memory LayerNorm -> span means and lexical means -> option query (three Linears,
    one bias) -> 2 x routing (pre-LN MultiheadAttention over the memory + pre-LN FFN,
    residuals) -> option LayerNorm -> learned option pooling -> field Linears + type
    Embedding -> 4 x TransformerEncoderLayer(norm_first) over the record's fields ->
    field LayerNorm -> scorer (prior cosine + sigmoid gate x (scale x joint cosine +
    MLP)) -> per-question softmax."""

    def __init__(self, p: HeadParams, shape: HeadShape):
        H, D, F = shape.H, shape.D, shape.F
        self.p, self.shape = p, shape
        self.mem_ln = _layer_norm(p, "mem_ln", H)
        self.q_ctx, self.q_lex, self.q_qst = (_linear(p[k]) for k in
                                              ("query.ctx.weight", "query.lex.weight", "query.question.weight"))
        self.routes = []
        for l in range(shape.n_route):
            q = f"route.{l}."
            mha = torch.nn.MultiheadAttention(D, shape.heads, bias=True, kdim=H, vdim=H, batch_first=True, **F64)
            with torch.no_grad():
                mha.q_proj_weight.copy_(T(p[q + "q.weight"]))
                mha.k_proj_weight.copy_(T(p[q + "k.weight"]))
                mha.v_proj_weight.copy_(T(p[q + "v.weight"]))
                mha.in_proj_bias.copy_(T(np.concatenate([p[q + "q.bias"], p[q + "k.bias"], p[q + "v.bias"]])))
                mha.out_proj.weight.copy_(T(p[q + "o.weight"]))
                mha.out_proj.bias.copy_(T(p[q + "o.bias"]))
            ffn = torch.nn.Sequential(_linear(p[q + "ffn1.weight"], p[q + "ffn1.bias"]), torch.nn.GELU(),
                                      _linear(p[q + "ffn2.weight"], p[q + "ffn2.bias"]))
            self.routes.append((_layer_norm(p, q + "attn_ln", D), mha, _layer_norm(p, q + "ffn_ln", D), ffn))
        self.option_ln = _layer_norm(p, "option_ln", D)
        self.pool = _linear(p["field.pool.weight"], p["field.pool.bias"])
        self.f_q, self.f_s, self.f_g = (_linear(p[k]) for k in
                                        ("field.question.weight", "field.summary.weight", "field.global.weight"))
        self.type_emb = torch.nn.Embedding(3, D, **F64)
        with torch.no_grad():
            self.type_emb.weight.copy_(T(p["field.type_embedding"]))
        self.joints = []
        for i in range(shape.n_joint):
            q = f"joint.{i}."
            layer = torch.nn.TransformerEncoderLayer(D, shape.heads, dim_feedforward=F, dropout=0.0,
                                                     activation="gelu", layer_norm_eps=1e-5, batch_first=True,
                                                     norm_first=True, **F64)
            with torch.no_grad():
                layer.self_attn.in_proj_weight.copy_(T(p[q + "qkv.weight"]))
                layer.self_attn.in_proj_bias.copy_(T(p[q + "qkv.bias"]))
                layer.self_attn.out_proj.weight.copy_(T(p[q + "o.weight"]))
                layer.self_attn.out_proj.bias.copy_(T(p[q + "o.bias"]))
                for a, b in (("norm1", "attn_ln"), ("norm2", "ffn_ln")):
                    getattr(layer, a).weight.copy_(T(p[q + b + ".weight"]))
                    getattr(layer, a).bias.copy_(T(p[q + b + ".bias"]))
                layer.linear1.weight.copy_(T(p[q + "ffn1.weight"]))
                layer.linear1.bias.copy_(T(p[q + "ffn1.bias"]))
                layer.linear2.weight.copy_(T(p[q + "ffn2.weight"]))
                layer.linear2.bias.copy_(T(p[q + "ffn2.bias"]))
            layer.eval()
            self.joints.append(layer)
        self.field_ln = _layer_norm(p, "field_ln", D)
        self.mlp = torch.nn.Sequential(_linear(p["scorer.mlp1.weight"], p["scorer.mlp1.bias"]), torch.nn.GELU(),
                                       _linear(p["scorer.mlp2.weight"], p["scorer.mlp2.bias"]))

    @torch.no_grad()
    def record(self, hidden_b, L_b, q_types, q_spans, opt_blocks, token_ids_b, lexical):
        """Logits and probabilities of one record's questions (lists, one per question)."""
        p = self.p
        mem = self.mem_ln(T(synth.bf16_to_f32(hidden_b[:L_b])))
        u = torch.stack([mem[s:e].mean(0) for (s, e) in q_spans])
        spans = [sp for blk in opt_blocks for sp in blk]
        c = torch.stack([mem[s:e].mean(0) for (s, e) in spans])
        x = torch.stack([T(synth.bf16_to_f32(lexical[np.asarray(token_ids_b[s:e])])).mean(0) for (s, e) in spans])
        g = mem[L_b - 1]
        o_q = torch.tensor([k for k, blk in enumerate(opt_blocks) for _ in blk])
        o = self.q_ctx(c) + self.q_lex(x) + self.q_qst(u)[o_q] + T(p["query.bias"])
        for ln1, mha, ln2, ffn in self.routes:
            a = ln1(o)
            att, _ = mha(a[None], mem[None], mem[None], need_weights=False)
            o = o + att[0]
            o = o + ffn(ln2(o))
        o_hat = self.option_ln(o)
        fields = []
        for k, t in enumerate(q_types):
            oh = o_hat[o_q == k]
            alpha = torch.softmax(self.pool(oh)[:, 0], dim=0)
            fields.append(self.f_q(u[k]) + self.f_s(alpha @ oh) + self.f_g(g) + T(p["field.bias"])
                          + self.type_emb(torch.tensor(t)))
        f = torch.stack(fields)[None]
        for layer in self.joints:
            f = layer(f)
        f_hat = self.field_ln(f[0])
        gate = torch.sigmoid(T(p["scorer.gate"])[0])
        scale = T(p["scorer.joint_scale"])[0]
        logits, probs = [], []
        for k in range(len(q_types)):
            sel = o_q == k
            xs, oh = x[sel], o_hat[sel]
            fk = f_hat[k][None].expand_as(oh)
            prior = torch.nn.functional.cosine_similarity(xs, (u[k] + g)[None].expand_as(xs), dim=1, eps=1e-8)
            joint = torch.nn.functional.cosine_similarity(fk, oh, dim=1, eps=1e-8)
            m = self.mlp(torch.cat([fk, oh, fk * oh, (fk - oh).abs()], dim=1))[:, 0]
            lg = prior + gate * (scale * joint + m)
            logits.append(lg.numpy())
            probs.append(torch.softmax(lg, dim=0).numpy())
        return logits, probs


def _tiny_batch(seed, B=2):
    spec = BatchSpec(name="tiny", B=B, H=TINY.H, vocab=TINY.vocab, length_law="uniform", length_range=(150, 260),
                     questions=(2, 4), options=(2, 5), instr_len=(3, 9), option_len=(2, 6))
    return synth.make_batch(spec, seed=seed)


@pytest.mark.parametrize("seed", [51, 52])
def test_whole_head_matches_torch_module_composition(seed):
    p = params(seed=seed)
    bt = _tiny_batch(seed)
    # the per-record hidden rows get a non-zero mean and an outlier channel, so that a
    # norm applied in the wrong place cannot hide
    hid = synth.bf16_to_f32(bt.hidden).copy()
    hid += np.random.default_rng(seed).uniform(-2, 2, size=(bt.B, bt.Lpad, 1)).astype(np.float32)
    hid[:, :, 5] *= 12.0
    bt = dataclasses.replace(bt, hidden=synth.f32_to_bf16(hid))
    ref = oracle.head_forward(p, TINY.heads, TINY.n_route, TINY.n_joint, bt.hidden, bt.lengths, bt.q_rec,
                              bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical)
    th = TorchHead(p, TINY)
    lex = bt.lexical.dense()
    for b in range(bt.B):
        qs = np.nonzero(bt.q_rec == b)[0]
        blocks = [[tuple(bt.o_span[j]) for j in range(bt.q_opt_off[q], bt.q_opt_off[q + 1])] for q in qs]
        lg, pr = th.record(bt.hidden[b], int(bt.lengths[b]), [int(t) for t in bt.q_type[qs]],
                           [tuple(s) for s in bt.q_span[qs]], blocks, bt.token_ids[b], lex)
        for k, q in enumerate(qs):
            lo, hi = bt.q_opt_off[q], bt.q_opt_off[q + 1]
            np.testing.assert_allclose(ref["logits"][lo:hi], lg[k], rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(ref["probs"][lo:hi], pr[k], rtol=1e-10, atol=1e-10)


def test_composition_pin_detects_a_skipped_option_norm():
    """The composition check is sharp: an oracle that fed raw option vectors to the
    field aggregation (a plausible slip) misses it by far more than the tolerance."""
    p = params(seed=53)
    bt = _tiny_batch(53, B=1)
    th = TorchHead(p, TINY)
    qs = np.nonzero(bt.q_rec == 0)[0]
    blocks = [[tuple(bt.o_span[j]) for j in range(bt.q_opt_off[q], bt.q_opt_off[q + 1])] for q in qs]
    args = (bt.hidden[0], int(bt.lengths[0]), [int(t) for t in bt.q_type[qs]], [tuple(s) for s in bt.q_span[qs]],
            blocks, bt.token_ids[0], bt.lexical.dense())
    good, _ = th.record(*args)
    th.option_ln = torch.nn.Identity()
    bad, _ = th.record(*args)
    assert max(np.abs(a - b).max() for a, b in zip(good, bad)) > 1e-3
