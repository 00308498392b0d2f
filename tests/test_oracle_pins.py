"""Pins of the fp64 oracle to things other than itself (CPU only).

Every check below is an independent statement of what the pages and the
mathematics fix: a library routine (torch.nn modules, scipy), a brute-force loop on
tiny inputs, a closed form of a special case, or an invariant of the method.  Each
is chosen so that a plausible slip in the oracle (a dropped term, a swapped
operand, a wrong index or axis) fails at least one of them.
"""
import dataclasses

import numpy as np
import pytest
import scipy.spatial.distance as ssd
import scipy.special as ssp
import torch

import oracle
import synth
from oracle.clef_head import HeadParams, linear
from synth import BatchSpec, HeadShape

F64 = dict(dtype=torch.float64)

TINY = HeadShape(H=48, D=32, heads=4, F=64, vocab=500)


def tiny_spec(**kw):
    base = dict(name="tiny", B=3, H=TINY.H, vocab=TINY.vocab, length_law="uniform",
                length_range=(150, 260), questions=(2, 4), options=(2, 5), instr_len=(3, 9),
                option_len=(2, 6))
    base.update(kw)
    return BatchSpec(**base)


def params(seed=0, shape=TINY):
    return HeadParams.from_bf16(synth.make_weights(shape, seed), shape.heads, shape.n_route, shape.n_joint)


def run(p, bt, shape=TINY, **kw):
    return oracle.head_forward(p, shape.heads, shape.n_route, shape.n_joint, bt.hidden, bt.lengths,
                               bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span,
                               bt.token_ids, bt.lexical, **kw)


def T(a):
    return torch.from_numpy(np.asarray(a, np.float64))


# ----------------------------------------------------------------- primitives

def test_layer_norm_matches_torch():
    rng = np.random.default_rng(0)
    x, w, b = rng.normal(size=(7, 33)) * 3 + 1, rng.normal(size=33), rng.normal(size=33)
    ref = torch.nn.functional.layer_norm(T(x), (33,), T(w), T(b), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layer_norm(x, w, b), ref, rtol=1e-12, atol=1e-12)


def test_gelu_is_exact_erf_form():
    x = np.linspace(-6, 6, 101)
    ref = torch.nn.functional.gelu(T(x), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu(x), ref, rtol=1e-13, atol=1e-15)


def test_cosine_matches_scipy():
    rng = np.random.default_rng(1)
    a, b = rng.normal(size=(5, 9)), rng.normal(size=(5, 9))
    ref = np.array([1.0 - ssd.cosine(a[i], b[i]) for i in range(5)])
    np.testing.assert_allclose(oracle.cosine(a, b), ref, rtol=1e-12, atol=1e-14)
    # a zero vector has cosine 0 rather than NaN (eps clamp)
    assert oracle.cosine(np.zeros((1, 4)), np.ones((1, 4)))[0] == 0.0


# -------------------------------------------------------------------- pooling

def _dense_lexical(bt):
    return synth.bf16_to_f32(bt.lexical.dense()).astype(np.float64)


def test_pooling_bruteforce_loops():
    bt = synth.make_batch(tiny_spec(B=2), seed=4)
    p = params()
    lex = _dense_lexical(bt)
    for b in range(bt.B):
        L = int(bt.lengths[b])
        h = synth.bf16_to_f32(bt.hidden[b]).astype(np.float64)
        ln_rows = torch.nn.functional.layer_norm(T(h[:L]), (bt.H,), T(p["mem_ln.weight"]),
                                                 T(p["mem_ln.bias"]), eps=1e-5).numpy()
        mem = oracle.memory_rows(bt.hidden[b], L, p)
        np.testing.assert_allclose(mem, ln_rows, rtol=1e-12, atol=1e-12)
        qs = np.nonzero(bt.q_rec == b)[0]
        osel = range(bt.q_opt_off[qs[0]], bt.q_opt_off[qs[-1] + 1])
        o_sp = bt.o_span[list(osel)]
        o_ids = [bt.token_ids[b][s:e] for (s, e) in o_sp]
        u, c, x, g = oracle.pool_record(mem, L, bt.q_span[qs], o_sp, o_ids, bt.lexical)
        for k, q in enumerate(qs):
            s, e = bt.q_span[q]
            acc = [0.0] * bt.H
            for t in range(s, e):
                for col in range(bt.H):
                    acc[col] += ln_rows[t, col]
            np.testing.assert_allclose(u[k], np.array(acc) / (e - s), rtol=1e-12, atol=1e-12)
        for j, (s, e) in enumerate(o_sp):
            accc, accx = [0.0] * bt.H, [0.0] * bt.H
            for t in range(s, e):
                tok = int(bt.token_ids[b, t])
                for col in range(bt.H):
                    accc[col] += ln_rows[t, col]
                    accx[col] += lex[tok, col]
            np.testing.assert_allclose(c[j], np.array(accc) / (e - s), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(x[j], np.array(accx) / (e - s), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g, ln_rows[L - 1], rtol=1e-12, atol=1e-12)


def test_single_row_spans_are_rows():
    bt = synth.make_batch(tiny_spec(B=1), seed=5)
    p = params()
    L = int(bt.lengths[0])
    mem = oracle.memory_rows(bt.hidden[0], L, p)
    spans = np.array([[10, 11], [L - 1, L]])
    ids = [bt.token_ids[0][s:e] for (s, e) in spans]
    u, c, x, g = oracle.pool_record(mem, L, spans, spans, ids, bt.lexical)
    np.testing.assert_array_equal(u[0], mem[10])
    np.testing.assert_array_equal(c[1], g)
    np.testing.assert_array_equal(x[0], synth.bf16_to_f32(bt.lexical.row(bt.token_ids[0, 10])))


def test_raw_span_sums_integer_bruteforce():
    rng = np.random.default_rng(6)
    hid = synth.f32_to_bf16(rng.integers(-8, 9, size=(40, 16)).astype(np.float32))
    table = synth.f32_to_bf16(rng.integers(-4, 5, size=(30, 16)).astype(np.float32))
    ids = rng.integers(0, 30, size=40)
    q_span, o_span = np.array([[0, 5], [7, 8]]), np.array([[9, 12], [12, 20], [39, 40]])
    o_ids = [ids[s:e] for (s, e) in o_span]
    sq, so, sx = oracle.span_raw_sums(hid, q_span, o_span, o_ids, table)
    hf, tf = synth.bf16_to_f32(hid), synth.bf16_to_f32(table)
    for k, (s, e) in enumerate(q_span):
        assert all(sq[k][col] == sum(int(hf[t, col]) for t in range(s, e)) for col in range(16))
    for k, (s, e) in enumerate(o_span):
        assert all(so[k][col] == sum(int(hf[t, col]) for t in range(s, e)) for col in range(16))
        assert all(sx[k][col] == sum(int(tf[ids[t], col]) for t in range(s, e)) for col in range(16))


# ------------------------------------------------------------- attention pins

def _mha_ref(qx, mem, Wq, bq, Wk, bk, Wv, bv, Wo, bo, heads):
    D, H = Wq.shape[0], Wk.shape[1]
    mha = torch.nn.MultiheadAttention(D, heads, bias=True, kdim=H, vdim=H, batch_first=True, **F64)
    with torch.no_grad():
        mha.q_proj_weight.copy_(T(Wq))
        mha.k_proj_weight.copy_(T(Wk))
        mha.v_proj_weight.copy_(T(Wv))
        mha.in_proj_bias.copy_(T(np.concatenate([bq, bk, bv])))
        mha.out_proj.weight.copy_(T(Wo))
        mha.out_proj.bias.copy_(T(bo))
        y, _ = mha(T(qx)[None], T(mem)[None], T(mem)[None], need_weights=False)
    return y[0].numpy()


def test_cross_attention_matches_torch_mha():
    rng = np.random.default_rng(7)
    D, H, heads, n, L = 32, 48, 4, 5, 37
    Wq, Wk, Wv, Wo = (rng.normal(size=s) * 0.3 for s in [(D, D), (D, H), (D, H), (D, D)])
    bq, bk, bv, bo = (rng.normal(size=D) * 0.1 for _ in range(4))
    qx, mem = rng.normal(size=(n, D)), rng.normal(size=(L, H))
    got = linear(oracle.cross_attention(qx, mem, Wq, bq, Wk, bk, Wv, bv, heads), Wo, bo)
    ref = _mha_ref(qx, mem, Wq, bq, Wk, bk, Wv, bv, Wo, bo, heads)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-11)


def test_cross_attention_uniform_when_keys_constant():
    rng = np.random.default_rng(8)
    D, H, heads, L = 32, 48, 4, 23
    Wq, Wv = rng.normal(size=(D, D)), rng.normal(size=(D, H))
    bq, bv, bk = rng.normal(size=D), rng.normal(size=D), rng.normal(size=D)
    qx, mem = rng.normal(size=(3, D)), rng.normal(size=(L, H))
    got = oracle.cross_attention(qx, mem, Wq, bq, np.zeros((D, H)), bk, Wv, bv, heads)
    closed = Wv @ mem.mean(axis=0) + bv  # every key alike -> uniform weights
    np.testing.assert_allclose(got, np.broadcast_to(closed, got.shape), rtol=1e-11, atol=1e-11)
    one = oracle.cross_attention(qx, mem[:1], Wq, bq, rng.normal(size=(D, H)), bk, Wv, bv, heads)
    np.testing.assert_allclose(one, np.broadcast_to(Wv @ mem[0] + bv, one.shape), rtol=1e-11, atol=1e-11)


def test_routing_layer_matches_torch_modules():
    p = params(seed=2)
    rng = np.random.default_rng(9)
    o, mem = rng.normal(size=(6, TINY.D)), rng.normal(size=(41, TINY.H))
    got = oracle.routing_layer(o, mem, 1, p)
    q = "route.1."
    D = TINY.D
    ln1 = torch.nn.LayerNorm(D, eps=1e-5, **F64)
    ln2 = torch.nn.LayerNorm(D, eps=1e-5, **F64)
    ffn = torch.nn.Sequential(torch.nn.Linear(D, TINY.F, **F64), torch.nn.GELU(), torch.nn.Linear(TINY.F, D, **F64))
    with torch.no_grad():
        ln1.weight.copy_(T(p[q + "attn_ln.weight"]))
        ln1.bias.copy_(T(p[q + "attn_ln.bias"]))
        ln2.weight.copy_(T(p[q + "ffn_ln.weight"]))
        ln2.bias.copy_(T(p[q + "ffn_ln.bias"]))
        ffn[0].weight.copy_(T(p[q + "ffn1.weight"]))
        ffn[0].bias.copy_(T(p[q + "ffn1.bias"]))
        ffn[2].weight.copy_(T(p[q + "ffn2.weight"]))
        ffn[2].bias.copy_(T(p[q + "ffn2.bias"]))
        a = ln1(T(o)).numpy()
    x = o + _mha_ref(a, mem, p[q + "q.weight"], p[q + "q.bias"], p[q + "k.weight"], p[q + "k.bias"],
                     p[q + "v.weight"], p[q + "v.bias"], p[q + "o.weight"], p[q + "o.bias"], TINY.heads)
    with torch.no_grad():
        ref = (T(x) + ffn(ln2(T(x)))).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("n", [1, 5])
def test_joint_layer_matches_torch_encoder_layer(n):
    p = params(seed=3)
    q = "joint.2."
    D = TINY.D
    layer = torch.nn.TransformerEncoderLayer(D, TINY.heads, dim_feedforward=TINY.F, dropout=0.0,
                                             activation="gelu", layer_norm_eps=1e-5,
                                             batch_first=True, norm_first=True, **F64)
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(T(p[q + "qkv.weight"]))
        layer.self_attn.in_proj_bias.copy_(T(p[q + "qkv.bias"]))
        layer.self_attn.out_proj.weight.copy_(T(p[q + "o.weight"]))
        layer.self_attn.out_proj.bias.copy_(T(p[q + "o.bias"]))
        layer.norm1.weight.copy_(T(p[q + "attn_ln.weight"]))
        layer.norm1.bias.copy_(T(p[q + "attn_ln.bias"]))
        layer.norm2.weight.copy_(T(p[q + "ffn_ln.weight"]))
        layer.norm2.bias.copy_(T(p[q + "ffn_ln.bias"]))
        layer.linear1.weight.copy_(T(p[q + "ffn1.weight"]))
        layer.linear1.bias.copy_(T(p[q + "ffn1.bias"]))
        layer.linear2.weight.copy_(T(p[q + "ffn2.weight"]))
        layer.linear2.bias.copy_(T(p[q + "ffn2.bias"]))
    layer.eval()
    f = np.random.default_rng(10).normal(size=(n, D))
    with torch.no_grad():
        ref = layer(T(f)[None])[0].numpy()
    np.testing.assert_allclose(oracle.joint_layer(f, 2, p), ref, rtol=1e-10, atol=1e-10)


# ------------------------------------------------------- fields and scoring

def test_field_aggregate_uniform_pool_and_terms():
    p = params(seed=4)
    rng = np.random.default_rng(11)
    t = dict(p.t)
    t["field.pool.weight"] = np.zeros_like(t["field.pool.weight"])  # alpha uniform
    pz = HeadParams(t, p.heads, p.n_route, p.n_joint)
    u, oh, g = rng.normal(size=TINY.H), rng.normal(size=(4, TINY.D)), rng.normal(size=TINY.H)
    got = oracle.field_aggregate(u, oh, g, 2, pz)
    lin = torch.nn.Linear(TINY.H, TINY.D, bias=False, **F64)
    with torch.no_grad():
        lin.weight.copy_(T(p["field.question.weight"]))
        a = lin(T(u)).numpy()
        lin.weight.copy_(T(p["field.global.weight"]))
        c = lin(T(g)).numpy()
    b = p["field.summary.weight"] @ oh.mean(axis=0)
    ref = a + b + c + p["field.bias"] + p["field.type_embedding"][2]
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)
    # the learned pooling weights follow a softmax of w_a . o + b_a
    w = np.random.default_rng(12).normal(size=(1, TINY.D))
    t["field.pool.weight"] = w
    pw = HeadParams(t, p.heads, p.n_route, p.n_joint)
    alpha = ssp.softmax(oh @ w[0] + p["field.pool.bias"][0])
    ref2 = ref - b + p["field.summary.weight"] @ (alpha @ oh)
    np.testing.assert_allclose(oracle.field_aggregate(u, oh, g, 2, pw), ref2, rtol=1e-11, atol=1e-11)


def _scorer_params(p, gate, scale):
    t = dict(p.t)
    t["scorer.gate"], t["scorer.joint_scale"] = np.array([gate]), np.array([scale])
    return HeadParams(t, p.heads, p.n_route, p.n_joint)


def test_scorer_gate_closed_gives_prior_only():
    p = _scorer_params(params(seed=5), -800.0, 5.0)
    rng = np.random.default_rng(13)
    x, u, g = rng.normal(size=(3, TINY.H)), rng.normal(size=TINY.H), rng.normal(size=TINY.H)
    f, oh = rng.normal(size=TINY.D), rng.normal(size=(3, TINY.D))
    got = oracle.scorer_logits(x, u, g, f, oh, p)
    ref = np.array([1.0 - ssd.cosine(x[j], u + g) for j in range(3)])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_scorer_open_gate_matches_torch_terms():
    scale = 3.25
    p = _scorer_params(params(seed=6), 800.0, scale)  # sigmoid(800) == 1
    rng = np.random.default_rng(14)
    x, u, g = rng.normal(size=(4, TINY.H)), rng.normal(size=TINY.H), rng.normal(size=TINY.H)
    f, oh = rng.normal(size=TINY.D), rng.normal(size=(4, TINY.D))
    D = TINY.D
    mlp = torch.nn.Sequential(torch.nn.Linear(4 * D, D, **F64), torch.nn.GELU(), torch.nn.Linear(D, 1, **F64))
    with torch.no_grad():
        mlp[0].weight.copy_(T(p["scorer.mlp1.weight"]))
        mlp[0].bias.copy_(T(p["scorer.mlp1.bias"]))
        mlp[2].weight.copy_(T(p["scorer.mlp2.weight"]))
        mlp[2].bias.copy_(T(p["scorer.mlp2.bias"]))
        ft = T(f)[None].expand(4, D)
        z = torch.cat([ft, T(oh), ft * T(oh), (ft - T(oh)).abs()], dim=1)
        m = mlp(z)[:, 0].numpy()
        jc = torch.nn.functional.cosine_similarity(ft, T(oh), dim=1).numpy()
    prior = np.array([1.0 - ssd.cosine(x[j], u + g) for j in range(4)])
    ref = prior + scale * jc + m
    np.testing.assert_allclose(oracle.scorer_logits(x, u, g, f, oh, p), ref, rtol=1e-11, atol=1e-11)


def test_softmax_and_answers():
    l2 = np.array([0.7, -1.2])
    p2 = oracle.question_softmax(l2)
    assert abs(p2[0] - ssp.expit(l2[0] - l2[1])) < 1e-15
    assert oracle.question_softmax(np.array([3.0]))[0] == 1.0
    z = np.random.default_rng(15).normal(size=7) * 4
    pz = oracle.question_softmax(z)
    np.testing.assert_allclose(pz, ssp.softmax(z), rtol=1e-14)
    assert abs(pz.sum() - 1) < 1e-14
    v, c, k = oracle.answers(0, p2)
    assert v == p2[0] and k == 0 and c == max(p2)
    v, c, k = oracle.answers(2, pz)
    assert 0 <= v <= 6 and abs(v - sum(i * pz[i] for i in range(7))) < 1e-13 and k == int(np.argmax(pz))
    v, c, k = oracle.answers(1, np.array([0.25, 0.375, 0.375]))
    assert k == 1 and v == c == 0.375  # first maximum wins ties


# ------------------------------------------------------------ whole-head laws

def test_padding_invariance():
    p = params(seed=7)
    a = synth.make_batch(tiny_spec(), seed=21)
    b = synth.make_batch(tiny_spec(), seed=21, lpad=int(a.Lpad) + 77)
    assert b.Lpad > a.Lpad
    np.testing.assert_array_equal(b.hidden[:, :a.Lpad][np.arange(a.Lpad)[None, :] < a.lengths[:, None]],
                                  a.hidden[np.arange(a.Lpad)[None, :] < a.lengths[:, None]])
    # pad rows differ, real rows equal
    ra, rb = run(p, a), run(p, b)
    np.testing.assert_array_equal(ra["logits"], rb["logits"])
    np.testing.assert_array_equal(ra["probs"], rb["probs"])


def test_batch_invariance_record_alone():
    p = params(seed=8)
    bt = synth.make_batch(tiny_spec(B=3), seed=22)
    full = run(p, bt)
    b = 1
    qs = np.nonzero(bt.q_rec == b)[0]
    lo, hi = bt.q_opt_off[qs[0]], bt.q_opt_off[qs[-1] + 1]
    alone = oracle.head_forward(p, TINY.heads, TINY.n_route, TINY.n_joint, bt.hidden[b:b + 1],
                                bt.lengths[b:b + 1], np.zeros(len(qs), np.int32), bt.q_type[qs],
                                bt.q_span[qs], bt.q_opt_off[qs[0]:qs[-1] + 2] - lo,
                                bt.o_span[lo:hi], bt.token_ids[b:b + 1], bt.lexical)
    np.testing.assert_array_equal(alone["logits"], full["logits"][lo:hi])


def _permuted(bt, b, order):
    """Reorder record b's questions (with their option blocks) by ``order``."""
    qs = np.nonzero(bt.q_rec == b)[0]
    new_q = np.concatenate([np.nonzero(bt.q_rec < b)[0], qs[order], np.nonzero(bt.q_rec > b)[0]])
    opt_blocks = [np.arange(bt.q_opt_off[q], bt.q_opt_off[q + 1]) for q in new_q]
    new_o = np.concatenate(opt_blocks)
    off = np.concatenate([[0], np.cumsum([len(x) for x in opt_blocks])]).astype(np.int32)
    nb = dataclasses.replace(bt, q_rec=bt.q_rec[new_q], q_type=bt.q_type[new_q],
                             q_span=bt.q_span[new_q], q_opt_off=off, o_span=bt.o_span[new_o])
    return nb, new_q, new_o


def test_question_permutation_equivariance():
    p = params(seed=9)
    bt = synth.make_batch(tiny_spec(B=2, questions=(4, 4)), seed=23)
    full = run(p, bt)
    nq = int((bt.q_rec == 0).sum())
    nb, new_q, new_o = _permuted(bt, 0, np.random.default_rng(0).permutation(nq))
    perm = run(p, nb)
    np.testing.assert_allclose(perm["logits"], full["logits"][new_o], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(perm["value"], full["value"][new_q], rtol=1e-11, atol=1e-12)


def test_option_permutation_equivariance_within_question():
    p = params(seed=10)
    spec = tiny_spec(B=1, fixed_types=[(1, 4), (2, 3)])
    bt = synth.make_batch(spec, seed=24)
    full = run(p, bt)
    o_perm = np.array([2, 0, 3, 1, 4, 5, 6])
    nb = dataclasses.replace(bt, o_span=bt.o_span[o_perm])
    perm = run(p, nb)
    np.testing.assert_allclose(perm["logits"], full["logits"][o_perm], rtol=1e-11, atol=1e-12)


def test_joint_layers_couple_questions():
    """Fields see each other: changing one question's instruction span moves another's logits."""
    p = params(seed=11)
    bt = synth.make_batch(tiny_spec(B=1, questions=(3, 3), length_range=(600, 700)), seed=25)
    assert bt.Q == 3
    base = run(p, bt)
    q_span = bt.q_span.copy()
    q_span[2] = q_span[2] + np.array([0, -1])
    moved = run(p, dataclasses.replace(bt, q_span=q_span))
    lo, hi = bt.q_opt_off[0], bt.q_opt_off[1]
    assert np.abs(moved["logits"][lo:hi] - base["logits"][lo:hi]).max() > 1e-9
