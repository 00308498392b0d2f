"""Random-init JointSchemaHead weights from a seed, stored as bf16.

The head's weight file is bf16 and not quantised (clef-4bit walkthrough, section 3
and FAQ "why the decision head stays bf16"); trained weights are not available, so
every tensor is drawn from a seed:  Linear W ~ N(0, 1/fan_in), bias ~ N(0, 0.02),
LayerNorm gamma = 1 + N(0, 0.05), beta ~ N(0, 0.02), type embedding ~ N(0, 0.02),
gate scalar ~ N(0, 1), joint_scale ~ U(2, 8).

Tensors follow the torch Linear convention [out_features, in_features].  The order
of ``weight_names`` is the order of the weight pointer table of the C library.
"""
from dataclasses import dataclass

import numpy as np

from .bf16 import f32_to_bf16


@dataclass(frozen=True)
class HeadShape:
    """Head hyper-parameters (joint_head_config.json fields as the pages list them)."""
    H: int = 4096        # hidden_size of the backbone
    D: int = 1024        # width
    heads: int = 16
    F: int = 4096        # feedforward
    n_route: int = 2     # routing_layers
    n_joint: int = 4     # layers
    vocab: int = 248320

    @property
    def dh(self):
        return self.D // self.heads


def _route_block(s: HeadShape, l: int):
    p, H, D, F = f"route.{l}.", s.H, s.D, s.F
    return [
        (p + "attn_ln.weight", (D,), "ln_w"), (p + "attn_ln.bias", (D,), "ln_b"),
        (p + "q.weight", (D, D), "lin"), (p + "q.bias", (D,), "bias"),
        (p + "k.weight", (D, H), "lin"), (p + "k.bias", (D,), "bias"),
        (p + "v.weight", (D, H), "lin"), (p + "v.bias", (D,), "bias"),
        (p + "o.weight", (D, D), "lin"), (p + "o.bias", (D,), "bias"),
        (p + "ffn_ln.weight", (D,), "ln_w"), (p + "ffn_ln.bias", (D,), "ln_b"),
        (p + "ffn1.weight", (F, D), "lin"), (p + "ffn1.bias", (F,), "bias"),
        (p + "ffn2.weight", (D, F), "lin"), (p + "ffn2.bias", (D,), "bias"),
    ]


def _joint_block(s: HeadShape, i: int):
    p, D, F = f"joint.{i}.", s.D, s.F
    return [
        (p + "attn_ln.weight", (D,), "ln_w"), (p + "attn_ln.bias", (D,), "ln_b"),
        (p + "qkv.weight", (3 * D, D), "lin"), (p + "qkv.bias", (3 * D,), "bias"),
        (p + "o.weight", (D, D), "lin"), (p + "o.bias", (D,), "bias"),
        (p + "ffn_ln.weight", (D,), "ln_w"), (p + "ffn_ln.bias", (D,), "ln_b"),
        (p + "ffn1.weight", (F, D), "lin"), (p + "ffn1.bias", (F,), "bias"),
        (p + "ffn2.weight", (D, F), "lin"), (p + "ffn2.bias", (D,), "bias"),
    ]


def weight_table(s: HeadShape):
    """[(name, shape, init kind)] in pointer-table order."""
    H, D = s.H, s.D
    t = [
        ("mem_ln.weight", (H,), "ln_w"), ("mem_ln.bias", (H,), "ln_b"),
        ("query.ctx.weight", (D, H), "lin"), ("query.lex.weight", (D, H), "lin"),
        ("query.question.weight", (D, H), "lin"), ("query.bias", (D,), "bias"),
    ]
    for l in range(s.n_route):
        t += _route_block(s, l)
    t += [
        ("option_ln.weight", (D,), "ln_w"), ("option_ln.bias", (D,), "ln_b"),
        ("field.pool.weight", (1, D), "lin"), ("field.pool.bias", (1,), "bias"),
        ("field.question.weight", (D, H), "lin"), ("field.summary.weight", (D, D), "lin"),
        ("field.global.weight", (D, H), "lin"), ("field.bias", (D,), "bias"),
        ("field.type_embedding", (3, D), "emb"),
    ]
    for i in range(s.n_joint):
        t += _joint_block(s, i)
    t += [
        ("field_ln.weight", (D,), "ln_w"), ("field_ln.bias", (D,), "ln_b"),
        ("scorer.gate", (1,), "gate"), ("scorer.joint_scale", (1,), "scale"),
        ("scorer.mlp1.weight", (D, 4 * D), "lin"), ("scorer.mlp1.bias", (D,), "bias"),
        ("scorer.mlp2.weight", (1, D), "lin"), ("scorer.mlp2.bias", (1,), "bias"),
    ]
    return t


def weight_names(s: HeadShape):
    return [n for (n, _, _) in weight_table(s)]


def make_weights(s: HeadShape, seed: int = 0):
    """{name: uint16 bf16 array}, every tensor seeded by (seed, its table index)."""
    out = {}
    for idx, (name, shape, kind) in enumerate(weight_table(s)):
        g = np.random.default_rng([seed, 101, idx])
        if kind == "lin":
            x = g.standard_normal(shape, dtype=np.float32) * np.float32(1.0 / np.sqrt(shape[1]))
        elif kind in ("bias", "ln_b", "emb"):
            x = g.standard_normal(shape, dtype=np.float32) * np.float32(0.02)
        elif kind == "ln_w":
            x = 1.0 + g.standard_normal(shape, dtype=np.float32) * np.float32(0.05)
        elif kind == "gate":
            x = g.standard_normal(shape, dtype=np.float32)
        elif kind == "scale":
            x = g.uniform(2.0, 8.0, size=shape).astype(np.float32)
        else:
            raise ValueError(kind)
        out[name] = f32_to_bf16(x)
    return out
