"""PyTorch-side helper around the C ABI: device buffers and streams only.

``ClefHead`` uploads a weight set, runs ``clef_prepare_weights`` once, and calls
``clef_head_forward`` with torch-allocated device buffers on torch's current
stream.  All arithmetic of the head happens in libclef_head.so.
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding as B


def weight_order(H, D, heads, F, n_route, n_joint):
    """Names of the weight pointer table, in the order the C header documents."""
    names = ["mem_ln.weight", "mem_ln.bias", "query.ctx.weight", "query.lex.weight",
             "query.question.weight", "query.bias"]
    for l in range(n_route):
        names += [f"route.{l}.{k}" for k in (
            "attn_ln.weight", "attn_ln.bias", "q.weight", "q.bias", "k.weight", "k.bias", "v.weight", "v.bias",
            "o.weight", "o.bias", "ffn_ln.weight", "ffn_ln.bias", "ffn1.weight", "ffn1.bias", "ffn2.weight",
            "ffn2.bias")]
    names += ["option_ln.weight", "option_ln.bias", "field.pool.weight", "field.pool.bias",
              "field.question.weight", "field.summary.weight", "field.global.weight", "field.bias",
              "field.type_embedding"]
    for i in range(n_joint):
        names += [f"joint.{i}.{k}" for k in (
            "attn_ln.weight", "attn_ln.bias", "qkv.weight", "qkv.bias", "o.weight", "o.bias", "ffn_ln.weight",
            "ffn_ln.bias", "ffn1.weight", "ffn1.bias", "ffn2.weight", "ffn2.bias")]
    names += ["field_ln.weight", "field_ln.bias", "scorer.gate", "scorer.joint_scale", "scorer.mlp1.weight",
              "scorer.mlp1.bias", "scorer.mlp2.weight", "scorer.mlp2.bias"]
    return names


def to_device_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> a torch bfloat16 tensor on ``device``."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def stream_handle(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


@dataclass
class Outputs:
    logits: torch.Tensor
    probs: torch.Tensor
    q_value: torch.Tensor
    q_conf: torch.Tensor
    q_argmax: torch.Tensor


class ClefHead:
    def __init__(self, weights: dict, H=4096, D=1024, heads=16, F=4096, n_route=2, n_joint=4, vocab=248320,
                 device="cuda"):
        self.cfg = B.make_config(H, D, heads, F, n_route, n_joint, vocab)
        self.H, self.D, self.heads, self.F, self.vocab = H, D, heads, F, vocab
        self.device = device
        names = weight_order(H, D, heads, F, n_route, n_joint)
        if B.clef_weight_count(self.cfg) != len(names):
            raise RuntimeError("weight table size mismatch with the C library")
        self.weights = [to_device_bf16(weights[n], device) for n in names]
        self.weight_ptrs = [w.data_ptr() for w in self.weights]
        nbytes = B.clef_prepared_size(self.cfg)
        self.prepared = torch.empty(nbytes, dtype=torch.uint8, device=device)
        B.clef_prepare_weights(self.cfg, self.weight_ptrs, self.prepared.data_ptr(), nbytes, stream_handle())
        self._ws = None

    def workspace(self, schema: B.Schema) -> torch.Tensor:
        n = B.clef_workspace_size(self.cfg, schema)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        return self._ws

    def alloc_outputs(self, schema: B.Schema) -> Outputs:
        dev = self.device
        return Outputs(torch.empty(schema.O, dtype=torch.float32, device=dev),
                       torch.empty(schema.O, dtype=torch.float32, device=dev),
                       torch.empty(schema.Q, dtype=torch.float32, device=dev),
                       torch.empty(schema.Q, dtype=torch.float32, device=dev),
                       torch.empty(schema.Q, dtype=torch.int32, device=dev))

    def forward(self, schema: B.Schema, hidden: torch.Tensor, token_ids: torch.Tensor, lexical: torch.Tensor,
                out: Optional[Outputs] = None, debug=None, stream=None, check=True) -> Outputs:
        ws = self.workspace(schema)
        out = out if out is not None else self.alloc_outputs(schema)
        B.clef_head_forward(self.cfg, self.weight_ptrs, self.prepared.data_ptr(), schema, hidden.data_ptr(),
                            token_ids.data_ptr(), lexical.data_ptr(), out.logits.data_ptr(), out.probs.data_ptr(),
                            out.q_value.data_ptr(), out.q_conf.data_ptr(), out.q_argmax.data_ptr(), ws.data_ptr(),
                            ws.numel(), debug=debug, stream=stream_handle(stream), check=check)
        return out

    def stream_begin(self, schema: B.Schema, stream=None):
        ws = self.workspace(schema)
        B.clef_stream_begin(self.cfg, schema, ws.data_ptr(), ws.numel(), stream_handle(stream))

    def stream_rows(self, schema: B.Schema, hidden: torch.Tensor, record: int, row0: int, n_rows: int, stream=None):
        """Statistics and K/V of rows [row0, row0 + n_rows) of ``record``; ``hidden`` is
        bf16 or fp16 (fp16 rows are rounded to bf16 where the head reads them)."""
        ws = self._ws
        fn = B.clef_stream_rows_f16 if hidden.dtype == torch.float16 else B.clef_stream_rows
        fn(self.cfg, self.prepared.data_ptr(), schema, hidden.data_ptr(), record, row0, n_rows, ws.data_ptr(),
           ws.numel(), stream_handle(stream))

    def stream_finish(self, schema: B.Schema, hidden: torch.Tensor, token_ids: torch.Tensor, lexical: torch.Tensor,
                      out: Optional[Outputs] = None, debug=None, stream=None) -> Outputs:
        ws = self._ws
        out = out if out is not None else self.alloc_outputs(schema)
        fn = B.clef_stream_finish_f16 if hidden.dtype == torch.float16 else B.clef_stream_finish
        fn(self.cfg, self.weight_ptrs, self.prepared.data_ptr(), schema, hidden.data_ptr(), token_ids.data_ptr(),
           lexical.data_ptr(), out.logits.data_ptr(), out.probs.data_ptr(), out.q_value.data_ptr(),
           out.q_conf.data_ptr(), out.q_argmax.data_ptr(), ws.data_ptr(), ws.numel(), debug=debug,
           stream=stream_handle(stream))
        return out

    def device_status(self, stream=None) -> int:
        return B.clef_device_status(self._ws.data_ptr(), stream_handle(stream))

    def shard_fn(self, hidden, token_ids, lexical: torch.Tensor, stream=None):
        """The per-rank compute of ``sharding.ShardedRunner``: the shard's records
        through this GPU's head.

        ``hidden`` [B, Lpad, H] bf16 and ``token_ids`` [B, Lpad] int32 hold the whole
        batch, as torch tensors on any device or as numpy arrays on the host (bf16 as
        uint16 bit patterns); only the shard's records, up to the shard's longest
        length, are copied to this GPU.  ``lexical`` is this GPU's copy of the table.
        Raises if the device reports an error."""
        def run(sb) -> dict:
            Lp = int(sb.lengths.max())
            if isinstance(hidden, np.ndarray):
                h = to_device_bf16(hidden[sb.records, :Lp], self.device)
            else:
                h = hidden[torch.as_tensor(sb.records, device=hidden.device), :Lp].to(self.device).contiguous()
            if isinstance(token_ids, np.ndarray):
                ids = torch.from_numpy(np.ascontiguousarray(token_ids[sb.records, :Lp], np.int32)).to(self.device)
            else:
                ids = token_ids[torch.as_tensor(sb.records, device=token_ids.device), :Lp].to(self.device).contiguous()
            schema = B.Schema(len(sb.records), Lp, self.H, sb.lengths, sb.q_rec, sb.q_type, sb.q_span, sb.q_opt_off,
                              sb.o_span)
            out = self.forward(schema, h, ids, lexical, stream=stream)
            st = self.device_status(stream)  # waits for the stream
            if st != 0:
                raise B.ClefError(st, "device status after a shard")
            return {"logits": out.logits.cpu().numpy(), "probs": out.probs.cpu().numpy(),
                    "value": out.q_value.cpu().numpy(), "conf": out.q_conf.cpu().numpy(),
                    "argmax": out.q_argmax.cpu().numpy()}
        return run
