"""Record sharding of one batch over several GPUs, one process per GPU.

Records are independent in the head (no reduction crosses records), so a batch
splits by records with no exchange on the data path: every rank runs the head on
its own records and only the small per-option / per-question outputs travel back.
Shards are contiguous record ranges balanced by memory rows (the K/V projection,
proportional to rows, dominates the cost).  ``ShardedRunner`` drives it over a
torch.distributed process group: it picks the rank's records, runs them through a
per-rank compute function (the CUDA head on that rank's GPU, with its own copy of
the weights and the lexical table) and gathers the outputs once.
"""
from dataclasses import dataclass
from typing import Callable, Dict, List, Optional

import numpy as np


def shard_records(lengths, world: int) -> List[np.ndarray]:
    """Contiguous record ranges, one per rank, with nearly equal total rows.

    Every rank gets at least one record when there are enough records; ranks
    beyond the record count get an empty range.
    """
    lengths = np.asarray(lengths, np.int64)
    B = len(lengths)
    if world < 1:
        raise ValueError("world must be >= 1")
    cum = np.concatenate([[0], np.cumsum(lengths)])
    bounds = [0]
    for r in range(1, world):
        target = cum[-1] * r / world
        cut = int(np.searchsorted(cum, target, side="left"))
        # nearest record boundary to the target, kept monotone and leaving a record for
        # every later rank where possible
        if cut > 0 and abs(cum[cut - 1] - target) <= abs(cum[min(cut, B)] - target):
            cut -= 1
        lo = bounds[-1] + (1 if bounds[-1] < B else 0)
        hi = max(lo, B - (world - r))
        bounds.append(int(min(max(cut, lo), hi)))
    bounds.append(B)
    return [np.arange(bounds[r], bounds[r + 1]) for r in range(world)]


@dataclass
class SubBatch:
    """Schema tables of a record subset, re-indexed from zero."""
    records: np.ndarray
    lengths: np.ndarray
    q_rec: np.ndarray
    q_type: np.ndarray
    q_span: np.ndarray
    q_opt_off: np.ndarray
    o_span: np.ndarray
    q_index: np.ndarray   # original question indices
    o_index: np.ndarray   # original option indices


def sub_batch(records, lengths, q_rec, q_type, q_span, q_opt_off, o_span) -> SubBatch:
    records = np.asarray(records, np.int64)
    q_rec = np.asarray(q_rec)
    q_opt_off = np.asarray(q_opt_off)
    remap = {int(b): i for i, b in enumerate(records)}
    qs = np.nonzero(np.isin(q_rec, records))[0]
    blocks = [np.arange(q_opt_off[q], q_opt_off[q + 1]) for q in qs]
    o_idx = np.concatenate(blocks) if blocks else np.zeros(0, np.int64)
    off = np.concatenate([[0], np.cumsum([len(x) for x in blocks])]).astype(np.int32)
    return SubBatch(records=records, lengths=np.asarray(lengths)[records].astype(np.int32),
                    q_rec=np.array([remap[int(b)] for b in q_rec[qs]], np.int32),
                    q_type=np.asarray(q_type)[qs].astype(np.int32),
                    q_span=np.asarray(q_span)[qs].astype(np.int32).reshape(-1, 2), q_opt_off=off,
                    o_span=np.asarray(o_span)[o_idx].astype(np.int32).reshape(-1, 2), q_index=qs, o_index=o_idx)


def assemble(parts, Q: int, O: int):
    """Put per-rank outputs back in the batch's order.

    ``parts`` is a list of (SubBatch, {"logits", "probs": [O_r], "value", "conf",
    "argmax": [Q_r]}) pairs, one per rank.
    """
    out = {"logits": np.full(O, np.nan), "probs": np.full(O, np.nan), "value": np.full(Q, np.nan),
           "conf": np.full(Q, np.nan), "argmax": np.full(Q, -1, np.int64)}
    for sb, res in parts:
        for k in ("logits", "probs"):
            out[k][sb.o_index] = res[k]
        for k in ("value", "conf", "argmax"):
            out[k][sb.q_index] = res[k]
    return out


OUTPUT_KEYS = ("logits", "probs", "value", "conf", "argmax")


def empty_outputs() -> Dict[str, np.ndarray]:
    """Outputs of a rank that holds no record."""
    return {"logits": np.zeros(0, np.float32), "probs": np.zeros(0, np.float32), "value": np.zeros(0, np.float32),
            "conf": np.zeros(0, np.float32), "argmax": np.zeros(0, np.int32)}


class ShardedRunner:
    """Record-sharded forward pass over the ranks of a torch.distributed group.

    Every rank calls ``forward`` with the whole batch's schema tables (a few KB of
    host arrays, the same on every rank).  ``shard_records`` gives each rank a
    contiguous, row-balanced record range, ``sub_batch`` re-indexes it from zero and
    ``run_shard(sub)`` computes it on the rank's own device; it returns the
    ``OUTPUT_KEYS`` arrays of the sub-batch (per option: logits, probs; per question:
    value, conf, argmax).  The outputs are then gathered once (``all_gather_object``:
    a few KB per rank, after the shard's compute is finished) and every rank returns
    the whole batch's outputs in batch order.  Without an initialised process group
    the runner is a single rank that holds every record.
    """

    def __init__(self, run_shard: Callable[[SubBatch], Dict[str, np.ndarray]], group=None):
        self.run_shard = run_shard
        self.group = group

    def _dist(self):
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            return dist
        return None

    def world_rank(self):
        d = self._dist()
        if d is None:
            return 1, 0
        return d.get_world_size(self.group), d.get_rank(self.group)

    def shards(self, lengths) -> List[np.ndarray]:
        return shard_records(lengths, self.world_rank()[0])

    def local(self, lengths, q_rec, q_type, q_span, q_opt_off, o_span) -> SubBatch:
        """This rank's sub-batch."""
        world, rank = self.world_rank()
        return sub_batch(shard_records(lengths, world)[rank], lengths, q_rec, q_type, q_span, q_opt_off, o_span)

    def forward(self, lengths, q_rec, q_type, q_span, q_opt_off, o_span) -> Dict[str, np.ndarray]:
        tables = (lengths, q_rec, q_type, q_span, q_opt_off, o_span)
        world, rank = self.world_rank()
        shards = shard_records(lengths, world)
        mine = sub_batch(shards[rank], *tables)
        res = self.run_shard(mine) if len(mine.records) else empty_outputs()
        res = {k: np.asarray(res[k]) for k in OUTPUT_KEYS}
        if len(res["logits"]) != len(mine.o_index) or len(res["value"]) != len(mine.q_index):
            raise ValueError("run_shard returned outputs of the wrong size")
        if world == 1:
            gathered = [res]
        else:
            gathered = [None] * world
            self._dist().all_gather_object(gathered, res, group=self.group)
        parts = [(mine if r == rank else sub_batch(shards[r], *tables), gathered[r]) for r in range(world)]
        Q, O = len(q_type), int(np.asarray(q_opt_off)[-1])
        return assemble(parts, Q, O)
