"""The allocation-free span-sum entry point against the workspace one.

Callers that cannot allocate device memory (a fixed pool owned by another runtime,
a plug-in handed only its buffers) use clef_span_sums_noalloc, whose scratch is a
static device array inside the library.  It must give the same sums as
clef_span_sums, bit for bit, call after call: the array keeps the previous call's
contents, so two different batches run back to back here.  This file is collected
last so that a failure here never hides another test's result.
"""
import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library

SCRATCH_BYTES = 1 << 20


def _batch(seed, B_, H, vocab, lengths=(200, 900)):
    spec = synth.BatchSpec(name="na", B=B_, H=H, vocab=vocab, length_law="uniform", length_range=lengths,
                           questions=(1, 6), options=(2, 7), instr_len=(1, 40), option_len=(1, 20))
    bt = synth.make_batch(spec, seed=seed, with_hidden=False)
    rng = np.random.default_rng(seed)
    bt.hidden = synth.f32_to_bf16(rng.standard_normal((bt.B, bt.Lpad, bt.H)).astype(np.float32))
    table = synth.f32_to_bf16(rng.standard_normal((vocab, bt.H)).astype(np.float32))
    return bt, table


def _schema(bt):
    return B.Schema(bt.B, bt.Lpad, bt.H, bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)


def test_oversized_schema_is_rejected_before_any_launch():
    build_library()
    cfg = B.make_config(H=256, vocab=1000)
    nrec, per = 1000, 40  # 40 000 one-row questions with one option each: > 1 MiB of plan
    n, L = nrec * per, 2 * per + 1
    lengths = np.full(nrec, L, np.int32)
    t = np.arange(per) * 2
    q_span = np.tile(np.stack([t, t + 1], 1), (nrec, 1))
    q_rec = np.repeat(np.arange(nrec), per)
    sch = B.Schema(nrec, L, 256, lengths, q_rec, np.ones(n), q_span, np.arange(n + 1), q_span)
    assert B.clef_workspace_size(cfg, sch) > 0  # the schema itself is valid
    st = B.clef_span_sums_noalloc(cfg, sch, 1 << 20, 1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25, None)
    assert st == 2  # CLEF_ERR_WORKSPACE_TOO_SMALL, nothing launched


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    build_library()
    B.load()
    H, vocab = 256, 3000
    cfg = B.make_config(H=H, vocab=vocab)
    stream = torch.cuda.current_stream().cuda_stream
    for seed, nrec in ((21, 4), (22, 7)):  # a different batch each call
        bt, table = _batch(seed, nrec, H, vocab)
        sch = _schema(bt)
        hidden = torch.from_numpy(bt.hidden.view(np.int16)).cuda().view(torch.bfloat16)
        lex = torch.from_numpy(table.view(np.int16)).cuda().view(torch.bfloat16)
        ids = torch.from_numpy(bt.token_ids).cuda()
        outs = []
        for use_ws in (True, False):
            q = torch.full((bt.Q, H), float("nan"), dtype=torch.float32, device="cuda")
            o = torch.full((bt.O, H), float("nan"), dtype=torch.float32, device="cuda")
            x = torch.full((bt.O, H), float("nan"), dtype=torch.float32, device="cuda")
            if use_ws:
                nws = B.clef_workspace_size(cfg, sch)
                ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
                B.clef_span_sums(cfg, sch, hidden.data_ptr(), ids.data_ptr(), lex.data_ptr(), q.data_ptr(),
                                 o.data_ptr(), x.data_ptr(), ws.data_ptr(), nws, stream)
                torch.cuda.synchronize()
                assert B.clef_device_status(ws.data_ptr(), stream) == 0
            else:
                st = B.clef_span_sums_noalloc(cfg, sch, hidden.data_ptr(), ids.data_ptr(), lex.data_ptr(),
                                              q.data_ptr(), o.data_ptr(), x.data_ptr(), stream)
                assert st == 0, B.STATUS.get(st, st)
            outs.append([t.cpu().numpy() for t in (q, o, x)])
        for a, b in zip(*outs):
            assert np.isfinite(a).all()
            np.testing.assert_array_equal(a, b)


@pytest.mark.gpu
def test_noalloc_reports_out_of_range_token_id_then_recovers():
    """An option token id outside the vocabulary is skipped by the pooling kernel and
    returned directly as CLEF_ERR_DEVICE_BOUNDS (the call waits for its stream); the
    other sums still equal the workspace entry's, and the next clean call returns OK,
    because every call clears the status word in the shared array first."""
    build_library()
    B.load()
    H, vocab = 256, 3000
    cfg = B.make_config(H=H, vocab=vocab)
    stream = torch.cuda.current_stream().cuda_stream
    bt, table = _batch(23, 3, H, vocab)
    sch = _schema(bt)
    hidden = torch.from_numpy(bt.hidden.view(np.int16)).cuda().view(torch.bfloat16)
    lex = torch.from_numpy(table.view(np.int16)).cuda().view(torch.bfloat16)
    bad_ids = bt.token_ids.copy()
    bad_ids[bt.q_rec[0], bt.o_span[0, 0]] = vocab + 7
    outs = []
    for ids_np, use_ws in ((bad_ids, True), (bad_ids, False)):
        ids = torch.from_numpy(ids_np).cuda()
        q, o, x = (torch.zeros((n, H), dtype=torch.float32, device="cuda") for n in (bt.Q, bt.O, bt.O))
        if use_ws:
            nws = B.clef_workspace_size(cfg, sch)
            ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
            B.clef_span_sums(cfg, sch, hidden.data_ptr(), ids.data_ptr(), lex.data_ptr(), q.data_ptr(),
                             o.data_ptr(), x.data_ptr(), ws.data_ptr(), nws, stream)
            torch.cuda.synchronize()
            assert B.clef_device_status(ws.data_ptr(), stream) == 5  # CLEF_ERR_DEVICE_BOUNDS
        else:
            st = B.clef_span_sums_noalloc(cfg, sch, hidden.data_ptr(), ids.data_ptr(), lex.data_ptr(),
                                          q.data_ptr(), o.data_ptr(), x.data_ptr(), stream)
            assert st == 5, B.STATUS.get(st, st)
        outs.append([t.cpu().numpy() for t in (q, o, x)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    ids = torch.from_numpy(bt.token_ids).cuda()
    q, o, x = (torch.zeros((n, H), dtype=torch.float32, device="cuda") for n in (bt.Q, bt.O, bt.O))
    st = B.clef_span_sums_noalloc(cfg, sch, hidden.data_ptr(), ids.data_ptr(), lex.data_ptr(), q.data_ptr(),
                                  o.data_ptr(), x.data_ptr(), stream)
    assert st == 0, B.STATUS.get(st, st)
