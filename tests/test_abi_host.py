"""The C ABI on the host (no GPU): symbols, weight table, and validation errors.

Every call here fails validation (or only computes sizes) before the library
touches CUDA, so nothing is launched and no GPU is needed.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library
from structured_decision_model_gb300.head import weight_order

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_library()
    return B.load()


def header_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"CLEF_API\s+[\w\s\*]+?\b(clef_\w+)\s*\(", text)
    return names


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(B.EXPORTED)


def test_status_strings(lib):
    assert B.clef_status_string(0) == "ok"
    assert "workspace" in B.clef_status_string(2)


def test_weight_table_order_matches_generators():
    s = synth.HeadShape()
    assert weight_order(s.H, s.D, s.heads, s.F, s.n_route, s.n_joint) == synth.weight_names(s)
    cfg = B.make_config()
    assert B.clef_weight_count(cfg) == len(synth.weight_names(s)) == 6 + 16 * 2 + 9 + 12 * 4 + 8


@pytest.mark.parametrize("bad", [dict(hidden=100), dict(width=1000), dict(heads=8), dict(ffn=100),
                                 dict(n_route=0), dict(n_route=5), dict(n_joint=9), dict(vocab=0)])
def test_unsupported_configs(bad):
    kw = dict(H=4096, D=1024, heads=16, F=4096, n_route=2, n_joint=4, vocab=248320)
    ren = {"hidden": "H", "width": "D", "ffn": "F"}
    for k, v in bad.items():
        kw[ren.get(k, k)] = v
    cfg = B.make_config(**kw)
    with pytest.raises(B.ClefError) as e:
        B.clef_prepared_size(cfg)
    assert e.value.status == 3


def _schema(bt, **over):
    d = dict(B=bt.B, Lpad=bt.Lpad, row_stride=bt.H, lengths=bt.lengths, q_rec=bt.q_rec, q_type=bt.q_type,
             q_span=bt.q_span, q_opt_off=bt.q_opt_off, o_span=bt.o_span)
    d.update(over)
    return B.Schema(**d)


@pytest.fixture(scope="module")
def small_batch():
    spec = synth.BatchSpec(name="t", B=3, H=256, vocab=1000, length_law="uniform", length_range=(300, 700),
                           questions=(2, 4), options=(2, 5), instr_len=(3, 9), option_len=(2, 6))
    return synth.make_batch(spec, seed=2, with_hidden=False)


def test_workspace_size_valid(small_batch):
    cfg = B.make_config(H=256, vocab=1000)
    n = B.clef_workspace_size(cfg, _schema(small_batch))
    assert n > small_batch.T * 4096 * 2  # at least the K/V memory of both routing layers


def _expect(status, cfg, schema):
    with pytest.raises(B.ClefError) as e:
        B.clef_workspace_size(cfg, schema)
    assert e.value.status == status


def test_validation_errors(small_batch):
    bt = small_batch
    cfg = B.make_config(H=256, vocab=1000)
    bad_span = bt.q_span.copy()
    bad_span[0] = [5, 5]                       # empty span
    _expect(1, cfg, _schema(bt, q_span=bad_span))
    bad_span = bt.q_span.copy()
    bad_span[0, 1] = bt.lengths[bt.q_rec[0]] + 1  # past the record's real rows
    _expect(1, cfg, _schema(bt, q_span=bad_span))
    bad_o = bt.o_span.copy()
    bad_o[-1] = [-1, 2]
    _expect(1, cfg, _schema(bt, o_span=bad_o))
    _expect(1, cfg, _schema(bt, q_type=np.where(np.arange(bt.Q) == 0, 3, bt.q_type)))
    lens = bt.lengths.copy()
    lens[0] = bt.Lpad + 1
    _expect(1, cfg, _schema(bt, lengths=lens))
    _expect(1, cfg, _schema(bt, row_stride=bt.H - 8))
    _expect(1, cfg, _schema(bt, row_stride=bt.H + 4))
    rec = bt.q_rec.copy()
    rec[0], rec[-1] = rec[-1], rec[0]          # not grouped by record
    _expect(1, cfg, _schema(bt, q_rec=rec))
    off = bt.q_opt_off.copy()
    off[-1] += 1                               # CSR end != O
    _expect(1, cfg, _schema(bt, q_opt_off=off))


def test_noul_needs_two_options_and_records_need_questions(small_batch):
    bt = small_batch
    cfg = B.make_config(H=256, vocab=1000)
    q = int(np.nonzero(np.diff(bt.q_opt_off) > 2)[0][0])
    _expect(1, cfg, _schema(bt, q_type=np.where(np.arange(bt.Q) == q, 0, bt.q_type)))
    # drop record 1's questions: a record without a schema is rejected
    keep = bt.q_rec != 1
    opt_blocks = [np.arange(bt.q_opt_off[i], bt.q_opt_off[i + 1]) for i in np.nonzero(keep)[0]]
    o = np.concatenate(opt_blocks)
    off = np.concatenate([[0], np.cumsum([len(x) for x in opt_blocks])])
    _expect(1, cfg, _schema(bt, q_rec=bt.q_rec[keep], q_type=bt.q_type[keep], q_span=bt.q_span[keep],
                            q_opt_off=off, o_span=bt.o_span[o]))


def test_forward_rejects_before_launch(small_batch):
    """Null / misaligned pointers and bad schemas return an error without touching CUDA."""
    bt = small_batch
    cfg = B.make_config(H=256, vocab=1000)
    n = B.clef_weight_count(cfg)
    fake = [4096 * (i + 1) for i in range(n)]
    sch = _schema(bt)
    args = dict(prepared_ptr=1 << 20, hidden_ptr=1 << 21, token_ids_ptr=1 << 22, lexical_ptr=1 << 23,
                logits_ptr=1 << 24, probs_ptr=1 << 25, q_value_ptr=1 << 26, q_conf_ptr=1 << 27,
                q_argmax_ptr=1 << 28, workspace_ptr=1 << 29, workspace_bytes=1 << 40)
    a = dict(args, hidden_ptr=0)
    assert B.clef_head_forward(cfg, fake, schema=sch, check=False, **a) == 1
    a = dict(args, hidden_ptr=(1 << 21) + 2)     # misaligned hidden
    assert B.clef_head_forward(cfg, fake, schema=sch, check=False, **a) == 1
    a = dict(args, workspace_ptr=(1 << 29) + 128)  # workspace not 256-byte aligned
    assert B.clef_head_forward(cfg, fake, schema=sch, check=False, **a) == 1
    bad = fake.copy()
    bad[7] = 0
    assert B.clef_head_forward(cfg, bad, schema=sch, check=False, **args) == 1
    bad_span = bt.o_span.copy()
    bad_span[0] = [9, 3]
    assert B.clef_head_forward(cfg, fake, schema=_schema(bt, o_span=bad_span), check=False, **args) == 1
    a = dict(args, workspace_bytes=1024)
    assert B.clef_head_forward(cfg, fake, schema=sch, check=False, **a) == 2


def test_gemm_entry_validation():
    lib = B.load()
    flags = ctypes.c_int32(0)
    p = 1 << 20
    assert lib.clef_gemm_bf16(p, 64, p, 64, None, p, 64, 10, 64, 60, ctypes.addressof(flags), None) == 1  # K % 64
    assert lib.clef_gemm_bf16(p, 64, p, 64, None, p, 64, 10, 48, 64, ctypes.addressof(flags), None) == 1  # N % 64
    assert lib.clef_gemm_bf16(p, 60, p, 64, None, p, 64, 10, 64, 64, ctypes.addressof(flags), None) == 1  # lda
    assert lib.clef_gemm_bf16(0, 64, p, 64, None, p, 64, 10, 64, 64, ctypes.addressof(flags), None) == 1


def test_stream_rows_rejects_bad_ranges(small_batch):
    """Row ranges outside a record are rejected before anything is launched."""
    bt = small_batch
    cfg = B.make_config(H=256, vocab=1000)
    sch = _schema(bt)
    lib = B.load()
    args = lambda rec, r0, n: (ctypes.byref(cfg), 1 << 20, ctypes.byref(sch.struct), 1 << 21, rec, r0, n, 1 << 24,
                               1 << 40, None)
    L0 = int(bt.lengths[0])
    assert lib.clef_stream_rows(*args(-1, 0, 64)) == 1
    assert lib.clef_stream_rows(*args(bt.B, 0, 64)) == 1
    assert lib.clef_stream_rows(*args(0, -1, 64)) == 1
    assert lib.clef_stream_rows(*args(0, 0, 0)) == 1
    assert lib.clef_stream_rows(*args(0, L0 - 10, 11)) == 1
    assert lib.clef_stream_begin(ctypes.byref(cfg), ctypes.byref(sch.struct), 1 << 24, 1024, None) == 2


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the compiled library the binding raises; there is no fallback path."""
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libclef_head.so"))
    with pytest.raises(FileNotFoundError):
        B.load()
    with pytest.raises(FileNotFoundError):
        B.clef_weight_count(B.make_config())


def test_selftest_wait_timeout_validation():
    """Bad workspace pointers or limits are rejected before anything is launched."""
    assert B.clef_selftest_wait_timeout(0, 1_000_000, check=False) == 1
    assert B.clef_selftest_wait_timeout((1 << 20) + 16, 1_000_000, check=False) == 1
    assert B.clef_selftest_wait_timeout(1 << 20, 10, check=False) == 1
    assert B.clef_selftest_wait_timeout(1 << 20, 10**9, check=False) == 1


def test_repeated_schema_is_revalidated_when_changed_in_place(small_batch):
    """The library keeps the validated plan of the last schema it saw; a table changed in
    place (same pointers) must be validated again, and the restored table accepted."""
    bt = small_batch
    cfg = B.make_config(H=256, vocab=1000)
    sch = _schema(bt, q_span=bt.q_span.copy(), o_span=bt.o_span.copy(), lengths=bt.lengths.copy())
    n0 = B.clef_workspace_size(cfg, sch)
    assert B.clef_workspace_size(cfg, sch) == n0
    os_ = sch.o_span.reshape(-1, 2)
    keep = int(os_[0, 1])
    os_[0, 1] = os_[0, 0]                      # empty option span, written into the same buffer
    _expect(1, cfg, sch)
    os_[0, 1] = keep
    assert B.clef_workspace_size(cfg, sch) == n0
    keep_len = int(sch.lengths[1])
    sch.lengths[1] = bt.Lpad + 1               # longer than the padded rows
    _expect(1, cfg, sch)
    sch.lengths[1] = keep_len
    assert B.clef_workspace_size(cfg, sch) == n0
    other = _schema(bt, q_type=np.where(bt.q_type == 1, 2, bt.q_type))  # another valid schema in between
    B.clef_workspace_size(cfg, other)
    assert B.clef_workspace_size(cfg, sch) == n0
