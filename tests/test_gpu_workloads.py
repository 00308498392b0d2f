"""Full-size workloads on the GPU, in the launch configuration the benchmark times.

The whole batch runs on the GPU in the launch configuration the benchmark times;
the oracle recomputes every record of it one by one (records are independent, so
each record's outputs are exact oracle outputs), and properties that hold at any
size are checked on every question as well.
"""
import numpy as np
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library
from structured_decision_model_gb300.head import to_device_bf16

from gpu_support import compare, device_lexical, head_for, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()


def device_hidden(bt):
    """[B, Lpad, H] on the device: real rows from the generator, padding zero."""
    hid = torch.zeros((bt.B, bt.Lpad, bt.H), dtype=torch.bfloat16, device="cuda")
    for b in range(bt.B):
        hid[b, :bt.lengths[b]] = to_device_bf16(bt.real_rows(b))
    return hid


def check_properties(bt, gpu):
    for q in range(bt.Q):
        lo, hi = bt.q_opt_off[q], bt.q_opt_off[q + 1]
        p = gpu["probs"][lo:hi]
        assert np.isfinite(gpu["logits"][lo:hi]).all()
        assert abs(p.sum() - 1.0) < 1e-4
        k = int(gpu["q_argmax"][q])
        assert 0 <= k < hi - lo and p[k] == p.max()
        assert abs(gpu["q_conf"][q] - p.max()) < 1e-6
        if bt.q_type[q] == 2:
            assert -1e-5 <= gpu["q_value"][q] <= hi - lo - 1 + 1e-5
        elif bt.q_type[q] == 0:
            assert abs(gpu["q_value"][q] - p[0]) < 1e-6


WORKLOADS = ["pr1_ref_b1_l512", "batch32_l1k_4k", "batch8_l16k", "wide_h5120_b16_l8k", "serving_mix_b64",
             "short_b256"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_every_record(name):
    spec = synth.workload_spec(name)
    shape = synth.HeadShape(H=spec.H)
    bt = synth.make_batch(spec, seed=1, with_hidden=False)
    head, w = head_for(shape)
    inputs = (device_hidden(bt), torch.from_numpy(bt.token_ids).cuda(), device_lexical(bt, shape.vocab))
    gpu = run_gpu(head, bt, inputs=inputs)
    check_properties(bt, gpu)
    ref = run_oracle(w, shape, bt)
    stats = compare(gpu, ref, bt)
    print(name, bt.B, "records", stats)
