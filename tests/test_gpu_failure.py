"""Failure detection on the GPU without a fault: bounded waits run out.

The self-test kernel waits on a shared-memory barrier that nothing completes, then on a
global flag that nothing sets (the two forms of every wait in the head's kernels), each
with a short limit.  Each wait gives up, sets the timeout bit of the workspace status
word and records itself; the kernel returns; the host reads CLEF_ERR_DEVICE_TIMEOUT, and
the context keeps working (a forward pass after it still matches the oracle).
"""
import pytest
import torch

import synth
from structured_decision_model_gb300 import binding as B
from structured_decision_model_gb300.build import build_library

from gpu_support import compare, head_for, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    B.load()
    torch.cuda.init()


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    B.clef_selftest_wait_timeout(ws.data_ptr(), 20_000_000, st)  # 20 ms per wait
    torch.cuda.synchronize()
    assert int(ws[8:12].view(torch.int32).item()) == 3             # both waits gave up
    assert B.clef_device_status(ws.data_ptr(), st) == 6            # CLEF_ERR_DEVICE_TIMEOUT
    assert B.clef_device_status(ws.data_ptr(), st) == 0            # read clears it
    shape = synth.HeadShape(H=256, vocab=2000)
    spec = synth.BatchSpec(name="after_timeout", B=2, H=256, vocab=2000, length_law="uniform",
                           length_range=(300, 500), questions=(2, 3), options=(2, 4), instr_len=(3, 8), option_len=(2, 5))
    bt = synth.make_batch(spec, seed=21)
    head, w = head_for(shape)
    compare(run_gpu(head, bt), run_oracle(w, shape, bt), bt)
