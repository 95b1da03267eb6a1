"""The bounded-wait path: a kernel whose wait runs out records SSD_ERR_TIMEOUT
in the device error word, frees its tensor memory and returns, and the
context stays usable (no trap, no fault).  The wait that runs out is the
self-test kernel's, on a barrier nothing completes, with a 20 ms limit."""
import numpy as np
import pytest
import torch

from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_reports_timeout():
    S.ssd_check_device_error()  # start from a clear error word
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    S.ssd_selftest_timeout(20_000_000)
    t1.record()
    with pytest.raises(S.SsdError) as e:
        S.ssd_check_device_error()
    assert e.value.status == S.SSD_ERR_TIMEOUT
    assert 15.0 <= t0.elapsed_time(t1) < 1000.0  # it waited for its limit, then returned
    S.ssd_check_device_error()  # reading the word cleared it


def test_context_usable_after_timeout():
    S.ssd_selftest_timeout(2_000_000)
    with pytest.raises(S.SsdError):
        S.ssd_check_device_error()
    # the tensor-core prefill still runs (tensor memory was freed) and is right
    shape = synth.FwdShape(1, 300, 2, 64, 128, 1, 1, 256, synth.BF16, "zero")
    inp = synth.make_fwd_inputs(shape, 5)
    d = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in inp.items()}
    for k in ("x", "B", "C"):
        d[k] = d[k].to(torch.bfloat16)
    y, hf = S.forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, chunk=256)
    S.ssd_check_device_error()
    assert torch.isfinite(y.float()).all() and torch.isfinite(hf).all()


def test_limit_out_of_range_is_rejected_before_launch():
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(S.SsdError) as e:
            S.ssd_selftest_timeout(bad)
        assert e.value.status == S.SSD_ERR_INVALID_ARG
