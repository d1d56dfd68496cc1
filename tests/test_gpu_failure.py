"""Device-side failure path, made without a fault: a kernel whose bounded
wait runs out (a barrier nothing arrives at) records a timeout in the device
error word and returns; the host reads LLAMA_ERR_TIMEOUT, the word is cleared,
and the context keeps running kernels (checked against the oracle)."""

import time

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    assert lb.get_device_error()[0] == lb.LLAMA_OK  # nothing pending
    t0 = time.monotonic()
    lb.selftest_wait_timeout()
    st, detail = lb.get_device_error()  # synchronises
    elapsed = time.monotonic() - t0
    assert st == lb.LLAMA_ERR_TIMEOUT and detail == 64, (st, detail)
    assert 1.5 < elapsed < 60, elapsed  # the 2 s wall-clock limit of every wait
    assert lb.get_device_error() == (lb.LLAMA_OK, 0)  # read once, then cleared
    # the context still runs the library's kernels
    x = I.normal_bf16((100, 256), 1.0, 0.0, 1, DEV)
    w = I.normal_bf16((384, 256), 0.02, 0.0, 2, DEV)
    y = torch.empty((100, 384), dtype=torch.bfloat16, device=DEV)
    lb.linear(x, w, y, lb.alloc_workspace(lb.linear_workspace_size(), DEV))
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    ref = O.linear(x.float().cpu().numpy().astype(np.float64), w.float().cpu().numpy().astype(np.float64))
    got = y.float().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 2e-2 * np.max(np.abs(ref))
