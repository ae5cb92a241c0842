"""The failure path of the bounded device waits, exercised without hanging or
faulting the GPU: a kernel waits on an mbarrier that nothing completes, gives
up after its wall-time bound and records WQ_ERR_DEVICE_TIMEOUT; the status is
read and cleared, and the context keeps working."""
import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import check_full

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_cleared():
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert wq.wq_selftest_timeout(None) == wq.WQ_OK
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_get_device_error() == wq.WQ_OK          # read clears it
    # the context is still usable: a full GEMM on both paths
    check_full(synth.make_problem("int4", 300, 256, 512, seed=1), "fp32", what="after timeout")
    check_full(synth.make_problem("nvfp4", 4, 256, 512, seed=2), "fp32", what="after timeout")
    assert wq.wq_get_device_error() == wq.WQ_OK
