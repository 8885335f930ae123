"""Failure detection on the GPU without a fault: a kernel waits on a barrier
that nothing will complete, gives up after its short limit, reports through
the device error word, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_reports_timeout():
    mx.mx_selftest_wait_timeout(2_000_000)  # 2 ms
    with pytest.raises(mx.MxError) as e:
        mx.mx_device_status()
    assert e.value.status == 5  # MX_ERR_TIMEOUT
    mx.mx_device_status()       # the word was cleared: a second check is clean
    # the context still works
    x = torch.randn(4, 64, device="cuda")
    codes, scales = mx.alloc_codes(4, 64, mx.E2M1), mx.alloc_scales(4, 64)
    mx.mx_quantize(x, mx.E2M1, codes, scales)
    mx.mx_device_status()
    oc, os_ = oracle.quantize(x.cpu().numpy(), oracle.E2M1)
    assert np.array_equal(codes.cpu().numpy().reshape(oc.shape), oc)
