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


# The GEMM kernels' own bounded waits, made to run out: in a child process
# whose wait limit is 1 us (the library reads MX_WAIT_LIMIT_NS once per
# process) a product runs until the device error word reports a timeout, and
# the same context must then quantize bit-exactly.  The cases:
#   512 x 512 x 32768 E4M3: the CTA-pair kernel (two-atom stages, two MMA
#     warps).  After the gate gives up the MMA warps issue nothing more, and
#     before the pair leaves every load either CTA issued has landed.
#   16 x 8192 x 32768 E4M3 x E2M1: the one-CTA decode kernel (operands
#     swapped, two MMA warps).  The producer refills a slot only once its
#     previous load has landed, and after a give-up the CTA waits for its last
#     loads before it leaves.
# The kernel whose activation warps quantize into the ring is not driven
# here: after a give-up its drain can wait for an activation warp's arrival
# that never comes, and then it waits out its limit of at least 1 s.
# K is long so that each CTA's waits last tens of microseconds: a wait looks
# at the clock only every 64 tries.  The waits that end a launch (loads and
# MMAs already issued) use at least 1 s.
_ABORT_CHILD = r"""
import sys
import numpy as np, torch
import bit_gemm_gb300 as mx
import oracle
M, N, K = (int(v) for v in sys.argv[1:4])
fa, fb = int(sys.argv[4]), int(sys.argv[5])
torch.manual_seed(7)
A = torch.randn(M, K, device="cuda")
B = torch.randn(N, K, device="cuda")
ac, as_ = mx.alloc_codes(M, K, fa), mx.alloc_scales(M, K, mx.SCALES_MMA)
bc, bs = mx.alloc_codes(N, K, fb), mx.alloc_scales(N, K, mx.SCALES_MMA)
mx.mx_quantize(A, fa, ac, as_, mx.SCALES_MMA)
mx.mx_quantize(B, fb, bc, bs, mx.SCALES_MMA)
mx.mx_device_status()
seen = 0
for attempt in range(20):
    C = torch.zeros(M, N, device="cuda")
    mx.mx_block_matmul(ac, as_, fa, bc, bs, fb, M, N, K, C, mx.SCALES_MMA)
    try:
        mx.mx_device_status()
    except mx.MxError as e:
        assert e.status == 5, e.status  # MX_ERR_TIMEOUT
        seen += 1
        break
assert seen, "no wait of the GEMM ran out within 1 us"
mx.mx_device_status()  # the word was cleared
x = torch.randn(64, 256, device="cuda")
codes, scales = mx.alloc_codes(64, 256, mx.E4M3FN), mx.alloc_scales(64, 256)
mx.mx_quantize(x, mx.E4M3FN, codes, scales)
mx.mx_device_status()
oc, os_ = oracle.quantize(x.cpu().numpy(), oracle.E4M3)
assert np.array_equal(codes.cpu().numpy().reshape(oc.shape), oc)
assert np.array_equal(scales.cpu().numpy().reshape(os_.shape), os_)
print("abort ok")
"""


@pytest.mark.parametrize("M,N,K,fa,fb", [
    (512, 512, 32768, mx.E4M3FN, mx.E4M3FN),  # CTA-pair kernel
    (16, 8192, 32768, mx.E4M3FN, mx.E2M1),    # one-CTA decode kernel
])
def test_gemm_waits_give_up_and_drain(M, N, K, fa, fb):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MX_WAIT_LIMIT_NS="1000")
    env["PYTHONPATH"] = os.pathsep.join([root, os.path.join(root, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", _ABORT_CHILD, str(M), str(N), str(K), str(fa), str(fb)], env=env,
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "abort ok" in r.stdout
