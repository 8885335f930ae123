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


# The pair GEMM's own bounded waits, made to run out: in a child process whose
# wait limit is 1 us (the library reads MX_WAIT_LIMIT_NS once per process), a
# 512 x 512 x 2048 E4M3 product takes the CTA-pair kernel with two-atom stages
# and two MMA warps; its gate gives up on a stage that has not landed within
# 1 us, the MMA warps stop issuing, the producers stop on their next slot wait,
# and before the CTAs leave, the even CTA waits (with a limit of at least 1 s)
# for every load either CTA issued and the MMA warps for every MMA.  The child
# checks that the device error word reports the timeout and that the same
# context then quantizes bit-exactly.
_PAIR_ABORT_CHILD = r"""
import numpy as np, torch
import bit_gemm_gb300 as mx
import oracle
rng = np.random.default_rng(7)
M = N = 512
K = 2048
A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).cuda()
B = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)).cuda()
ac, as_ = mx.alloc_codes(M, K, mx.E4M3FN), mx.alloc_scales(M, K, mx.SCALES_MMA)
bc, bs = mx.alloc_codes(N, K, mx.E4M3FN), mx.alloc_scales(N, K, mx.SCALES_MMA)
mx.mx_quantize(A, mx.E4M3FN, ac, as_, mx.SCALES_MMA)
mx.mx_quantize(B, mx.E4M3FN, bc, bs, mx.SCALES_MMA)
mx.mx_device_status()
seen = 0
for attempt in range(5):
    C = torch.zeros(M, N, device="cuda")
    mx.mx_block_matmul(ac, as_, mx.E4M3FN, bc, bs, mx.E4M3FN, M, N, K, C, mx.SCALES_MMA)
    try:
        mx.mx_device_status()
    except mx.MxError as e:
        assert e.status == 5, e.status  # MX_ERR_TIMEOUT
        seen += 1
        break
assert seen, "no wait of the pair kernel ran out within 1 us"
mx.mx_device_status()  # the word was cleared
x = torch.randn(64, 256, device="cuda")
codes, scales = mx.alloc_codes(64, 256, mx.E4M3FN), mx.alloc_scales(64, 256)
mx.mx_quantize(x, mx.E4M3FN, codes, scales)
mx.mx_device_status()
oc, os_ = oracle.quantize(x.cpu().numpy(), oracle.E4M3)
assert np.array_equal(codes.cpu().numpy().reshape(oc.shape), oc)
assert np.array_equal(scales.cpu().numpy().reshape(os_.shape), os_)
print("pair abort ok")
"""


def test_pair_gemm_waits_give_up_and_drain():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MX_WAIT_LIMIT_NS="1000")
    env["PYTHONPATH"] = os.pathsep.join([root, os.path.join(root, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", _PAIR_ABORT_CHILD], env=env, cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "pair abort ok" in r.stdout
