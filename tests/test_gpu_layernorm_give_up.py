"""The LayerNorm kernel's give-up path, exercised without any fault.

Each CTA of the LayerNorm kernel waits at most one second for the bulk copy of
each batch of rows.  Should a wait run out, the CTA marks *amax with the bit
pattern 0x7FFFFFFF, waits (bounded) for the copies it still has in flight and
returns.  In correct operation every copy arrives, so this test uses the
library built once more with the test hook FP8Q_TEST_LN_GIVE_UP_AT=1: the wait
for each CTA's second batch then reports failure although its copy did arrive.
The call must return, leave the marker in amax, have finished each CTA's first
batch exactly as the normal library does, and leave the device usable.  Rows longer
than 4096 run on thread-block clusters, whose CTAs agree at the cluster barrier: the
whole cluster stops after its first batch.
"""
import numpy as np
import pytest
import torch

from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,H", [(4096, 4096), (4096, 12288)])   # one CTA a batch; a cluster of 3 a batch
def test_layernorm_give_up_marks_amax_and_returns(hooks_lib, rows, H):
    hooked = hooks_lib
    dev = torch.device("cuda:0")
    x = W.residual_stream(seed=13, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, device=dev)
    scale = torch.full((1,), 0.03, device=dev)
    q = torch.zeros((rows, H), dtype=torch.uint8, device=dev)
    am = torch.zeros(1, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    status = hooked.fp8q_layernorm_quantize_amax(x.data_ptr(), None, q.data_ptr(), rows, H, gamma.data_ptr(),
                                                 beta.data_ptr(), 1e-6, fp8q.E4M3FN, scale.data_ptr(),
                                                 am.data_ptr(), st)
    assert status == 0
    torch.cuda.synchronize()                 # the call returns: nothing waits forever
    assert am.view(torch.int32).item() == 0x7FFFFFFF
    assert np.isnan(am.item())
    # each CTA finished its first batch before giving up: those rows match the normal library
    q_ok = torch.empty_like(q)
    am_ok = torch.zeros(1, device=dev)
    fp8q.fp8q_layernorm_quantize_amax(x, None, q_ok, gamma, beta, fp8q.E4M3FN, scale, am_ok)
    torch.cuda.synchronize()
    done = (q != 0).any(dim=1)
    assert int(done.sum()) > 0
    assert torch.equal(q[done], q_ok[done])
    # and most rows were never written: every CTA stopped after one batch
    assert int(done.sum()) < rows // 2
    # the device is still usable
    assert torch.isfinite(am_ok).all() and am_ok.item() > 0
