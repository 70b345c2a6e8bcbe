"""Failure detection on the GPU without a fault: a kernel waits on a barrier
that nothing arrives on; the bounded wait gives up after 20 ms, the kernel
returns, and the host sees FA_ERR_TIMEOUT.  The context stays usable."""
import pytest
import torch

import exact_tiled_attention_10_gb300 as fa

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    fa.check_device_status()  # clean start
    flag = fa.selftest_wait_timeout(20000)
    assert flag == 0
    with pytest.raises(fa.FAError) as ei:
        fa.check_device_status()
    assert ei.value.status == fa.FA_ERR_TIMEOUT
    fa.check_device_status()  # the word was cleared
    # the context still works: a normal forward runs and matches a second run
    from exact_tiled_attention_10_gb300.inputs import qkv
    q, k, v = qkv(1, 2, 256, 64, 3, device="cuda", with_dout=False)
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    fa.check_device_status()
