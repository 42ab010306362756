"""Failure detection on the GPU without a fault: every wait in the library's
kernels is bounded, and a wait that runs out is reported through the device
status word while the context stays usable.  The self-test kernel waits on a
barrier that nothing completes (ql_selftest_wait); the test checks the status
the host reads, that reading it clears it, and that ordinary work still runs
and stays correct afterwards."""
import numpy as np
import pytest
import torch

from oracle import nf4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def test_bounded_wait_reports_timeout_and_context_survives(ql):
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, normal_bf16
    ql.device_status()  # nothing pending
    ql.selftest_wait(5_000_000)  # 5 ms
    with pytest.raises(ql.QLError) as e:
        ql.device_status()
    assert e.value.code == ql.QL_ERR_TIMEOUT
    ql.device_status()  # the read cleared the word

    # the context still works: a quantization afterwards is bit-exact
    W = normal_bf16((256, 512), 0.02, 11)
    q = ql.nf4_quantize(W.to("cuda"))
    torch.cuda.synchronize()
    ql.device_status()
    ref = nf4.quantize(bf16_bits(W), 64, 256)
    assert np.array_equal(q.packed.cpu().numpy().reshape(-1), ref["packed"].reshape(-1))
    assert np.array_equal(q.absmax_code.cpu().numpy().reshape(-1), ref["code"].reshape(-1))
    assert np.array_equal(q.dq_step.cpu().numpy().view(np.uint32), ref["step"].view(np.uint32))


def test_timeout_does_not_leak_into_the_next_call(ql):
    ql.selftest_wait(1_000_000)
    with pytest.raises(ql.QLError):
        ql.device_status()
    for _ in range(3):
        ql.device_status()
