"""The bounded-wait path every kernel relies on, exercised on the GPU without a fault: a wait
that nothing completes runs out, reports through the status and the error word, and the
context stays usable for the next layer."""
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, linear
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_the_context_stays_usable():
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    assert binding.read_error_flags() == 0
    assert binding.selftest_wait_timeout(10000) == 1          # 10 ms limit
    assert binding.read_error_flags() == 1 << 5               # recorded, then cleared by the read
    assert binding.read_error_flags() == 0
    # a layer right after it runs and is correct
    W = inputs.weights(91, 300, 512, 0.05)
    pk = int4_g128.quantize(W)
    xb, xf = inputs.activations(92, 3, 512)
    Y = binding.gemm_w4a16("int4_g128", x_to_dev(xb), *[to_dev(a) for a in pk])
    assert_close(y_to_host(Y), linear.linear_w4a16("int4_g128", xf, *pk), "after the diagnostic")
    assert binding.read_error_flags() == 0
