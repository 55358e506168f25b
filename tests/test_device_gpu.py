"""The device the library runs on has the SM count its plans assume.

The launch plans cut every shape into 152 x (CTAs per SM) persistent CTAs
(a function of the shape alone, for determinism); every launching call
checks the current device's SM count against that and refuses a smaller
device. This test reads the count the way the library does and the way
torch does, prints it, and checks that the device passes.
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def test_device_sm_count_meets_the_plans():
    n = m.mcc1d_device_sm_count()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    print(f"{props.name}: {n} SMs (torch: {props.multi_processor_count}); plans assume {m.PLAN_SMS}")
    assert n == props.multi_processor_count
    assert m.mcc1d_check_sm_count(n) == 0, m.mcc1d_status_string(m.mcc1d_check_sm_count(n))
