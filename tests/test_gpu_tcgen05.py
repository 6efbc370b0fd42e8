"""fc1 rows on the tcgen05 kernel (dv_set_row_kernel(1)): the layer decode
against the oracle at batch tiles of 16 and 32 rows, ragged batches, and the
switch back to the default kernel."""
import pytest

import dv_inputs
from parity import check_layer_parity, make_case, run_gpu_layer

pytestmark = pytest.mark.gpu
CFG = dv_inputs.CONFIGS


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


@pytest.fixture
def tc(dv):
    dv.dv_set_row_kernel(1)
    yield dv
    dv.dv_set_row_kernel(0)


@pytest.mark.parametrize("B", [9, 16, 25, 32])
def test_opt67b_fc1_on_tcgen05(tc, B):
    case = make_case(CFG["opt6.7b"], B=B, gen_device="cuda", norm_affine=True, seed=70 + B)
    g = run_gpu_layer(tc, case)
    check_layer_parity(case, g)


def test_opt175b_fc1_on_tcgen05_batch16(tc):
    # d = 12288: six K segments of 2048, partials added in segment order
    case = make_case(CFG["opt175b"], B=16, gen_device="cuda", norm_affine=False, seed=5)
    g = run_gpu_layer(tc, case)
    check_layer_parity(case, g)

