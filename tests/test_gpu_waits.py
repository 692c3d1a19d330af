"""Every wait in the kernels is bounded: a wait on a condition nothing satisfies gives up, records
MOE_ERR_TIMEOUT's bit in the device error word, and leaves the context usable.  The failure is
made without any fault: a counter nobody increments, an mbarrier no producer fills."""
import time

import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import Shape
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1])
def test_wait_gives_up_and_reports(kind):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    Bn.debug_wait_timeout(kind, err)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(err.item()) & 2
    # the context still works: a normal forward right after
    shape = Shape("after", 128, 64, 4, 2, 4, 4, 4, seed=61)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    blk = Bn.MoeDecode(layer)
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                      C.dev(r, torch.bfloat16))
    torch.cuda.synchronize()
    assert blk.get_error() == 0
    blk.close()
    C.assert_parity(out.cpu().numpy()[0], C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0]))
