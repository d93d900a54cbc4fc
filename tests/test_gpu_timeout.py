"""A bounded device wait that runs out, on purpose, through the test hook.

kda_test_set_fault makes CTA 0 of one kernel withhold one mbarrier arrival
(the scan: an epilogue arrival; the preparation and the single-pass kernel:
their first MMA group and its commit).  Its wait then gives up after about a
second: the kernel must write KDA_ERR_TIMEOUT to the status word, let its
copies and MMAs in flight finish, release its tensor memory and return, with
no CUDA error.  The next ordinary call must give exactly the bits of a run
made before the fault.  Nothing here traps or faults the GPU: the lost
arrival is a flag that nothing sets, and every wait on it is bounded."""
import pytest
import torch

from kimi_delta_attention_10_gb300 import kda_chunk_fwd, kda_gate
from kimi_delta_attention_10_gb300.binding import (KDA_ERR_TIMEOUT, KDA_TEST_FAULT_NONE,
                                                   KDA_TEST_FAULT_PREP, KDA_TEST_FAULT_SCAN,
                                                   KDA_TEST_FAULT_SINGLE_PASS, set_test_fault)
from kimi_delta_attention_10_gb300.inputs import make_inputs

from gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def _call(d, g, beta, x, workspace, mode):
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           mode=mode, workspace=workspace, status=status,
                           out_dtype=torch.float32 if mode == "fp32_exact" else None,
                           cu_seqlens_host=x.cu_seqlens.tolist())
    torch.cuda.synchronize()                 # raises if the kernel faulted
    return out.clone(), S.clone(), int(status[0])


# (fault, mode, workspace, lengths, heads): the short problem runs the scan in V
# halves, the 8192-token one the full-width scan in three chunk windows (its CTA
# 0 gives up once per window); the FP32-exact mode's scan is a tensor-core
# scan in V halves too
CASES = [(KDA_TEST_FAULT_SCAN, "bf16_tc", "auto", [300, 77], 2),
         (KDA_TEST_FAULT_SCAN, "bf16_tc", "auto", [8192], 1),
         (KDA_TEST_FAULT_PREP, "bf16_tc", "auto", [300, 77], 2),
         (KDA_TEST_FAULT_SINGLE_PASS, "bf16_tc", None, [300, 77], 2),
         (KDA_TEST_FAULT_SCAN, "fp32_exact", "auto", [300, 77], 2)]


@pytest.mark.parametrize("where,mode,workspace,lens,H", CASES)
def test_lost_arrival_times_out_and_the_next_call_is_clean(where, mode, workspace, lens, H):
    x = make_inputs(lens, H, 128, 128, torch.bfloat16, 71)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    o_ref, S_ref, st = _call(d, g, beta, x, workspace, mode)
    assert st == 0
    set_test_fault(where)
    try:
        _, _, st_fault = _call(d, g, beta, x, workspace, mode)
    finally:
        set_test_fault(KDA_TEST_FAULT_NONE)
    assert st_fault == KDA_ERR_TIMEOUT
    o2, S2, st2 = _call(d, g, beta, x, workspace, mode)
    assert st2 == 0
    assert torch.equal(o2, o_ref) and torch.equal(S2, S_ref)
