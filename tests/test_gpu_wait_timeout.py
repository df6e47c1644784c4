"""The failure path of the kernels' bounded waits (GPU).

Every mbarrier wait in the kernels gives up after a fixed budget (~2 s), raises
PA_DEV_TIMEOUT in the sticky status word and makes the thread block's later waits
return at once, so a copy that never lands ends the kernel with an error instead of
hanging the GPU.  Here the same wait helper runs on a barrier that nothing arrives on
(no fault, no trap: the wait simply runs out), and afterwards the context must still
decode correctly.
"""

import pytest
import torch

from _gpu_common import check_outputs, run_both
import workloads

pytestmark = pytest.mark.gpu


def test_wait_gives_up_reports_timeout_and_context_survives(pa):
    assert pa.pa_get_device_status() == 0
    first_ok, second_ok, first_cycles, second_cycles = pa.pa_selftest_wait_timeout()
    assert first_ok == 0 and second_ok == 0
    assert first_cycles > 4_000_000_000       # the whole budget was spent
    assert second_cycles < 1_000_000          # the aborting block's later wait returns at once
    assert pa.pa_get_device_status() & pa.PA_DEV_TIMEOUT
    assert pa.pa_get_device_status() == 0     # reading clears the sticky bits
    # the context is usable: a decode afterwards matches the oracle, with the automatic
    # launch options and with every context split into partitions (the arrival counters
    # of the workspace, re-zeroed after a timeout was read, decide which partition merges)
    w = workloads.build(1, small=True)
    _, outs, ref = run_both(pa, w)
    check_outputs(w, outs, ref)
    _, outs, ref = run_both(pa, w, params={"partition_tokens": 64})
    check_outputs(w, outs, ref)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
