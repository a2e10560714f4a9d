"""Bounded device-side waits: a wait that can never complete gives up after
the configured limit, records LL_ERR_DEVICE_TIMEOUT in the status word and
returns; the context stays usable.  No fault, trap or hang is involved."""
import pytest
import torch

from cross_entropy_rl_gb300 import synth
from gpu_util import dev

pytestmark = pytest.mark.gpu


def test_unsatisfied_wait_times_out_and_reports(lib):
    L = lib.load()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.ll_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        st = L.ll_debug_unsatisfied_wait(lib._ptr(flag), lib._stream())
        assert st == 0
        assert lib.check_status() == 7     # LL_ERR_DEVICE_TIMEOUT
        assert int(flag.item()) == 1       # the kernel took its timeout path
        assert lib.check_status() == 0     # the status word was cleared
    finally:
        L.ll_set_wait_limit_ns(0)          # back to the default limit
    # the context is still usable: a normal call succeeds
    p = synth.linear_inputs(64, 64, 300, dtype="bf16", seed=1)
    logp, lse = lib.forward(dev(p["h"], "bf16"), dev(p["W"], "bf16"), None, dev(p["y"]))
    torch.cuda.synchronize()
    assert torch.isfinite(logp).all()
    assert lib.check_status() == 0
