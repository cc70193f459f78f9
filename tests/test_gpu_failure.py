"""Failure detection on the GPU without a fault: the kernels' bounded mbarrier
wait is made to run out on a barrier that nothing arrives on.  The expiry is
reported in a status word, the kernel finishes, and the context keeps working
(a prefill right after matches the oracle and reports status 0)."""
import time

import pytest
import torch

from kimi_delta_attention_varlen_gb300 import (kda_prefill_varlen, kda_prefill_workspace_size,
                                               kda_prefill_workspace_status, kda_selftest_bounded_wait)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, f64, oracle_prefill_from_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_completes_reports_zero():
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    kda_selftest_bounded_wait(status, polls=1000, arrive=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("polls", [1, 1000, 20000])
def test_wait_that_never_completes_expires_and_reports(polls):
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    kda_selftest_bounded_wait(status, polls=polls, arrive=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


def test_wait_is_bounded_in_time():
    """With a poll budget that would never run out, the global-timer bound ends the
    wait after about one second."""
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t = time.perf_counter()
    kda_selftest_bounded_wait(status, polls=0xFFFFFFFF, arrive=False)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t
    assert int(status.item()) == 1
    assert 0.5 < dt < 10.0, dt


def test_context_usable_after_an_expired_wait():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_selftest_bounded_wait(status, polls=1000, arrive=False)
    lengths = [130, 64, 1]
    H, D = 2, 128
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=4, device=DEV)
    out = torch.empty(cu[-1], H, D, dtype=torch.bfloat16, device=DEV)
    fin = torch.empty(len(lengths), H, D, D, dtype=torch.float32, device=DEV)
    ws = torch.empty(kda_prefill_workspace_size(cu[-1], len(lengths), H, D, D), dtype=torch.uint8, device=DEV)
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                       torch.tensor(cu, dtype=torch.int32, device=DEV), out, ws, final_state=fin)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert kda_prefill_workspace_status(ws) == 0
    o_ref, f_ref, _ = oracle_prefill_from_device(inp, cu, None, D ** -0.5)
    assert_out_close(f64(out), o_ref)
    assert_state_close(f64(fin), f_ref)
