"""Device-side failure detection on a GB300, without a fault: a bounded wait that nothing
satisfies gives up by its limit, the status word reports it, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

from parity_rules import dev, dev_bf16, host
from speculative_decoding_drafter_gb300 import dflash2 as df
from speculative_decoding_drafter_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

DF2_ERR_TIMEOUT = 5


def test_bounded_wait_times_out_and_reports():
    x = make_inputs("tiny", 0)
    cfg = x["cfg"]
    ws = df.Workspace(df.make_dims(cfg.B, cfg.T, cfg.H, cfg.V, cfg.k, cfg.D))
    df.dflash2_check_device_status(ws)  # clean start
    limit_us = 20000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    df.dflash2_selftest_wait_timeout(ws, limit_us)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed >= limit_us * 1e-6, f"the wait ended after {elapsed:.4f} s, before its limit"
    assert elapsed < 5.0
    with pytest.raises(df.DFlash2Error) as err:
        df.dflash2_check_device_status(ws)
    assert err.value.status == DF2_ERR_TIMEOUT
    df.dflash2_check_device_status(ws)  # the check cleared the word

    # the context is still usable: the same workspace runs the selector head
    d = {n: dev_bf16(x[n]) for n in ("hidden", "W_vocab", "W_sel", "pred_cb", "succ_cb")}
    lat, draft = df.dflash2_select(d["hidden"], d["W_vocab"], d["W_sel"], d["pred_cb"], d["succ_cb"],
                                   dev(x["anchor"]), cfg.k, cfg.T, workspace=ws)
    torch.cuda.synchronize()
    df.dflash2_check_device_status(ws)
    ids = host(lat)[:, :cfg.k]
    assert np.all((ids >= 0) & (ids < cfg.V))
    assert host(draft).shape == (cfg.B, cfg.T)


@pytest.mark.parametrize("pinned_status", [True, False])
def test_host_call_reports_a_sticky_status(pinned_status):
    """A status bit left in the workspace reaches the host call's result on both of its paths:
    the finish kernel's write into the page-locked status word, and the copy into a stack word."""
    x = make_inputs("tiny", 0)
    cfg = x["cfg"]
    d = {n: dev_bf16(x[n]) for n in ("W_vocab", "W_sel", "pred_cb", "succ_cb")}
    h_hidden = torch.from_numpy(x["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_anchor = torch.from_numpy(x["anchor"]).pin_memory()
    hw = df.HostWorkspace(df.make_dims(cfg.B, cfg.T, cfg.H, cfg.V, cfg.k, cfg.D))
    plan = df.SelectHostPlan(h_hidden, d["W_vocab"], d["W_sel"], d["pred_cb"], d["succ_cb"], h_anchor, cfg.k, cfg.T,
                             workspace=hw, pinned_status=pinned_status)
    _, draft_ok = plan()
    draft_ok = draft_ok.clone()
    df.dflash2_selftest_wait_timeout(hw, 2000)  # sets the sticky bit, nothing else
    torch.cuda.synchronize()
    with pytest.raises(df.DFlash2Error) as err:
        plan()
    assert err.value.status == DF2_ERR_TIMEOUT
    with pytest.raises(df.DFlash2Error):
        df.dflash2_check_device_status(hw)  # reports the word once more and clears it
    _, draft = plan()
    assert np.array_equal(draft.numpy(), draft_ok.numpy())
