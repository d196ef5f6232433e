"""Failure detection without a GPU fault.

* Device side: every pipeline wait in the kernels is bounded and, when it runs
  out, leaves HYPIC_ETIMEOUT in the caller's status word and returns.  The
  bounded-wait diagnostic runs that wait on its own with a short limit on a
  barrier nothing arrives on; the status comes back, and the context stays
  usable (a scan right after it matches the oracle).
* Host side: a scratch allocation that fails inside the Python binding raises
  before anything is launched (the outputs keep their contents)."""
import numpy as np
import pytest

import oracle
from helpers import TOL_SCAN_BF16, rel_fro, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ETIMEOUT = -6


def test_bounded_wait_gives_up_and_reports():
    import torch
    import linear_attention_state_gated_gb300 as hy
    limit = 2_000_000   # about 1 ms of SM clock
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    hy.selftest_wait(limit, arrive=False, d_err=err, cycles=cyc)
    torch.cuda.synchronize()
    assert int(err.item()) == ETIMEOUT
    # gave up at its own short limit, far below the pipelines' ~4e9-cycle one
    assert limit < int(cyc.item()) < 500 * limit
    # the context is still usable: a scan right after it is correct
    w = wl.scalar_diag(wl.DIAG, lengths=[100, 37], n_layers=1, H=2, d=128, seed=400)
    got = hy.segment_scan(wl.DIAG, to_dev(w["k"]).to(torch.bfloat16), to_dev(w["v"]).to(torch.bfloat16),
                          to_dev(w["alpha"]), to_dev(w["seg_offsets"]), d_err=err)
    ref = oracle.segment_scan(wl.DIAG, w["k"], w["v"], w["alpha"], w["seg_offsets"])
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_SCAN_BF16
    assert int(err.item()) == ETIMEOUT   # the scan leaves the status word alone when it succeeds


def test_bounded_wait_completes_when_arrived():
    import torch
    import linear_attention_state_gated_gb300 as hy
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cyc = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    hy.selftest_wait(2_000_000, arrive=True, d_err=err, cycles=cyc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert 0 <= int(cyc.item()) < 100_000


def test_failed_scratch_allocation_raises_before_launch(monkeypatch):
    """The binding allocates the two-pass scan's scratch through torch; an
    allocation failure there surfaces as the caller's exception and nothing runs."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    w = wl.dense_stack(lengths=[90], n_layers=1, H=2, d=128, seed=401)
    args = (wl.DENSE, to_dev(w["k"]).to(torch.bfloat16), to_dev(w["v"]).to(torch.bfloat16), to_dev(w["alpha"]),
            to_dev(w["seg_offsets"]))
    out = {"lam": torch.full((1, 1, 2), 7.0, device="cuda"), "M": torch.full((1, 1, 2, 128, 128), 7.0, device="cuda"),
           "S": torch.full((1, 1, 2, 128, 128), 7.0, device="cuda")}
    real_empty = torch.empty

    def failing_empty(*a, **kw):
        if kw.get("dtype") == torch.uint8:
            raise torch.cuda.OutOfMemoryError("injected: scratch allocation failed")
        return real_empty(*a, **kw)

    monkeypatch.setattr(hy.torch, "empty", failing_empty)
    with pytest.raises(torch.cuda.OutOfMemoryError):
        hy.segment_scan(*args, beta=to_dev(w["beta"]), out=out)
    monkeypatch.undo()
    torch.cuda.synchronize()
    for t in out.values():
        assert torch.all(t == 7.0)
    # with the allocator back the same call runs and is correct
    got = hy.segment_scan(*args, beta=to_dev(w["beta"]), out=out)
    ref = oracle.segment_scan(wl.DENSE, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_SCAN_BF16
