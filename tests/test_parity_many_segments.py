"""GPU scans of batches past the host-side segment limits: the longest-first
ranking of the two-pass dense scan covers up to 4096 segments (beyond that the
state pass keeps the given order), and the diagonal scan's balanced schedule
indexes up to 512 segments in shared memory (beyond that, scratch or not, the
per-chain kernel runs).  Every segment is checked against the fp64 oracle, and
sampled segments bit for bit against the same segment scanned alone."""
import numpy as np
import pytest

import oracle
from helpers import TOL_SCAN_BF16, rel_fro, t_err, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def lengths(n, seed):
    """Mostly 0-3 tokens (empty segments included), a few spanning several chunks."""
    g = np.random.default_rng(seed)
    lens = g.integers(0, 4, size=n)
    lens[g.choice(n, size=6, replace=False)] = [64, 65, 130, 1, 200, 63]
    return [int(x) for x in lens]


def make(fam, lens, seed, H=1):
    if fam == wl.DENSE:
        return wl.dense_stack(lengths=lens, n_layers=1, H=H, d=128, seed=seed)
    return wl.scalar_diag(fam, lengths=lens, n_layers=1, H=H, d=128, seed=seed)


def scan(w, workspace="auto"):
    import torch
    import linear_attention_state_gated_gb300 as hy
    dev = lambda x: None if x is None else to_dev(x)   # noqa: E731
    got = hy.segment_scan(w["family"], to_dev(w["k"]).to(torch.bfloat16), to_dev(w["v"]).to(torch.bfloat16),
                          to_dev(w["alpha"]), to_dev(w["seg_offsets"]), beta=dev(w["beta"]), workspace=workspace)
    return {k: to_host(v) for k, v in got.items()}


def alone(w, s):
    offs = w["seg_offsets"]
    sl = slice(int(offs[s]), int(offs[s + 1]))
    one = dict(w, seg_offsets=np.array([0, sl.stop - sl.start], np.int64))
    for key in ("k", "v", "alpha", "beta"):
        if w.get(key) is not None:
            one[key] = np.ascontiguousarray(w[key][:, sl])
    return one


def check(w, got, sample_alone=(), workspace="auto"):
    fam = w["family"]
    ref = oracle.segment_scan(fam, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    assert rel_fro(got["S"], ref["S"]).max() <= TOL_SCAN_BF16
    assert t_err(fam, got["lam"], ref["lam"], got.get("M"), ref.get("M")).max() <= TOL_SCAN_BF16
    offs = w["seg_offsets"]
    empty = np.flatnonzero(offs[1:] == offs[:-1])
    assert np.all(got["S"][:, empty] == 0) and np.all(got["lam"][:, empty] == 0)
    for s in sample_alone:
        if offs[s + 1] == offs[s]:
            continue
        one = scan(alone(w, int(s)), workspace)
        for key in ("lam", "M", "S"):
            if key in got:
                assert np.array_equal(one[key][:, 0], got[key][:, s]), (key, s)


def test_dense_two_pass_beyond_the_ranking_limit():
    """4100 segments: more than the 4096 the longest-first ranking covers."""
    lens = lengths(4100, seed=500)
    w = make(wl.DENSE, lens, seed=501)
    got = scan(w)
    check(w, got, sample_alone=[int(np.argmax(lens)), 0, 4099, 2048])


def test_dense_two_pass_at_the_ranking_limit():
    lens = lengths(4096, seed=502)
    w = make(wl.DENSE, lens, seed=503)
    got = scan(w)
    check(w, got, sample_alone=[int(np.argmax(lens)), 4095])


@pytest.mark.parametrize("n_seg", [512, 600])
def test_diag_with_scratch_around_the_balanced_limit(n_seg):
    """512 segments: the balanced schedule's limit (it runs); 600: the per-chain
    kernel runs although scratch is given.  Both match the oracle; the
    per-chain one is also bit-exact against a segment scanned alone."""
    lens = lengths(n_seg, seed=510 + n_seg)
    w = make(wl.DIAG, lens, seed=511 + n_seg, H=2)
    got = scan(w, workspace="auto")
    # alone, a segment would take the balanced schedule again: compare with the
    # per-chain kernel (no scratch), which the 600-segment batch ran
    check(w, got, sample_alone=[int(np.argmax(lens))] if n_seg > 512 else (), workspace=None)


def test_scalar_many_segments():
    lens = lengths(5000, seed=520)
    w = make(wl.SCALAR, lens, seed=521, H=2)
    got = scan(w, workspace=None)
    check(w, got, sample_alone=[int(np.argmax(lens)), 4999], workspace=None)
