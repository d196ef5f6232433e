"""GPU segment scan against the fp64 oracle on the same seeded inputs.

Small ragged cases are compared element by element over every (layer,
segment, head); the full-size workloads run in the configuration the
benchmark times and are compared on sampled (layer, segment, head) units the
oracle computes one by one."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, TOL_O_BF16, TOL_SCAN_BF16, rel_fro, t_err, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCALAR, DIAG, DENSE = wl.SCALAR, wl.DIAG, wl.DENSE


def gpu_scan(w, want_o=False, d_err=None, workspace="auto"):
    import linear_attention_state_gated_gb300 as hy
    dt = w["dtype"]
    return hy.segment_scan(w["family"], to_dev(w["k"], dt), to_dev(w["v"], dt),
                           to_dev(w["alpha"]), to_dev(w["seg_offsets"]), beta=to_dev(w["beta"]),
                           q=to_dev(w["q"], dt) if want_o else None, want_o=want_o, d_err=d_err,
                           workspace=workspace)


# the dense bf16 d = 128 scan has two forms: two passes over scratch (the
# default, "auto") and the single-pass kernel (no scratch, None)
DENSE_FORMS = pytest.mark.parametrize("form", ["auto", None], ids=["two_pass", "single_pass"])


def host(out):
    return {k: to_host(v) for k, v in out.items()}


def check(fam, got, ref, tol, o_tol=None, seg_offsets=None):
    e_s = rel_fro(got["S"], ref["S"])
    e_t = t_err(fam, got["lam"], ref["lam"], got.get("M"), ref.get("M"))
    assert e_s.max() <= tol, f"S error {e_s.max():.3e} > {tol}"
    assert e_t.max() <= tol, f"T error {e_t.max():.3e} > {tol}"
    if o_tol is not None:
        # per (layer, segment, head): relative Frobenius over the segment's rows of o
        go, ro = got["o"], ref["o"]
        for s in range(len(seg_offsets) - 1):
            a, b = seg_offsets[s], seg_offsets[s + 1]
            if b > a:
                e_o = rel_fro(np.moveaxis(go[:, a:b], 1, -2), np.moveaxis(ro[:, a:b], 1, -2))
                assert e_o.max() <= o_tol, f"o error {e_o.max():.3e} (segment {s})"
    return float(e_s.max()), float(e_t.max())


def oracle_scan(w, want_o=False):
    return oracle.segment_scan(w["family"], w["k"], w["v"], w["alpha"], w["seg_offsets"],
                               beta=w["beta"], q=w["q"], want_o=want_o)


def test_tiny_dense_fp32_scan_compose_vs_sequential():
    """1 layer, 2 heads, d=32, two 64-token segments, fp32: scan both segments,
    compose, and compare with the straight recurrence over 128 tokens."""
    import linear_attention_state_gated_gb300 as hy
    w = wl.tiny_dense(seed=0)
    got = gpu_scan(w, want_o=True)
    ref = oracle_scan(w, want_o=True)
    check(DENSE, host(got), ref, TOL_F32, o_tol=TOL_F32, seg_offsets=w["seg_offsets"])
    comp = hy.compose("dense", got["lam"][:, 1], got["S"][:, 1], S_prev=got["S"][:, 0].contiguous(),
                      M=got["M"][:, 1].contiguous(), lam_prev=got["lam"][:, 0].contiguous(),
                      M_prev=got["M"][:, 0].contiguous())
    seq = oracle.sequential(DENSE, w["k"], w["v"], w["alpha"], w["beta"])
    assert rel_fro(to_host(comp["S"]), seq["S"]).max() <= TOL_F32
    assert t_err(DENSE, to_host(comp["lam"]), seq["lam"], to_host(comp["M"]), seq["M"]).max() <= TOL_F32


RAGGED = [1, 0, 63, 64, 65, 300, 129, 2]


@pytest.mark.parametrize("fam", [SCALAR, DIAG, DENSE], ids=["scalar", "diag", "dense"])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_scan_ragged_all_units(fam, d):
    """Ragged segments (empty, one token, tile edges, several tiles + tail), o_t."""
    if fam == DENSE:
        w = wl.dense_stack(lengths=RAGGED, n_layers=2, H=3, d=d, seed=7, with_q=True)
    else:
        w = wl.scalar_diag(fam, lengths=RAGGED, n_layers=2, H=3, d=d, seed=7, with_q=True)
    got = host(gpu_scan(w, want_o=True))
    ref = oracle_scan(w, want_o=True)
    check(fam, got, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])
    # the empty segment: lambda = 0, M = I, S = 0 exactly
    assert np.all(got["S"][:, 1] == 0) and np.all(got["lam"][:, 1] == 0)
    if fam == DENSE:
        assert np.array_equal(got["M"][:, 1], np.broadcast_to(np.eye(d), got["M"][:, 1].shape))


@pytest.mark.parametrize("fam", [SCALAR, DIAG, DENSE], ids=["scalar", "diag", "dense"])
def test_scan_ragged_state_only(fam):
    """d = 128, no o_t (the tensor-core path for scalar/diag): ragged segments
    including empty, one-token, chunk-edge and multi-chunk-plus-tail lengths."""
    lens = RAGGED + [31, 32, 33, 127, 128, 129, 1000]
    if fam == DENSE:
        w = wl.dense_stack(lengths=lens, n_layers=2, H=3, d=128, seed=8)
    else:
        w = wl.scalar_diag(fam, lengths=lens, n_layers=2, H=3, d=128, seed=8)
    got = host(gpu_scan(w))
    ref = oracle_scan(w)
    check(fam, got, ref, TOL_SCAN_BF16)
    assert np.all(got["S"][:, 1] == 0) and np.all(got["lam"][:, 1] == 0)


def test_scan_with_beta_and_mamba_like_gates():
    """Scalar gates that vary per token and a write scale beta (Mamba2-style),
    including strong decays; diagonal gates with beta."""
    import linear_attention_state_gated_gb300 as hy
    g = np.random.default_rng(12)
    lens = [300, 77, 0, 640]
    for fam in (SCALAR, DIAG):
        w = wl.scalar_diag(fam, lengths=lens, n_layers=1, H=4, d=128, seed=9)
        shape = w["alpha"].shape
        w["alpha"] = np.exp(-g.exponential(0.5, size=shape)).astype(np.float32)
        w["beta"] = g.uniform(0.0, 2.0, size=w["k"].shape[:3]).astype(np.float32)
        got = host(gpu_scan(w))
        ref = oracle_scan(w)
        check(fam, got, ref, TOL_SCAN_BF16)


@pytest.mark.parametrize("fam", [SCALAR, DIAG], ids=["scalar", "diag"])
def test_o_mamba_like_gates_and_beta(fam):
    """o_t on the tensor-core paths (chunks in order): per-token decays (per channel
    for the diagonal family), some strong, a write scale beta in [0, 2], segments
    across chunk edges and empty."""
    g = np.random.default_rng(13)
    lens = [300, 77, 0, 640, 64, 1, 65]
    w = wl.scalar_diag(fam, lengths=lens, n_layers=2, H=4, d=128, seed=10, with_q=True)
    w["alpha"] = np.exp(-g.exponential(0.5, size=w["alpha"].shape)).astype(np.float32)
    w["beta"] = g.uniform(0.0, 2.0, size=w["k"].shape[:3]).astype(np.float32)
    got = host(gpu_scan(w, want_o=True))
    ref = oracle_scan(w, want_o=True)
    e = check(fam, got, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])
    print(f"family {fam} o_t path: S error {e[0]:.3e}, T error {e[1]:.3e}")
    assert np.all(got["S"][:, 2] == 0) and np.all(got["lam"][:, 2] == 0)


def test_diag_o_steep_channels():
    """Diagonal gates with o_t where some channels decay by more than e^60 inside a
    chunk (those chunks take the exact Gram on CUDA cores and the end-of-chunk
    references): still equal to the oracle."""
    lens = [200, 130, 64]
    w = wl.scalar_diag(DIAG, lengths=lens, n_layers=1, H=2, d=128, seed=11, with_q=True)
    w["alpha"][:, 40:170, 0, :5] = np.float32(0.02)   # ln 0.02 = -3.9 a token
    got = host(gpu_scan(w, want_o=True))
    ref = oracle_scan(w, want_o=True)
    check(DIAG, got, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])


@pytest.mark.parametrize("case", ["no_decay", "all_steep"])
def test_diag_o_degenerate_gates(case):
    """Diagonal o_t path at alpha = 1 (plain linear attention) and with every chunk
    too steep for the factored Gram (the exact CUDA-core Gram everywhere)."""
    lens = [130, 64, 1, 0, 200]
    w = wl.scalar_diag(DIAG, lengths=lens, n_layers=1, H=2, d=128, seed=12, with_q=True)
    w["alpha"] = np.ones_like(w["alpha"]) if case == "no_decay" else np.full_like(w["alpha"], np.float32(0.02))
    got = host(gpu_scan(w, want_o=True))
    ref = oracle_scan(w, want_o=True)
    check(DIAG, got, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])


def test_diag_o_gla_full_size_sampled():
    """GLA-style gates, 8 segments x 2048 tokens x 32 heads with o_t (the benchmark's
    launch), sampled (segment, head) units against the straight recurrence."""
    w = wl.scalar_diag(DIAG, seg_len=2048, n_seg=8, with_q=True)
    got = host(gpu_scan(w, want_o=True))
    rs = np.random.default_rng(2049)
    for seg, h in [(0, 0), (7, 31)] + [tuple(x) for x in rs.integers([0, 0], [8, 32], size=(2, 2))]:
        a, b = w["seg_offsets"][seg], w["seg_offsets"][seg + 1]
        ref = oracle.sequential(DIAG, w["k"][:, a:b, h:h + 1], w["v"][:, a:b, h:h + 1],
                                w["alpha"][:, a:b, h:h + 1], q=w["q"][:, a:b, h:h + 1], want_o=True)
        sub = {"S": got["S"][:, seg, h:h + 1], "lam": got["lam"][:, seg, h:h + 1],
               "o": got["o"][:, a:b, h:h + 1]}
        check(DIAG, sub, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=[0, b - a])


def test_scalar_o_retnet_full_size_sampled():
    """RetNet gates, 8 segments x 2048 tokens x 32 heads with o_t (the benchmark's
    launch), sampled (segment, head) units against the straight recurrence."""
    w = wl.scalar_diag(SCALAR, seg_len=2048, n_seg=8, with_q=True)
    got = host(gpu_scan(w, want_o=True))
    rs = np.random.default_rng(2048)
    for seg, h in [(0, 0), (7, 31), (3, 26)] + [tuple(x) for x in rs.integers([0, 0], [8, 32], size=(2, 2))]:
        a, b = w["seg_offsets"][seg], w["seg_offsets"][seg + 1]
        ref = oracle.sequential(SCALAR, w["k"][:, a:b, h:h + 1], w["v"][:, a:b, h:h + 1],
                                w["alpha"][:, a:b, h:h + 1], q=w["q"][:, a:b, h:h + 1], want_o=True)
        sub = {"S": got["S"][:, seg, h:h + 1], "lam": got["lam"][:, seg, h:h + 1],
               "o": got["o"][:, a:b, h:h + 1]}
        check(SCALAR, sub, ref, TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=[0, b - a])


@pytest.mark.parametrize("fam", [SCALAR, DIAG], ids=["scalar", "diag"])
@pytest.mark.parametrize("L", [512, 2048, 8192])
def test_scalar_diag_full_size_sampled(fam, L):
    """32 heads, d=128, batch of 8 segments of L tokens (the benchmark's launch);
    sampled units at the batch's ends, in interior segments and at random."""
    w = wl.scalar_diag(fam, seg_len=L, n_seg=8)
    got = host(gpu_scan(w))
    rs = np.random.default_rng(L + fam)
    picks = [(0, 0), (7, 31), (3, 15), (4, 16)] + [tuple(x) for x in rs.integers([1, 0], [7, 32], size=(2, 2))]
    for seg, h in picks:
        a, b = w["seg_offsets"][seg], w["seg_offsets"][seg + 1]
        ref = oracle.sequential(fam, w["k"][:, a:b, h:h + 1], w["v"][:, a:b, h:h + 1],
                                w["alpha"][:, a:b, h:h + 1])
        sub = {"S": got["S"][:, seg, h:h + 1], "lam": got["lam"][:, seg, h:h + 1]}
        check(fam, sub, ref, TOL_SCAN_BF16)


@DENSE_FORMS
@pytest.mark.parametrize("L", [512, 2048])
def test_dense_full_stack_sampled(L, form):
    """30 layers x 32 heads x 128, one segment per layer (the benchmark's launch)."""
    w = wl.dense_stack(seg_len=L)
    got = host(gpu_scan(w, workspace=form))
    for l, h in [(0, 0), (29, 31), (13, 7)]:
        ref = oracle.sequential(DENSE, w["k"][l:l + 1, :, h:h + 1], w["v"][l:l + 1, :, h:h + 1],
                                w["alpha"][l:l + 1, :, h:h + 1], w["beta"][l:l + 1, :, h:h + 1])
        sub = {"S": got["S"][l:l + 1, 0, h:h + 1], "lam": got["lam"][l:l + 1, 0, h:h + 1],
               "M": got["M"][l:l + 1, 0, h:h + 1]}
        check(DENSE, sub, ref, TOL_SCAN_BF16)


@DENSE_FORMS
@pytest.mark.parametrize("L", [8192, 32768])
def test_dense_longest_segments_sampled(L, form):
    """The dense stack's longest segments (8192 and 32768 tokens: 128 / 512
    chunks, transitions far below fp32 range) on 2 layers x 32 heads (the
    benchmark's launch shape per layer); sampled heads against the oracle."""
    w = wl.dense_stack(seg_len=L, n_layers=2, H=32, d=128, seed=2)
    got = host(gpu_scan(w, workspace=form))
    for l, h in [(0, 0), (1, 31), (1, 9)]:
        ref = oracle.sequential(DENSE, w["k"][l:l + 1, :, h:h + 1], w["v"][l:l + 1, :, h:h + 1],
                                w["alpha"][l:l + 1, :, h:h + 1], w["beta"][l:l + 1, :, h:h + 1])
        sub = {"S": got["S"][l:l + 1, 0, h:h + 1], "lam": got["lam"][l:l + 1, 0, h:h + 1],
               "M": got["M"][l:l + 1, 0, h:h + 1]}
        check(DENSE, sub, ref, TOL_SCAN_BF16)


@DENSE_FORMS
def test_dense_long_segment_and_special_gates(form):
    """Gated delta rule on long segments (many chunks of transition renormalisation),
    beta = 0 (pure decay: S = 0, T = prod(alpha) I) and alpha = beta = 1 (plain delta rule)."""
    w = wl.dense_stack(lengths=[8192, 3000], n_layers=1, H=2, d=128, seed=13)
    check(DENSE, host(gpu_scan(w, workspace=form)), oracle_scan(w), TOL_SCAN_BF16)
    w0 = dict(w)
    w0["beta"] = np.zeros_like(w["beta"])
    got = host(gpu_scan(w0, workspace=form))
    ref = oracle_scan(w0)
    check(DENSE, got, ref, TOL_SCAN_BF16)
    assert np.all(got["S"] == 0)
    w1 = wl.dense_stack(lengths=[700, 129], n_layers=1, H=2, d=128, seed=14)
    w1["alpha"] = np.ones_like(w1["alpha"])
    w1["beta"] = np.ones_like(w1["beta"])
    check(DENSE, host(gpu_scan(w1, workspace=form)), oracle_scan(w1), TOL_SCAN_BF16)
    # strong decay: chunks whose total decay is below e^-40 alternate with mild ones
    w2 = wl.dense_stack(lengths=[1000, 333], n_layers=1, H=2, d=128, seed=15)
    t = np.arange(w2["alpha"].shape[1])
    w2["alpha"][:, (t // 64) % 3 == 1] = 0.3
    check(DENSE, host(gpu_scan(w2, workspace=form)), oracle_scan(w2), TOL_SCAN_BF16)


@DENSE_FORMS
def test_dense_o_long_and_special_gates(form):
    """o_t of the gated delta rule over several chunks (both forms): a long
    segment with a ragged tail, alpha = beta = 1, strong decay (chunks below
    e^-40 alternating with mild ones), and every chunk decaying by e^-38 (just
    above that bound: the largest b_t / b_C the output products take)."""
    w = wl.dense_stack(lengths=[2048 + 17, 700], n_layers=1, H=2, d=128, seed=16, with_q=True)
    got = host(gpu_scan(w, want_o=True, workspace=form))
    check(DENSE, got, oracle_scan(w, want_o=True), TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])
    w1 = dict(w)
    w1["alpha"] = np.ones_like(w["alpha"])
    w1["beta"] = np.ones_like(w["beta"])
    got = host(gpu_scan(w1, want_o=True, workspace=form))
    check(DENSE, got, oracle_scan(w1, want_o=True), TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])
    w2 = dict(w)
    w2["alpha"] = w["alpha"].copy()
    t = np.arange(w2["alpha"].shape[1])
    w2["alpha"][:, (t // 64) % 3 == 1] = 0.3
    got = host(gpu_scan(w2, want_o=True, workspace=form))
    check(DENSE, got, oracle_scan(w2, want_o=True), TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])
    w3 = dict(w)
    w3["alpha"] = np.full_like(w["alpha"], np.float32(0.55))   # 64 ln 0.55 = -38.3
    got = host(gpu_scan(w3, want_o=True, workspace=form))
    check(DENSE, got, oracle_scan(w3, want_o=True), TOL_SCAN_BF16, o_tol=TOL_O_BF16, seg_offsets=w["seg_offsets"])


@pytest.mark.parametrize("fam", [SCALAR, DIAG, DENSE], ids=["scalar", "diag", "dense"])
def test_segment_independence_bitwise(fam):
    """T_C and S(C|0) depend only on the segment's tokens: the same segment
    alone or inside a batch at another offset gives identical bits."""
    import torch
    lens = [200, 77, 130]
    mk = wl.dense_stack if fam == DENSE else (lambda **kw: wl.scalar_diag(fam, **kw))
    w = mk(lengths=lens, n_layers=1, H=2, d=128, seed=11)
    # the per-chain kernels (the balanced diagonal schedule splits chains
    # by the batch's total work, so its rounding depends on the batch)
    form = "auto" if fam == DENSE else None
    got = gpu_scan(w, workspace=form)
    a, b = w["seg_offsets"][1], w["seg_offsets"][2]
    alone = dict(w)
    for key in ("k", "v", "alpha", "beta"):
        if w[key] is not None:
            alone[key] = np.ascontiguousarray(w[key][:, a:b])
    alone["seg_offsets"] = np.array([0, b - a], dtype=np.int64)
    g1 = gpu_scan(alone, workspace=form)
    for key in g1:
        assert torch.equal(g1[key][:, 0], got[key][:, 1]), key


@DENSE_FORMS
def test_dense_ragged_batch_and_bad_offsets(form):
    """Several segments of ragged lengths in one call (chunk slots of neighbours
    interleave in the scratch), and a segment whose offsets leave [0, N]:
    reported through d_err, treated as empty (S = 0, T = I)."""
    import torch
    lens = [1, 63, 64, 65, 0, 300, 129]
    w = wl.dense_stack(lengths=lens, n_layers=2, H=3, d=128, seed=21)
    check(DENSE, host(gpu_scan(w, workspace=form)), oracle_scan(w), TOL_SCAN_BF16)
    w["seg_offsets"] = np.concatenate([w["seg_offsets"][:-1], [w["seg_offsets"][-1] + 5000]])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_scan(w, d_err=err, workspace=form)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    assert torch.all(got["S"][:, -1] == 0)
    assert torch.all(got["lam"][:, -1] == 0)
    assert torch.equal(got["M"][:, -1], torch.eye(128, device="cuda").expand_as(got["M"][:, -1]))


@pytest.mark.parametrize("fam", [DIAG], ids=["diag"])
def test_balanced_schedule_matches_per_chain(fam):
    """With scratch the diagonal scan splits all chains' chunks evenly
    over two CTAs per SM and folds the pieces of chains that straddle CTAs
    (S = T_late S_early + S_late).  It must match the oracle and the
    one-chain-per-CTA kernel (rounding only), for ragged, empty and
    one-token segments and for chains shorter and longer than a CTA's share."""
    lens = [5000, 0, 1, 64, 65, 3000, 129, 7000, 33]
    w = wl.scalar_diag(fam, lengths=lens, n_layers=2, H=7, d=128, seed=23)
    bal = host(gpu_scan(w))
    per = host(gpu_scan(w, workspace=None))
    check(fam, bal, oracle_scan(w), TOL_SCAN_BF16)
    # both forms sit ~1e-5 from the oracle; they round the weighted keys to bf16
    # hi + lo at different weights (relative to the piece's end, not the segment's)
    assert rel_fro(bal["S"], per["S"]).max() <= 1e-4
    assert np.abs(bal["lam"] - per["lam"]).max() <= 1e-5 * max(1.0, float(np.abs(per["lam"]).max()))
    assert np.all(bal["S"][:, 1] == 0) and np.all(bal["lam"][:, 1] == 0)
    # a chain longer than several CTAs' shares: one long segment, one head
    w1 = wl.scalar_diag(fam, lengths=[40000], n_layers=1, H=1, d=128, seed=24)
    check(fam, host(gpu_scan(w1)), oracle_scan(w1), TOL_SCAN_BF16)


@pytest.mark.parametrize("fam", [DIAG], ids=["diag"])
def test_balanced_schedule_bad_offsets(fam):
    """Offsets out of [0, N] on the balanced path: reported, segment empty."""
    import torch
    w = wl.scalar_diag(fam, lengths=[640, 64], n_layers=1, H=2, d=128, seed=3)
    w["seg_offsets"] = np.array([0, 640, 5000], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_scan(w, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    assert torch.all(got["S"][:, 1] == 0) and torch.all(got["lam"][:, 1] == 0)
    ref = oracle.sequential(fam, w["k"][:, :640], w["v"][:, :640], w["alpha"][:, :640])
    check(fam, {"S": host(got)["S"][:, 0], "lam": host(got)["lam"][:, 0]}, ref, TOL_SCAN_BF16)


def test_bad_offsets_flag_error_without_fault():
    """Offsets out of [0, N] are reported through d_err and the segment is treated as empty."""
    import torch
    w = wl.scalar_diag(SCALAR, lengths=[64, 64], n_layers=1, H=2, d=64, seed=3)
    w["seg_offsets"] = np.array([0, 64, 1000], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_scan(w, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    assert torch.all(got["S"][:, 1] == 0)


def test_long_mix_full_size_sampled():
    """131072-token prompt, 64 x 2048 segments (48 cached / 16 uncached), gated
    delta rule, 30 layers x 32 heads, in the benchmark's launches (cached segments
    one scan call each; the 16 uncached in one call over their (layer, segment)
    units, with o_t; chains with the layers as requests): the state folded over
    all 64 pairs equals the straight recurrence over the prompt (sampled layer and
    head, oracle), segment-boundary states equal the oracle's own composition of
    its pairs, and o_t of an uncached segment equals the oracle's isolated scan."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    n_seg, L, Lyr, H, d = 64, 2048, 30, 32, 128
    unc, cached, rows = wl.long_mix_layout(n_seg=n_seg, n_layers=Lyr)
    nu = len(unc)
    dev = torch.device("cuda")
    P = Lyr * n_seg
    pool_lam = torch.empty((P, 1, H), dtype=torch.float32, device=dev)
    pool_M = torch.empty((P, 1, H, d, d), dtype=torch.float32, device=dev)
    pool_S = torch.empty((P, 1, H, d, d), dtype=torch.float32, device=dev)
    offs1 = torch.tensor([0, L], dtype=torch.int64, device=dev)
    for c, s in enumerate(cached):
        w = wl.long_mix_segment_device(s, seg_len=L, n_layers=Lyr, H=H, d=d, with_q=False)
        r0 = Lyr * nu + c * Lyr
        out = {"lam": pool_lam[r0:r0 + Lyr].view(Lyr, 1, H), "M": pool_M[r0:r0 + Lyr].view(Lyr, 1, H, d, d),
               "S": pool_S[r0:r0 + Lyr].view(Lyr, 1, H, d, d)}
        hy.segment_scan(2, w["k"], w["v"], w["alpha"], offs1, beta=w["beta"], out=out)
        del w
    flat, offs = wl.long_mix_uncached_flat(unc, seg_len=L, n_layers=Lyr, H=H, d=d)
    out = {"lam": pool_lam[:Lyr * nu].view(1, Lyr * nu, H), "M": pool_M[:Lyr * nu].view(1, Lyr * nu, H, d, d),
           "S": pool_S[:Lyr * nu].view(1, Lyr * nu, H, d, d)}
    o = hy.segment_scan(2, flat["k"], flat["v"], flat["alpha"], to_dev(offs), beta=flat["beta"], q=flat["q"],
                        want_o=True, out=out)["o"]
    del flat
    # prefix chains of the sampled layer: request r folds segments 0..r in prompt order
    l, h = 17, 5
    clen = torch.arange(1, n_seg + 1, dtype=torch.int32, device=dev)
    idx = torch.from_numpy(np.ascontiguousarray(np.repeat(rows[l][None], n_seg, axis=0))).to(dev)
    S_pref = hy.compose_chain(2, clen, idx, pool_lam, pool_S, pool_M=pool_M)
    S_pref = to_host(S_pref[:, 0, h])
    # oracle: inputs of the sampled layer and head for every segment
    parts = [wl.long_mix_segment_device(s, seg_len=L, n_layers=Lyr, H=H, d=d, layers=[l], heads=[h])
             for s in range(n_seg)]
    cat = {key: torch.cat([p[key] for p in parts], dim=1).float().cpu().numpy().astype(np.float64)
           for key in ("k", "v", "alpha", "beta", "q")}
    seq = oracle.sequential(DENSE, cat["k"], cat["v"], cat["alpha"], cat["beta"])
    assert rel_fro(S_pref[-1], seq["S"][0, 0]) <= TOL_SCAN_BF16
    seg_pairs = oracle.segment_scan(DENSE, cat["k"], cat["v"], cat["alpha"],
                                    np.arange(n_seg + 1, dtype=np.int64) * L, beta=cat["beta"])
    pl = np.moveaxis(seg_pairs["lam"], 1, 0)
    pS = np.moveaxis(seg_pairs["S"], 1, 0)
    pM = np.moveaxis(seg_pairs["M"], 1, 0)
    for r in (0, 15, 31, 62):
        ref = oracle.compose_chain(DENSE, [r + 1], np.arange(n_seg, dtype=np.int32)[None], pl, pS, pool_M=pM)
        assert rel_fro(S_pref[r], ref[0, 0, 0]) <= TOL_SCAN_BF16, r
    # o_t of the first uncached segment from its own zero start (rows of (layer l, uncached 0))
    a0 = unc[0] * L
    iso = oracle.segment_scan(DENSE, cat["k"][:, a0:a0 + L], cat["v"][:, a0:a0 + L], cat["alpha"][:, a0:a0 + L],
                              [0, L], beta=cat["beta"][:, a0:a0 + L], q=cat["q"][:, a0:a0 + L], want_o=True)
    f0 = (l * nu + 0) * L
    go = to_host(o[0, f0:f0 + L, h])
    assert rel_fro(go, iso["o"][0, :, 0], axes=(-2, -1)) <= TOL_O_BF16
