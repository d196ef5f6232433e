"""GPU KDA-style family (T_t = diag(alpha_t)(I - beta_t k_t k_t^T)) against the
fp64 oracle: the token-by-token scan (T_C = exp(lambda) M, S(C|0), o_t), the
composition and chains of its pairs, and the seam-window advance."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, TOL_O_BF16, TOL_SCAN_BF16, rel_fro, t_err, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KDA = wl.KDA


def gpu_scan(w, bf16=True, want_o=False):
    import torch
    import linear_attention_state_gated_gb300 as hy
    dt = torch.bfloat16 if bf16 else torch.float32
    dev = lambda x: None if x is None else to_dev(x)   # noqa: E731
    return hy.segment_scan(KDA, dev(w["k"]).to(dt), dev(w["v"]).to(dt), dev(w["alpha"]),
                           to_dev(w["seg_offsets"]), beta=dev(w["beta"]),
                           q=dev(w["q"]).to(dt) if want_o else None, want_o=want_o)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bf16", [True, False], ids=["bf16", "f32"])
def test_kda_scan_matches_oracle(d, bf16):
    """Ragged segments (an empty one among them), outputs included."""
    lens = [70, 0, 129, 5, 200]
    w = wl.kda_stack(lengths=lens, n_layers=2, H=3, d=d, seed=80 + d, with_q=True)
    if not bf16:   # fp32 inputs off the bf16 grid
        g = np.random.default_rng(81)
        w = dict(w, k=w["k"] + np.float32(1e-3) * g.standard_normal(w["k"].shape).astype(np.float32),
                 v=w["v"] + np.float32(1e-3) * g.standard_normal(w["v"].shape).astype(np.float32))
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"], q=w["q"],
                              want_o=True)
    got = gpu_scan(w, bf16=bf16, want_o=True)
    tol = TOL_SCAN_BF16 if bf16 else TOL_F32
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= tol
    assert t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"]).max() <= tol
    mx = np.abs(to_host(got["M"])).max(axis=(-2, -1))
    assert np.all((mx >= 1) & (mx < 2))
    o_g = to_host(got["o"])
    for s in range(len(lens)):
        sl = slice(int(w["seg_offsets"][s]), int(w["seg_offsets"][s + 1]))
        if sl.stop > sl.start:
            e = rel_fro(np.moveaxis(o_g[:, sl], 1, 2), np.moveaxis(ref["o"][:, sl], 1, 2))
            assert e.max() <= (TOL_O_BF16 if bf16 else TOL_F32), s
    # the empty segment: lambda = 0, M = I, S = 0
    assert np.all(to_host(got["S"])[:, 1] == 0) and np.all(to_host(got["lam"])[:, 1] == 0)
    assert np.array_equal(to_host(got["M"])[0, 1, 0], np.eye(d))


def test_kda_one_gate_per_channel_matches_dense_family():
    """All channels gated alike: the GPU KDA scan equals the gated delta rule
    (the oracle's dense family on the same tokens)."""
    w = wl.kda_stack(lengths=[300, 77], n_layers=1, H=2, d=128, seed=85)
    one = np.ascontiguousarray(w["alpha"][..., 0])
    kda = gpu_scan(dict(w, alpha=np.ascontiguousarray(np.repeat(one[..., None], 128, axis=-1))))
    ref = oracle.segment_scan(wl.DENSE, w["k"], w["v"], one, w["seg_offsets"], beta=w["beta"])
    assert rel_fro(to_host(kda["S"]), ref["S"]).max() <= TOL_SCAN_BF16
    assert t_err(2, to_host(kda["lam"]), ref["lam"], to_host(kda["M"]), ref["M"]).max() <= TOL_SCAN_BF16


def kda_pool(lens, Lyr, H, d, seed):
    """Pool pairs (lambda, M, S) [P, Lyr, H, ...] from oracle scans of seeded KDA segments."""
    w = wl.kda_stack(lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    pool = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    mv = {k: np.ascontiguousarray(np.moveaxis(v, 1, 0)).astype(np.float32) for k, v in pool.items()}
    return w, mv


@pytest.mark.parametrize("d", [64, 128])
def test_kda_compose_and_operator(d):
    """S = T_C S_prev + S_C and T(C1.C2) = T(C2) T(C1) for KDA pairs (the dense
    kernels serve them: the pair is (lambda, M) either way)."""
    import linear_attention_state_gated_gb300 as hy
    _, pool = kda_pool([60, 90, 33, 120], 1, 3, d, seed=86 + d)
    c1 = {k: v[:2, 0] for k, v in pool.items()}
    c2 = {k: v[2:, 0] for k, v in pool.items()}
    ref = oracle.compose(KDA, c2["lam"], c2["S"], S_prev=c1["S"], M=c2["M"], lam_prev=c1["lam"], M_prev=c1["M"])
    got = hy.compose(KDA, to_dev(c2["lam"]), to_dev(c2["S"]), S_prev=to_dev(c1["S"]), M=to_dev(c2["M"]),
                     lam_prev=to_dev(c1["lam"]), M_prev=to_dev(c1["M"]))
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    assert t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"]).max() <= TOL_F32


def test_kda_chain_equals_straight_recurrence():
    """Chains of KDA pool pairs on the GPU against the oracle chain (fp32 tolerance)
    and against the straight fp64 recurrence over the concatenated tokens."""
    import linear_attention_state_gated_gb300 as hy
    lens = [40, 130, 7, 64]
    Lyr, H, d = 2, 2, 128
    w, pool = kda_pool(lens, Lyr, H, d, seed=88)
    idx = np.array([[3, 0, 2, 1], [1, 1, 0, 0]], np.int32)
    clen = np.array([4, 2], np.int32)
    ref = oracle.compose_chain(KDA, clen, idx, pool["lam"], pool["S"], pool_M=pool["M"])
    got = to_host(hy.compose_chain(KDA, to_dev(clen), to_dev(idx), to_dev(pool["lam"]), to_dev(pool["S"]),
                                   pool_M=to_dev(pool["M"])))
    assert rel_fro(got, ref).max() <= TOL_F32
    offs = w["seg_offsets"]
    for r in range(2):
        tok = np.concatenate([np.arange(offs[s], offs[s + 1]) for s in idx[r, :clen[r]]])
        seq = oracle.sequential(KDA, w["k"][:, tok], w["v"][:, tok], w["alpha"][:, tok], w["beta"][:, tok])
        assert rel_fro(got[r], seq["S"]).max() <= TOL_SCAN_BF16, r


def test_kda_seam_window():
    """hypic_seam_compose with KDA gates: the window from S_prev (outputs) then the
    cached rest, against the oracle and end to end against the straight recurrence."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    n_pre, w_len, n_body, H, d = 150, 8, 200, 3, 128
    w = wl.kda_stack(lengths=[n_pre, w_len, n_body], n_layers=1, H=H, d=d, seed=89, with_q=True)
    whole = oracle.sequential(KDA, w["k"], w["v"], w["alpha"], w["beta"], q=w["q"], want_o=True)
    pre, seam, body = slice(0, n_pre), slice(n_pre, n_pre + w_len), slice(n_pre + w_len, None)
    sub = lambda x, sl: np.ascontiguousarray(x[:, sl])   # noqa: E731
    bf = lambda x: to_dev(x).to(torch.bfloat16)          # noqa: E731
    S_prev = oracle.sequential(KDA, sub(w["k"], pre), sub(w["v"], pre), sub(w["alpha"], pre),
                               sub(w["beta"], pre))["S"].astype(np.float32)
    cached = oracle.sequential(KDA, sub(w["k"], body), sub(w["v"], body), sub(w["alpha"], body),
                               sub(w["beta"], body))
    lam, M, S_C = (cached[k].astype(np.float32) for k in ("lam", "M", "S"))
    args = [sub(w[k], seam) for k in ("k", "v", "alpha", "beta", "q")]
    ref = oracle.seam_compose(KDA, args[0], args[1], args[2], lam, S_C, S_prev=S_prev, M=M, beta=args[3],
                              q=args[4], want_o=True)
    got = hy.seam_compose(KDA, bf(args[0]), bf(args[1]), to_dev(args[2]), to_dev(lam), to_dev(S_C),
                          S_prev=to_dev(S_prev), M=to_dev(M), beta=to_dev(args[3]), q=bf(args[4]), want_o=True)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    o_err = rel_fro(np.moveaxis(to_host(got["o"]), 1, 2), np.moveaxis(ref["o"], 1, 2))
    assert o_err.max() <= TOL_O_BF16
    assert rel_fro(to_host(got["S"]), whole["S"]).max() <= TOL_SCAN_BF16
    o_whole = rel_fro(np.moveaxis(to_host(got["o"]), 1, 2), np.moveaxis(whole["o"][:, seam], 1, 2))
    assert o_whole.max() <= TOL_O_BF16


def test_kda_scan_full_size_sampled():
    """30 layers x 32 heads x 128, one 2048-token segment per layer (the dense stack's
    shape with per-channel gates); sampled (layer, head) chains checked one by one."""
    L, Lyr, H, d = 2048, 30, 32, 128
    w = wl.kda_stack(seg_len=L, n_layers=Lyr, H=H, d=d, seed=90)
    got = gpu_scan(w)
    S, lam, M = to_host(got["S"]), to_host(got["lam"]), to_host(got["M"])
    g = np.random.default_rng(91)
    for l, h in zip(g.integers(0, Lyr, 3), g.integers(0, H, 3)):
        one = lambda x: np.ascontiguousarray(x[l:l + 1, :, h:h + 1])   # noqa: E731
        ref = oracle.segment_scan(KDA, one(w["k"]), one(w["v"]), one(w["alpha"]), w["seg_offsets"],
                                  beta=one(w["beta"]))
        assert rel_fro(S[l:l + 1, :, h:h + 1], ref["S"]).max() <= TOL_SCAN_BF16, (l, h)
        assert t_err(2, lam[l:l + 1, :, h:h + 1], ref["lam"], M[l:l + 1, :, h:h + 1], ref["M"]).max() \
            <= TOL_SCAN_BF16, (l, h)


def test_kda_chunked_tensor_core_scan_ragged():
    """The chunked tensor-core form (d = 128, bf16, no o_t): ragged segments with
    an empty one, a one-token one and exact multiples of the chunk, against the oracle."""
    lens = [70, 0, 129, 1, 200, 64, 128]
    w = wl.kda_stack(lengths=lens, n_layers=2, H=3, d=128, seed=92)
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    got = gpu_scan(w)
    err_s = rel_fro(to_host(got["S"]), ref["S"])
    err_t = t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"])
    print(f"chunked KDA scan: S error max {err_s.max():.3e}, T error max {err_t.max():.3e}")
    assert err_s.max() <= TOL_SCAN_BF16 and err_t.max() <= TOL_SCAN_BF16
    mx = np.abs(to_host(got["M"])).max(axis=(-2, -1))
    assert np.all((mx >= 1) & (mx < 2))
    assert np.all(to_host(got["S"])[:, 1] == 0) and np.all(to_host(got["lam"])[:, 1] == 0)
    assert np.array_equal(to_host(got["M"])[0, 1, 0], np.eye(128))


def test_kda_chunked_scan_steep_channels():
    """Channels that decay by more than e^60 inside a chunk send that chunk's pair
    to the token-by-token kernel; mixed with ordinary chunks the result still
    matches the oracle."""
    lens = [150, 300, 40]
    w = wl.kda_stack(lengths=lens, n_layers=1, H=2, d=128, seed=93)
    alpha = w["alpha"].copy()
    # head 0: channels 0..7 forget fast (alpha = 0.05, ln = -3 a token) on tokens 100..229
    alpha[:, 100:230, 0, :8] = np.float32(0.05)
    w = dict(w, alpha=alpha)
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    got = gpu_scan(w)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_SCAN_BF16
    assert t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"]).max() <= TOL_SCAN_BF16


def test_kda_chunked_scan_uses_scratch_and_matches_token_kernel():
    """The workspace form takes the chunked path (positive scratch); without a
    workspace the token-by-token kernel runs; both agree within the scan tolerance."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    w = wl.kda_stack(lengths=[500, 260], n_layers=2, H=2, d=128, seed=94)
    assert hy.segment_scan_workspace_bytes(KDA, torch.bfloat16, 2, 2, 760, 2, 128, 128) > 0
    a = gpu_scan(w)
    dev = lambda x: to_dev(x)   # noqa: E731
    b = hy.segment_scan(KDA, dev(w["k"]).to(torch.bfloat16), dev(w["v"]).to(torch.bfloat16), dev(w["alpha"]),
                        to_dev(w["seg_offsets"]), beta=dev(w["beta"]), workspace=None)
    assert rel_fro(to_host(a["S"]), to_host(b["S"])).max() <= TOL_SCAN_BF16
    assert t_err(2, to_host(a["lam"]), to_host(b["lam"]), to_host(a["M"]), to_host(b["M"])).max() <= TOL_SCAN_BF16


@pytest.mark.parametrize("case", ["no_decay", "no_write", "all_steep"])
def test_kda_chunked_scan_degenerate_gates(case):
    """The tensor-core KDA scan at its degenerate gates: alpha = 1 (the delta rule
    without decay), beta = 0 (pure per-channel decay: S = 0, T diagonal) and every
    chunk too steep for the factored Gram (all pairs token by token)."""
    lens = [130, 64, 1]
    w = wl.kda_stack(lengths=lens, n_layers=1, H=2, d=128, seed=95)
    if case == "no_decay":
        w = dict(w, alpha=np.ones_like(w["alpha"]))
    elif case == "no_write":
        w = dict(w, beta=np.zeros_like(w["beta"]))
    else:
        w = dict(w, alpha=np.full_like(w["alpha"], np.float32(0.01)))
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    got = gpu_scan(w)
    if case == "no_write":
        assert np.all(to_host(got["S"]) == 0)
    else:
        assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_SCAN_BF16
    assert t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"]).max() <= TOL_SCAN_BF16


def test_kda_chunked_scan_bad_offsets_flag_error():
    """A segment whose offsets leave [0, N]: reported through d_err (no fault) and
    treated as empty (S = 0, T = I) on the tensor-core path; the others unchanged."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    lens = [100, 64, 70]
    w = wl.kda_stack(lengths=lens, n_layers=1, H=2, d=128, seed=96)
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    offs = np.concatenate([w["seg_offsets"][:-1], [w["seg_offsets"][-1] + 5000]])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bf = lambda x: to_dev(x).to(torch.bfloat16)   # noqa: E731
    got = hy.segment_scan(KDA, bf(w["k"]), bf(w["v"]), to_dev(w["alpha"]), to_dev(offs), beta=to_dev(w["beta"]),
                          d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    S, lam, M = to_host(got["S"]), to_host(got["lam"]), to_host(got["M"])
    assert np.all(S[:, -1] == 0) and np.all(lam[:, -1] == 0)
    assert np.array_equal(M[0, -1, 0], np.eye(128))
    assert rel_fro(S[:, :2], ref["S"][:, :2]).max() <= TOL_SCAN_BF16


def test_kda_chunked_scan_many_ragged_segments():
    """Forty ragged segments (empty ones, one-token ones, chunk multiples) in one
    call: every chunk slot mapping of the tensor-core path against the oracle."""
    g = np.random.default_rng(97)
    lens = [int(x) for x in g.integers(0, 300, size=40)]
    lens[3], lens[7], lens[11], lens[20] = 0, 1, 64, 128
    w = wl.kda_stack(lengths=lens, n_layers=2, H=2, d=128, seed=97)
    ref = oracle.segment_scan(KDA, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    got = gpu_scan(w)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_SCAN_BF16
    assert t_err(2, to_host(got["lam"]), ref["lam"], to_host(got["M"]), ref["M"]).max() <= TOL_SCAN_BF16
    assert np.all(to_host(got["S"])[:, 3] == 0)
