"""GPU seam-window advance + composition (hypic_seam_compose) against the fp64
oracle: the window's recurrence from a nonzero state, its per-token outputs,
and the composition of the cached rest of the segment."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, TOL_O_BF16, TOL_SCAN_BF16, rel_fro, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCALAR, DIAG, DENSE = wl.SCALAR, wl.DIAG, wl.DENSE
FAMS = [SCALAR, DIAG, DENSE]
IDS = ["scalar", "diag", "dense"]


def seam_tokens(fam, n, w, H, dk, dv, seed, bf16=True):
    """Seam-window inputs [n, w, H, .]: k unit rows, q, v ~ N(0,1) (bf16-valued when
    bf16), alpha by family, beta = sigmoid(N(0,1))."""
    g = np.random.default_rng(seed)
    k = g.standard_normal((n, w, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = g.standard_normal((n, w, H, dk))
    v = g.standard_normal((n, w, H, dv))
    if bf16:
        k, q, v = wl.bf16_round(k), wl.bf16_round(q), wl.bf16_round(v)
    ash = (n, w, H, dk) if fam == DIAG else (n, w, H)
    alpha = g.uniform(0.85, 1.0, size=ash).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-g.standard_normal((n, w, H))))).astype(np.float32)
    return (k.astype(np.float32), v.astype(np.float32), q.astype(np.float32), alpha, beta)


def body_pair(fam, n, H, dk, dv, seed):
    g = np.random.default_rng(seed)
    lam = -g.uniform(0, 3, size=(n, H, dk) if fam == DIAG else (n, H)).astype(np.float32)
    S_C = g.standard_normal((n, H, dk, dv)).astype(np.float32)
    M = None
    if fam == DENSE:
        M = (g.standard_normal((n, H, dk, dk)) / np.sqrt(dk)).astype(np.float32)
        M /= np.abs(M).max(axis=(-2, -1), keepdims=True)
        M *= np.float32(1.5)
    S_prev = g.standard_normal((n, H, dk, dv)).astype(np.float32)
    return lam, S_C, M, S_prev


def o_err(got, ref):
    """Relative Frobenius error of the window's outputs per (item, head)."""
    return rel_fro(np.moveaxis(got, 1, 2), np.moveaxis(ref, 1, 2))


def run(fam, k, v, q, alpha, beta, lam, S_C, M, S_prev, bf16, **kw):
    import torch
    import linear_attention_state_gated_gb300 as hy
    dt = torch.bfloat16 if bf16 else torch.float32
    return hy.seam_compose(fam, to_dev(k).to(dt), to_dev(v).to(dt), to_dev(alpha), to_dev(lam), to_dev(S_C),
                           S_prev=to_dev(S_prev), M=to_dev(M), beta=to_dev(beta),
                           q=None if q is None else to_dev(q).to(dt), want_o=q is not None, **kw)


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
@pytest.mark.parametrize("bf16", [True, False], ids=["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (32, 128)])
def test_seam_compose_matches_oracle(fam, bf16, dk, dv):
    n, w, H = 5, 8, 3
    k, v, q, alpha, beta = seam_tokens(fam, n, w, H, dk, dv, seed=dk + 3 * dv + fam, bf16=bf16)
    lam, S_C, M, S_prev = body_pair(fam, n, H, dk, dv, seed=7 + dk + dv + fam)
    ref = oracle.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M, beta=beta, q=q, want_o=True)
    got = run(fam, k, v, q, alpha, beta, lam, S_C, M, S_prev, bf16)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    assert o_err(to_host(got["o"]), ref["o"]).max() <= (TOL_O_BF16 if bf16 else TOL_F32)


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
def test_seam_in_place_ragged_window_and_edges(fam):
    import torch
    import linear_attention_state_gated_gb300 as hy
    n, H, d = 4, 2, 128
    lam, S_C, M, S_prev = body_pair(fam, n, H, d, d, seed=40 + fam)
    for w in (1, 13, 17):   # one token, a block and a tail, two blocks and one token
        k, v, q, alpha, beta = seam_tokens(fam, n, w, H, d, d, seed=41 + w + fam)
        ref = oracle.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M, beta=beta, q=q,
                                  want_o=True)
        Sp = to_dev(S_prev)
        got = run(fam, k, v, q, alpha, beta, lam, S_C, M, None, True, S_out=Sp)
        # S_prev=None above: the window starts from zero; now in place from S_prev
        ref0 = oracle.seam_compose(fam, k, v, alpha, lam, S_C, M=M, beta=beta, q=q, want_o=True)
        assert rel_fro(to_host(got["S"]), ref0["S"]).max() <= TOL_F32
        assert o_err(to_host(got["o"]), ref0["o"]).max() <= TOL_O_BF16
        Sp = to_dev(S_prev)
        got = hy.seam_compose(fam, to_dev(k).to(torch.bfloat16), to_dev(v).to(torch.bfloat16),
                              to_dev(alpha), to_dev(lam), to_dev(S_C), S_prev=Sp, M=to_dev(M),
                              beta=to_dev(beta), q=to_dev(q).to(torch.bfloat16), want_o=True, S_out=Sp)
        assert got["S"].data_ptr() == Sp.data_ptr()
        assert rel_fro(to_host(Sp), ref["S"]).max() <= TOL_F32
        assert o_err(to_host(got["o"]), ref["o"]).max() <= TOL_O_BF16
    # no window: the plain composition; beta absent (=> 1) and no outputs asked
    k, v, q, alpha, beta = seam_tokens(fam, n, 0, H, d, d, seed=49 + fam)
    got = run(fam, k, v, None, alpha, None, lam, S_C, M, S_prev, True)
    ref = oracle.compose(fam, lam, S_C, S_prev=S_prev, M=M)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    k, v, q, alpha, beta = seam_tokens(fam, n, 8, H, d, d, seed=50 + fam)
    got = run(fam, k, v, None, alpha, None, lam, S_C, M, S_prev, True)
    ref = oracle.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M)
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
def test_reuse_with_seam_window_equals_straight_prefill(fam):
    """The reuse path end to end on the GPU: the prefix scanned, the segment's
    rest scanned alone into its cached pair, then the seam window advanced from
    the prefix state and the pair composed -- against the straight fp64
    recurrence over prefix + segment (state, and the seam tokens' outputs)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    n_pre, w, n_body, H, d = 200, 8, 300, 4, 128
    lens = [n_pre, w, n_body]
    if fam == DENSE:
        wk = wl.dense_stack(lengths=lens, n_layers=1, H=H, d=d, seed=60, with_q=True)
    else:
        wk = wl.scalar_diag(fam, lengths=lens, n_layers=1, H=H, d=d, seed=60 + fam, with_q=True)
    k, v, q, alpha, beta = wk["k"], wk["v"], wk["q"], wk["alpha"], wk["beta"]
    whole = oracle.sequential(fam, k, v, alpha, beta, q=q, want_o=True)
    dev = lambda x: None if x is None else to_dev(x)
    bf = lambda x: to_dev(x).to(torch.bfloat16)
    pre, seam, body = slice(0, n_pre), slice(n_pre, n_pre + w), slice(n_pre + w, n_pre + w + n_body)
    sub = lambda x, sl: None if x is None else np.ascontiguousarray(x[:, sl])
    p = hy.segment_scan(fam, bf(sub(k, pre)), bf(sub(v, pre)), dev(sub(alpha, pre)),
                        to_dev(np.array([0, n_pre], np.int64)), beta=dev(sub(beta, pre)))
    c = hy.segment_scan(fam, bf(sub(k, body)), bf(sub(v, body)), dev(sub(alpha, body)),
                        to_dev(np.array([0, n_body], np.int64)), beta=dev(sub(beta, body)))
    # seam window as [n = 1, w, H, .]
    got = hy.seam_compose(fam, bf(sub(k, seam)), bf(sub(v, seam)), dev(sub(alpha, seam)), c["lam"][0],
                          c["S"][0], S_prev=p["S"][0], M=c["M"][0] if fam == DENSE else None,
                          beta=dev(sub(beta, seam)), q=bf(sub(q, seam)), want_o=True)
    assert rel_fro(to_host(got["S"]), whole["S"]).max() <= TOL_SCAN_BF16
    o_ref = whole["o"][:, seam]
    assert o_err(to_host(got["o"]), o_ref).max() <= TOL_O_BF16


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
def test_seam_full_size_sampled(fam):
    """The benchmark's launch: 1920 items x 32 heads x 128 x 128, w = 8 (inputs
    drawn on the device); sampled (item, head) pairs checked one by one."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    n, w, H, d = 1920, 8, 32, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(70 + fam)
    f = dict(device="cuda", generator=gen)
    k = torch.nn.functional.normalize(torch.randn((n, w, H, d), **f), dim=-1).to(torch.bfloat16)
    q = torch.randn((n, w, H, d), **f).to(torch.bfloat16)
    v = torch.randn((n, w, H, d), **f).to(torch.bfloat16)
    alpha = 0.85 + 0.15 * torch.rand((n, w, H, d) if fam == DIAG else (n, w, H), **f)
    beta = torch.sigmoid(torch.randn((n, w, H), **f))
    lam = -3 * torch.rand((n, H, d) if fam == DIAG else (n, H), **f)
    S_C = torch.randn((n, H, d, d), **f)
    S_prev = torch.randn((n, H, d, d), **f)
    M = torch.randn((n, H, d, d), **f) * 0.1 if fam == DENSE else None
    got = hy.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M, beta=beta, q=q, want_o=True)
    torch.cuda.synchronize()
    g = np.random.default_rng(71)
    for i, h in zip(g.integers(0, n, 12), g.integers(0, H, 12)):
        sl = lambda x: None if x is None else to_host(x[i:i + 1, :, h:h + 1].float())
        sh = lambda x: None if x is None else to_host(x[i:i + 1, h:h + 1].float())
        ref = oracle.seam_compose(fam, sl(k), sl(v), sl(alpha), sh(lam), sh(S_C), S_prev=sh(S_prev),
                                  M=sh(M), beta=sl(beta), q=sl(q), want_o=True)
        assert rel_fro(to_host(got["S"][i:i + 1, h:h + 1]), ref["S"]).max() <= TOL_F32, (i, h)
        assert o_err(to_host(got["o"][i:i + 1, :, h:h + 1].float()), ref["o"]).max() <= TOL_O_BF16, (i, h)
