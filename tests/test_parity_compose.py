"""GPU composition (single step and chained) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, TOL_SCAN_BF16, rel_fro, t_err, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCALAR, DIAG, DENSE = wl.SCALAR, wl.DIAG, wl.DENSE
FAMS = [SCALAR, DIAG, DENSE]
IDS = ["scalar", "diag", "dense"]


def random_pairs(fam, n, H, dk, dv, seed):
    g = np.random.default_rng(seed)
    lam = -g.uniform(0, 30, size=(n, H, dk) if fam == DIAG else (n, H)).astype(np.float32)
    S = g.standard_normal((n, H, dk, dv)).astype(np.float32)
    M = None
    if fam == DENSE:
        M = (g.standard_normal((n, H, dk, dk)) / np.sqrt(dk)).astype(np.float32)
        M /= np.abs(M).max(axis=(-2, -1), keepdims=True)
        M *= np.float32(1.5)
    return lam, S, M


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (32, 128)])
def test_compose_step(fam, dk, dv):
    import linear_attention_state_gated_gb300 as hy
    n, H = 5, 3
    lam, S_C, M = random_pairs(fam, n, H, dk, dv, seed=dk + dv + fam)
    lam_p, S_p, M_p = random_pairs(fam, n, H, dk, dv, seed=1 + dk + dv + fam)
    ref = oracle.compose(fam, lam, S_C, S_prev=S_p, M=M, lam_prev=lam_p, M_prev=M_p)
    got = hy.compose(fam, to_dev(lam), to_dev(S_C), S_prev=to_dev(S_p), M=to_dev(M),
                     lam_prev=to_dev(lam_p), M_prev=to_dev(M_p))
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    assert t_err(fam, to_host(got["lam"]), ref["lam"],
                 to_host(got["M"]) if fam == DENSE else None, ref.get("M")).max() <= TOL_F32
    if fam == DENSE:
        mx = np.abs(to_host(got["M"])).max(axis=(-2, -1))
        assert np.all((mx >= 1) & (mx < 2))
    # in place (S_out is S_prev) and without a previous state
    Sp_dev = to_dev(S_p)
    hy.compose(fam, to_dev(lam), to_dev(S_C), S_prev=Sp_dev, M=to_dev(M), S_out=Sp_dev)
    assert rel_fro(to_host(Sp_dev), ref["S"]).max() <= TOL_F32
    z = hy.compose(fam, to_dev(lam), to_dev(S_C), M=to_dev(M))
    assert np.array_equal(to_host(z["S"]), S_C.astype(np.float64))


def scanned_pool(fam, lens, Lyr, H, d, seed):
    """Pool pairs from oracle scans of seeded segments (bf16-valued inputs)."""
    if fam == DENSE:
        w = wl.dense_stack(lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    else:
        w = wl.scalar_diag(fam, lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    pool = oracle.segment_scan(fam, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    mv = {k: np.ascontiguousarray(np.moveaxis(v, 1, 0)).astype(np.float32) for k, v in pool.items()}
    return w, mv


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
def test_chain_matches_oracle_chain_and_sequential(fam):
    """Chains over oracle-scanned pool entries: equal to the oracle's chain (fp32
    tolerance) and to the straight recurrence over the concatenated tokens."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    lens = [40, 130, 7, 64, 99]
    Lyr, H, d = 2, 2, 128
    w, pool = scanned_pool(fam, lens, Lyr, H, d, seed=21 + fam)
    idx = np.array([[3, 0, 4, 1, 2], [2, 2, 1, 0, 0], [4, 3, 0, 0, 0], [0, 0, 0, 0, 0]], np.int32)
    clen = np.array([5, 3, 2, 0], np.int32)
    g = np.random.default_rng(5)
    S_init = g.standard_normal((4, Lyr, H, d, d)).astype(np.float32)
    ref = oracle.compose_chain(fam, clen, idx, pool["lam"], pool["S"], pool_M=pool.get("M"),
                               S_init=S_init)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = to_host(hy.compose_chain(fam, to_dev(clen), to_dev(idx), to_dev(pool["lam"]),
                                   to_dev(pool["S"]), pool_M=to_dev(pool.get("M")),
                                   S_init=to_dev(S_init), d_err=err))
    assert int(err.item()) == 0
    assert rel_fro(got, ref).max() <= TOL_F32
    # zero start vs the straight recurrence (scan tolerance: pool pairs came from the oracle)
    got0 = to_host(hy.compose_chain(fam, to_dev(clen[:3]), to_dev(idx[:3]), to_dev(pool["lam"]),
                                    to_dev(pool["S"]), pool_M=to_dev(pool.get("M"))))
    offs = w["seg_offsets"]
    for r in range(3):
        tok = np.concatenate([np.arange(offs[s], offs[s + 1]) for s in idx[r, :clen[r]]])
        seq = oracle.sequential(fam, w["k"][:, tok], w["v"][:, tok], w["alpha"][:, tok],
                                None if w["beta"] is None else w["beta"][:, tok])
        assert rel_fro(got0[r], seq["S"]).max() <= TOL_SCAN_BF16


def test_chain_bad_index_is_flagged_not_faulted():
    import torch
    import linear_attention_state_gated_gb300 as hy
    P, Lyr, H, d = 3, 1, 2, 64
    lam, S, _ = random_pairs(SCALAR, P * Lyr, H, d, d, seed=3)
    lam = lam.reshape(P, Lyr, H)
    S = S.reshape(P, Lyr, H, d, d)
    idx = np.array([[0, 7, 1]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hy.compose_chain(SCALAR, to_dev(np.array([3], np.int32)), to_dev(idx), to_dev(lam), to_dev(S),
                     d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    err.zero_()
    hy.compose_chain(SCALAR, to_dev(np.array([9], np.int32)), to_dev(idx), to_dev(lam), to_dev(S),
                     d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5


@pytest.mark.parametrize("fam", [SCALAR, DIAG], ids=["scalar", "diag"])
def test_rag_chain_full_size_sampled(fam):
    """Pool of 200 cached pairs x 30 layers x 32 heads x 128^2; 64 requests x 20
    Zipf(1.1) segments in random order (the benchmark's launch); sampled units."""
    import linear_attention_state_gated_gb300 as hy
    pool = wl.rag_pool(fam)
    clen, idx = wl.rag_requests()
    got = hy.compose_chain(fam, to_dev(clen), to_dev(idx), to_dev(pool["lam"]), to_dev(pool["S"]))
    rs = np.random.default_rng(17)
    for r, l, h in [(0, 0, 0), (63, 29, 31)] + [tuple(x) for x in rs.integers([0, 0, 0], [64, 30, 32], size=(2, 3))]:
        sub_lam = np.ascontiguousarray(pool["lam"][:, l:l + 1, h:h + 1])
        sub_S = np.ascontiguousarray(pool["S"][:, l:l + 1, h:h + 1])
        ref = oracle.compose_chain(fam, clen[r:r + 1], idx[r:r + 1], sub_lam, sub_S)
        g = to_host(got[r, l, h])
        assert rel_fro(g, ref[0, 0, 0]) <= TOL_F32


@pytest.mark.parametrize("fam,dk,dv", [(DIAG, 64, 128), (SCALAR, 128, 64), (DENSE, 128, 128), (DENSE, 64, 64)])
def test_chain_shapes_and_long_chains(fam, dk, dv):
    """Random pool pairs, chains of 0..40 steps with repeats, other head sizes."""
    import linear_attention_state_gated_gb300 as hy
    P, Lyr, H = 9, 2, 3
    lam, S, M = random_pairs(fam, P * Lyr, H, dk, dv, seed=dk + dv + 7 * fam)
    lam = lam.reshape((P, Lyr) + lam.shape[1:])
    S = S.reshape(P, Lyr, H, dk, dv)
    M = None if M is None else M.reshape(P, Lyr, H, dk, dk)
    lam = np.minimum(lam, -0.05).astype(np.float32)        # decaying operators keep the state bounded
    g = np.random.default_rng(31)
    clen = np.array([40, 0, 1, 17], np.int32)
    idx = g.integers(0, P, size=(4, 40)).astype(np.int32)
    ref = oracle.compose_chain(fam, clen, idx, lam, S, pool_M=M)
    got = to_host(hy.compose_chain(fam, to_dev(clen), to_dev(idx), to_dev(lam), to_dev(S), pool_M=to_dev(M)))
    assert rel_fro(got, ref).max() <= TOL_F32
    assert np.all(got[1] == 0)


def test_dense_chain_bad_index_is_flagged_not_faulted():
    import torch
    import linear_attention_state_gated_gb300 as hy
    P, Lyr, H, d = 3, 1, 2, 128
    lam, S, M = random_pairs(DENSE, P * Lyr, H, d, d, seed=5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hy.compose_chain(DENSE, to_dev(np.array([3], np.int32)), to_dev(np.array([[0, 7, -1]], np.int32)),
                     to_dev(lam.reshape(P, Lyr, H)), to_dev(S.reshape(P, Lyr, H, d, d)),
                     pool_M=to_dev(M.reshape(P, Lyr, H, d, d)), d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
