"""GPU composed prefixes (hypic_compose_prefix): the cached pair (T, S) of an
ordered group of pool entries, against the fp64 oracle, and its reuse as a pool
entry in later chains."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, rel_fro, t_err, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FAMS = [wl.SCALAR, wl.DIAG, wl.DENSE, wl.KDA]
IDS = ["scalar", "diag", "dense", "kda"]
WITH_M = (wl.DENSE, wl.KDA)


def scanned_pool(fam, lens, Lyr, H, d, seed):
    if fam == wl.DENSE:
        w = wl.dense_stack(lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    elif fam == wl.KDA:
        w = wl.kda_stack(lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    else:
        w = wl.scalar_diag(fam, lengths=lens, n_layers=Lyr, H=H, d=d, seed=seed)
    pool = oracle.segment_scan(fam, w["k"], w["v"], w["alpha"], w["seg_offsets"], beta=w["beta"])
    return {k: np.ascontiguousarray(np.moveaxis(v, 1, 0)).astype(np.float32) for k, v in pool.items()}


def t_fam(fam):   # operator error metric: the dense one for every family with M
    return 2 if fam in WITH_M else fam


def check(fam, got, ref):
    assert rel_fro(to_host(got["S"]), ref["S"]).max() <= TOL_F32
    M_g = to_host(got["M"]) if fam in WITH_M else None
    assert t_err(t_fam(fam), to_host(got["lam"]), ref["lam"], M_g, ref.get("M")).max() <= TOL_F32
    if fam in WITH_M:
        mx = np.abs(M_g).max(axis=(-2, -1))
        assert np.all((mx >= 1) & (mx < 2))


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
@pytest.mark.parametrize("d", [128, 64])
def test_prefix_matches_oracle(fam, d):
    """Groups of several lengths (one empty, one with a repeated entry), d = 128 on
    the tensor-core chain, d = 64 on the CUDA-core one."""
    import linear_attention_state_gated_gb300 as hy
    lens = [50, 120, 9, 64, 33, 80]
    Lyr, H = 2, 2
    pool = scanned_pool(fam, lens, Lyr, H, d, seed=100 + fam + d)
    idx = np.array([[3, 0, 5, 1, 2, 4, 3, 1, 0], [2, 2, 1, 0, 0, 0, 0, 0, 0], [0] * 9, [5, 4, 3, 2, 1, 0, 5, 4, 3]],
                   np.int32)
    clen = np.array([9, 3, 0, 9], np.int32)
    ref = oracle.compose_prefix(fam, clen, idx, pool["lam"], pool["S"], pool_M=pool.get("M"))
    got = hy.compose_prefix(fam, to_dev(clen), to_dev(idx), to_dev(pool["lam"]), to_dev(pool["S"]),
                            pool_M=to_dev(pool.get("M")))
    check(fam, got, ref)
    # the empty group: lambda = 0, M = I, S = 0
    assert np.all(to_host(got["S"])[2] == 0) and np.all(to_host(got["lam"])[2] == 0)
    if fam in WITH_M:
        assert np.array_equal(to_host(got["M"])[2, 0, 0], np.eye(d))


@pytest.mark.parametrize("d", [128, 64])
def test_prefix_long_group_with_growing_operators(d):
    """Pool operators drawn with entries ~N(0, 1) (products grow by orders of
    magnitude a step): 40-entry groups exercise the power-of-two rescaling."""
    import linear_attention_state_gated_gb300 as hy
    g = np.random.default_rng(110 + d)
    P, Lyr, H = 12, 1, 3
    lam = -g.uniform(0, 5, size=(P, Lyr, H)).astype(np.float32)
    M = g.standard_normal((P, Lyr, H, d, d)).astype(np.float32)
    S = g.standard_normal((P, Lyr, H, d, d)).astype(np.float32)
    idx = g.integers(0, P, size=(2, 40)).astype(np.int32)
    clen = np.array([40, 37], np.int32)
    ref = oracle.compose_prefix(wl.DENSE, clen, idx, lam, S, pool_M=M)
    got = hy.compose_prefix(wl.DENSE, to_dev(clen), to_dev(idx), to_dev(lam), to_dev(S), pool_M=to_dev(M))
    M_g = to_host(got["M"])
    err = t_err(2, to_host(got["lam"]), ref["lam"], M_g, ref["M"])
    print(f"d={d} operator chain error max {err.max():.3e} mean {err.mean():.3e}")
    assert err.max() <= TOL_F32
    mx = np.abs(M_g).max(axis=(-2, -1))
    assert np.all((mx >= 1) & (mx < 2))


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
def test_prefix_reused_as_pool_entry(fam):
    """A cached prefix stands in for its members: chain [prefix, x] equals chain
    [members..., x] (GPU both ways)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    lens = [70, 20, 45, 90]
    Lyr, H, d = 2, 2, 128
    pool = scanned_pool(fam, lens, Lyr, H, d, seed=120 + fam)
    grp = np.array([[2, 0, 3]], np.int32)
    pre = hy.compose_prefix(fam, to_dev(np.array([3], np.int32)), to_dev(grp), to_dev(pool["lam"]),
                            to_dev(pool["S"]), pool_M=to_dev(pool.get("M")))
    ext = lambda key: torch.cat([to_dev(pool[key]), pre[key]], dim=0).contiguous()   # noqa: E731
    P = len(lens)
    a = hy.compose_chain(fam, to_dev(np.array([2], np.int32)), to_dev(np.array([[P, 1]], np.int32)), ext("lam"),
                         ext("S"), pool_M=ext("M") if fam in WITH_M else None)
    b = hy.compose_chain(fam, to_dev(np.array([4], np.int32)), to_dev(np.array([[2, 0, 3, 1]], np.int32)),
                         to_dev(pool["lam"]), to_dev(pool["S"]), pool_M=to_dev(pool.get("M")))
    assert rel_fro(to_host(a), to_host(b)).max() <= 1e-4
