"""Two-level tree composition (hypic_compose_chain_ws): when few (request, layer,
head) units carry long chains, groups of consecutive pool entries are first folded
in parallel into cached pairs (T(C1.C2) = T(C2) T(C1), xix.ai/fr linear-layer
paragraph), then each chain folds its groups' pairs in order.  Checked against the
fp64 oracle's chain and against the plain GPU chain, every family, on the
tensor-core (d = 128) and CUDA-core (d = 64) paths, with ragged chain lengths,
repeated entries and a previous state."""
import numpy as np
import pytest

import oracle
from helpers import TOL_F32, rel_fro, to_dev, to_host
from linear_attention_state_gated_gb300 import workloads as wl
from test_parity_prefix import WITH_M, scanned_pool

pytestmark = pytest.mark.gpu

FAMS = [wl.SCALAR, wl.DIAG, wl.DENSE, wl.KDA]
IDS = ["scalar", "diag", "dense", "kda"]


@pytest.mark.parametrize("fam", FAMS, ids=IDS)
@pytest.mark.parametrize("d", [128, 64])
def test_tree_matches_oracle_and_plain_chain(fam, d):
    import torch
    import linear_attention_state_gated_gb300 as hy
    g = np.random.default_rng(200 + fam + d)
    lens = [int(x) for x in g.integers(4, 40, size=24)]
    Lyr, H = 1, 3
    pool = scanned_pool(fam, lens, Lyr, H, d, seed=210 + fam + d)
    P = len(lens)
    mc = 64
    clen = np.array([64, 37, 0, 4, 9], np.int32)            # full, ragged, empty, one group, one entry past it
    idx = g.integers(0, P, size=(len(clen), mc)).astype(np.int32)
    S_init = g.standard_normal((len(clen), Lyr, H, d, d)).astype(np.float32) * np.float32(0.1)
    need = hy.compose_chain_workspace_bytes(fam, len(clen), Lyr, H, d, d, mc)
    assert need > 0                                           # 15 units, 64-entry chains: the tree
    pl, pS, pM = to_dev(pool["lam"]), to_dev(pool["S"]), to_dev(pool.get("M"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = hy.compose_chain(fam, to_dev(clen), to_dev(idx), pl, pS, pool_M=pM, S_init=to_dev(S_init),
                           workspace="auto", d_err=err)
    plain = hy.compose_chain(fam, to_dev(clen), to_dev(idx), pl, pS, pool_M=pM, S_init=to_dev(S_init))
    ref = oracle.compose_chain(fam, clen, idx, pool["lam"], pool["S"], pool_M=pool.get("M"), S_init=S_init)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert rel_fro(to_host(got), ref).max() <= TOL_F32
    assert rel_fro(to_host(got), to_host(plain)).max() <= TOL_F32
    assert np.array_equal(to_host(got)[2], S_init[2])        # an empty chain leaves S_init


def test_tree_bad_lengths_and_indices_are_flagged():
    import torch
    import linear_attention_state_gated_gb300 as hy
    lens = [10, 20, 30]
    Lyr, H, d = 1, 2, 64
    pool = scanned_pool(wl.SCALAR, lens, Lyr, H, d, seed=230)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = np.zeros((2, 16), np.int32)
    idx[1, 3] = 7                                             # outside the pool
    hy.compose_chain(wl.SCALAR, to_dev(np.array([16, 16], np.int32)), to_dev(idx), to_dev(pool["lam"]),
                     to_dev(pool["S"]), workspace="auto", d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -5
    err.zero_()
    hy.compose_chain(wl.SCALAR, to_dev(np.array([17, 3], np.int32)), to_dev(np.zeros((2, 16), np.int32)),
                     to_dev(pool["lam"]), to_dev(pool["S"]), workspace="auto", d_err=err)   # length past max_chain
    torch.cuda.synchronize()
    assert int(err.item()) == -5


def test_many_units_take_the_plain_chain():
    import linear_attention_state_gated_gb300 as hy
    assert hy.compose_chain_workspace_bytes(wl.SCALAR, 64, 30, 32, 128, 128, 20) == 0
    assert hy.compose_chain_workspace_bytes(wl.DENSE, 1, 1, 4, 128, 128, 4) == 0     # short chains
