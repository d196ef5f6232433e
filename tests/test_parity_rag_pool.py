"""RAG-style composition over a pool scanned on the GPU: 200 segments of
U{1024..4096} tokens under the scalar / diagonal law (drawn on the device), 2
layers x 32 heads, scanned into the pool (hypic_segment_scan), then 64 requests
x 20 distinct Zipf(1.1) entries folded in draw order (hypic_compose_chain), the
launch the benchmark times (there over 30 layers).  For sampled (request,
layer, head) units the oracle scans the request's 20 segments itself from the
same inputs (fp64, token by token) and chains them; the GPU pool entries and
the chained state must match within the bf16-input scan tolerance."""
import numpy as np
import pytest

import oracle
from helpers import TOL_SCAN_BF16, rel_fro, t_err, to_host
from linear_attention_state_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fam", [wl.SCALAR, wl.DIAG], ids=["scalar", "diag"])
def test_rag_chain_over_scanned_pool(fam):
    import torch
    import linear_attention_state_gated_gb300 as hy
    from bench import scan_rag_pool
    Lyr, H, d = 2, 32, 128
    lens, pool_lam, pool_S = scan_rag_pool(fam, Lyr, H=H, d=d)
    offs = np.concatenate([[0], np.cumsum(lens)])
    clen, idx = wl.rag_requests()
    dev = torch.device("cuda")
    got = hy.compose_chain(fam, torch.from_numpy(clen).to(dev), torch.from_numpy(idx).to(dev), pool_lam, pool_S)
    torch.cuda.synchronize()
    rs = np.random.default_rng(23)
    units = [(0, 0, 0), (63, 1, 31)] + [tuple(x) for x in rs.integers([0, 0, 0], [64, Lyr, H], size=(2, 3))]
    for r, l, h in units:
        k, v, a, _ = wl.scalar_diag_layer_device(fam, lens, l, H=H, d=d, heads=[h])
        k, v, a = to_host(k), to_host(v), to_host(a)
        segs = idx[r, :clen[r]]
        rows = np.concatenate([np.arange(offs[p], offs[p + 1]) for p in segs])
        so = np.concatenate([[0], np.cumsum(lens[segs])]).astype(np.int64)
        ref = oracle.segment_scan(fam, np.ascontiguousarray(k[:, rows]), np.ascontiguousarray(v[:, rows]),
                                  np.ascontiguousarray(a[:, rows]), so)
        # the GPU's pool entries of this request, layer and head
        g_lam = to_host(pool_lam[torch.from_numpy(segs.astype(np.int64)).to(dev), l, h])
        g_S = to_host(pool_S[torch.from_numpy(segs.astype(np.int64)).to(dev), l, h])
        assert rel_fro(g_S, ref["S"][0, :, 0]).max() <= TOL_SCAN_BF16
        assert t_err(fam, g_lam, ref["lam"][0, :, 0]).max() <= TOL_SCAN_BF16
        # the chain of the oracle's own scans, in the request's order
        n = len(segs)
        lam_o = np.ascontiguousarray(np.moveaxis(ref["lam"], 1, 0)).astype(np.float32)   # [n, 1, 1(, d)]
        S_o = np.ascontiguousarray(np.moveaxis(ref["S"], 1, 0)).astype(np.float32)       # [n, 1, 1, d, d]
        chain = oracle.compose_chain(fam, np.array([n], np.int32), np.arange(n, dtype=np.int32)[None], lam_o, S_o)
        assert rel_fro(to_host(got[r, l, h]), chain[0, 0, 0]) <= TOL_SCAN_BF16
