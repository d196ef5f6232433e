"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every symbol ``include/hypic.h`` declares, and rejects bad arguments on the
host with the documented status codes before touching the device.  Fake
(never dereferenced) device addresses stand in for tensors here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hypic.h")

OK, EINVAL, EUNSUP, EALIGN = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    from linear_attention_state_gated_gb300 import _build, library
    _build.build()
    return library()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("hypic_segment_scan", "hypic_compose", "hypic_compose_chain", "hypic_status_string"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    from linear_attention_state_gated_gb300 import SIGNATURES
    for s in declared_symbols():
        assert hasattr(lib, s), s
        assert s in SIGNATURES, f"binding lacks a signature for {s}"


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(lib.hypic_status_string(st), bytes)
    assert lib.hypic_version() >= 100


A = 0x10000          # fake 16-byte aligned device address (never dereferenced)


def P(x):
    return ctypes.c_void_p(x)


def scan(lib, fam=0, dtype=0, L=1, S=2, N=64, H=2, dk=128, dv=128, offs=A, q=0, k=A, v=A,
         alpha=A, beta=0, lam=A, M=0, Sout=A, o=0, err=0):
    return lib.hypic_segment_scan(fam, dtype, L, S, N, H, dk, dv, P(offs), P(q or None),
                                  P(k or None), P(v or None), P(alpha or None), P(beta or None),
                                  P(lam or None), P(M or None), P(Sout or None), P(o or None),
                                  P(err or None), P(None))


def test_scan_rejects_bad_arguments(lib):
    assert scan(lib, fam=4) == EINVAL
    assert scan(lib, dtype=2) == EINVAL
    assert scan(lib, dk=96) == EUNSUP
    assert scan(lib, dv=256) == EUNSUP
    assert scan(lib, H=0) == EINVAL
    assert scan(lib, N=-1) == EINVAL
    assert scan(lib, k=0) == EINVAL
    assert scan(lib, alpha=0) == EINVAL
    assert scan(lib, Sout=0) == EINVAL
    assert scan(lib, fam=2, M=0) == EINVAL          # dense needs M_out
    assert scan(lib, fam=3, M=0) == EINVAL          # so does KDA
    assert scan(lib, fam=3, M=A + 0x100000, alpha=A + 4) == EALIGN   # KDA gates: 16-byte rows
    assert scan(lib, fam=0, M=A) == EINVAL          # scalar must not get M_out
    assert scan(lib, o=A, q=0) == EINVAL            # o_t needs q
    assert scan(lib, k=A + 8) == EALIGN
    assert scan(lib, Sout=A + 4) == EALIGN
    assert scan(lib, fam=1, alpha=A + 4) == EALIGN  # diag gates are 16-byte rows
    assert scan(lib, offs=A + 4) == EALIGN
    assert scan(lib, L=0) == OK                     # nothing to do: no launch
    assert scan(lib, S=0) == OK


def scan_ws(lib, fam=2, dtype=0, L=1, S=2, N=64, H=2, dk=128, dv=128, ws=0x40000000, ws_bytes=1 << 30,
            M=A + 0x1000000, o=0, q=0):
    return lib.hypic_segment_scan_ws(fam, dtype, L, S, N, H, dk, dv, P(A), P(q or None), P(A), P(A), P(A),
                                     P(None), P(A), P(M or None), P(A + 0x2000000), P(o or None),
                                     P(ws or None), ws_bytes, P(None), P(None))


def test_workspace_size_and_checks(lib):
    """The two-pass dense scan: one 49424-byte record (50192 with o_t) per
    (layer, head, chunk slot), n_seg + N / 64 slots, then the segments' order
    (int32 each), both 256-byte aligned; the chunked KDA scan: a pair per
    (layer, chunk slot, head) and its index arrays; the balanced
    diagonal scan: a fixed 2 x 512 partial slots; other options take none."""
    ws = lib.hypic_segment_scan_workspace_bytes
    up = lambda b: (b + 255) // 256 * 256   # noqa: E731

    def dense(L, n_seg, N, H, rec):   # records, then the segment order (int32 each)
        return up(L * H * (n_seg + N // 64) * rec) + up(4 * n_seg)

    assert ws(2, 0, 30, 1, 2048, 32, 128, 128, 0) == dense(30, 1, 2048, 32, 49424)
    assert ws(2, 0, 1, 3, 200, 2, 128, 128, 0) == dense(1, 3, 200, 2, 49424)
    assert ws(2, 0, 1, 1, 2048, 2, 128, 128, 1) == dense(1, 1, 2048, 2, 50192)   # with o_t: Gq tiles and b_t too
    assert ws(2, 1, 1, 1, 2048, 2, 128, 128, 0) == 0     # fp32 inputs
    def kda(L, n_seg, N, H):   # per chunk slot: M_c, S_c (fp32), lambda; steep list; slot starts; chains
        slots = n_seg + N // 64
        rows = L * slots * H
        return (2 * up(rows * 128 * 128 * 4) + up(rows * 4) + up((rows + 1) * 4) + up((slots + 1) * 8)
                + 2 * up(L * n_seg * 4))

    assert ws(3, 0, 30, 1, 2048, 32, 128, 128, 0) == kda(30, 1, 2048, 32)   # KDA: chunk pairs, then chains
    assert ws(3, 0, 2, 7, 592, 3, 128, 128, 0) == kda(2, 7, 592, 3)
    assert ws(3, 0, 1, 1, 2048, 2, 128, 128, 1) == 0     # KDA with o_t: the token-by-token kernel
    assert ws(3, 1, 1, 1, 2048, 2, 128, 128, 0) == 0     # ... fp32 inputs too
    assert ws(3, 0, 1, 1, 2048, 2, 64, 64, 0) == 0
    assert ws(3, 0, 30, 2000, 1 << 20, 32, 128, 128, 0) == 0   # above 64 GiB of pairs: token by token
    assert ws(2, 0, 1, 1, 2048, 2, 64, 64, 0) == 0
    sd = 2 * 512 * (128 + 128 * 128) * 4      # diag: two partial slots per CTA, up to 512 CTAs
    assert ws(1, 0, 1, 1, 2048, 2, 128, 128, 0) == sd
    assert ws(1, 0, 30, 8, 8192, 32, 128, 128, 0) == sd
    assert ws(0, 0, 1, 1, 2048, 2, 128, 128, 0) == 0     # scalar: one chain per CTA, no scratch
    assert ws(1, 0, 1, 1, 2048, 2, 128, 128, 1) == 0     # o_t: the recurrent kernel
    assert ws(1, 0, 1, 600, 2048, 2, 128, 128, 0) == 0   # more segments than the schedule indexes
    assert ws(1, 0, 1, 1, 2048, 2, 64, 64, 0) == 0
    assert ws(2, 0, 1, 1, 2048, 0, 128, 128, 0) == EINVAL
    need = ws(2, 0, 1, 2, 64, 2, 128, 128, 0)
    assert scan_ws(lib, ws_bytes=need - 16) == EINVAL
    assert scan_ws(lib, ws=0) == EINVAL
    assert scan_ws(lib, ws=0x40000000 + 16) == EALIGN
    assert scan_ws(lib, ws_bytes=-1) == EINVAL
    assert scan_ws(lib, dk=96) == EUNSUP
    assert scan_ws(lib, M=0) == EINVAL
    assert scan_ws(lib, L=0) == OK


def compose(lib, fam=0, n=3, H=2, dk=64, dv=64, lam=A, M=0, Sp=A, Sc=A + 0x100000,
            So=A + 0x200000, lp=0, Mp=0, lo=0, Mo=0):
    return lib.hypic_compose(fam, n, H, dk, dv, P(lam or None), P(M or None), P(Sp or None),
                             P(Sc or None), P(So or None), P(lp or None), P(Mp or None),
                             P(lo or None), P(Mo or None), P(None))


def test_compose_rejects_bad_arguments(lib):
    assert compose(lib, fam=5) == EINVAL
    assert compose(lib, fam=3, M=0) == EINVAL       # KDA composes like dense: needs M
    assert compose(lib, dk=48) == EUNSUP
    assert compose(lib, lam=0) == EINVAL
    assert compose(lib, Sc=0) == EINVAL
    assert compose(lib, fam=2, M=0) == EINVAL
    assert compose(lib, fam=0, M=A) == EINVAL
    assert compose(lib, lp=A) == EINVAL              # lam_prev without lam_out
    assert compose(lib, fam=2, M=A + 0x300000, lp=A, lo=A, Mp=0, Mo=A) == EINVAL
    assert compose(lib, Sc=A + 0x100008) == EALIGN
    assert compose(lib, So=A + 0x100000 + 64) == EINVAL  # S_out overlaps S_C
    # lam_out aliasing lam or lam_prev (no in-place operator accumulation), any family
    for fam, M_ in ((0, 0), (1, 0), (2, A + 0x300000)):
        Mp = A + 0x400000 if fam == 2 else 0
        Mo = A + 0x500000 if fam == 2 else 0
        assert compose(lib, fam=fam, M=M_, lp=A + 0x600000, lo=A, Mp=Mp, Mo=Mo) == EINVAL
        assert compose(lib, fam=fam, M=M_, lp=A + 0x600000, lo=A + 0x600000, Mp=Mp, Mo=Mo) == EINVAL
    assert compose(lib, n=0) == OK


def chain(lib, fam=0, R=2, L=2, H=2, dk=64, dv=64, mc=3, cl=A, idx=A, P_=5, pl=A, pM=0,
          pS=A, Si=0, So=A + 0x800000, err=0):
    return lib.hypic_compose_chain(fam, R, L, H, dk, dv, mc, P(cl or None), P(idx or None), P_,
                                   P(pl or None), P(pM or None), P(pS or None), P(Si or None),
                                   P(So or None), P(err or None), P(None))


def test_chain_rejects_bad_arguments(lib):
    assert chain(lib, fam=4) == EINVAL
    assert chain(lib, fam=3, pM=0) == EINVAL
    assert chain(lib, dv=16) == EUNSUP
    assert chain(lib, cl=0) == EINVAL
    assert chain(lib, idx=0) == EINVAL
    assert chain(lib, P_=0) == EINVAL
    assert chain(lib, fam=2, pM=0) == EINVAL
    assert chain(lib, pS=A + 4) == EALIGN
    assert chain(lib, cl=A + 2) == EALIGN
    assert chain(lib, So=A + 0x10000) == EINVAL     # S_out inside the pool's states
    assert chain(lib, pl=A + 0x801000) == EINVAL    # the pool's lambdas inside S_out
    assert chain(lib, Si=A + 0x800000 + 0x100) == EINVAL   # S_init partly overlapping S_out
    assert chain(lib, R=0) == OK


def chain_ws(lib, fam=0, R=2, L=1, H=2, dk=64, dv=64, mc=64, cl=A, idx=A + 0x1000, P_=5, pl=A + 0x2000, pM=0,
             pS=A + 0x100000, Si=0, So=A + 0x800000, ws=A + 0x1000000, wsb=1 << 30, err=0):
    return lib.hypic_compose_chain_ws(fam, R, L, H, dk, dv, mc, P(cl or None), P(idx or None), P_,
                                      P(pl or None), P(pM or None), P(pS or None), P(Si or None),
                                      P(So or None), P(ws or None), wsb, P(err or None), P(None))


def test_chain_ws_rejects_bad_arguments(lib):
    need = lib.hypic_compose_chain_workspace_bytes(0, 2, 1, 2, 64, 64, 64)
    assert need > 0                                   # 4 units with 64-entry chains: the two-level tree
    assert lib.hypic_compose_chain_workspace_bytes(0, 2, 1, 2, 64, 64, 4) == 0     # short chains: plain
    assert lib.hypic_compose_chain_workspace_bytes(0, 64, 30, 32, 64, 64, 64) == 0  # many units: plain
    assert lib.hypic_compose_chain_workspace_bytes(5, 2, 1, 2, 64, 64, 64) == EINVAL
    assert lib.hypic_compose_chain_workspace_bytes(0, 2, 1, 2, 48, 64, 64) == EUNSUP
    assert chain_ws(lib, wsb=need - 1) == EINVAL     # scratch too small
    assert chain_ws(lib, ws=0) == EINVAL
    assert chain_ws(lib, wsb=-1) == EINVAL
    assert chain_ws(lib, ws=A + 0x1000000 + 16) == EALIGN
    assert chain_ws(lib, ws=A + 0x100000) == EINVAL   # scratch over the pool
    assert chain_ws(lib, ws=A + 0x800000) == EINVAL   # scratch over S_out
    assert chain_ws(lib, So=A + 0x100100) == EINVAL   # S_out inside the pool
    assert chain_ws(lib, fam=2, pM=0) == EINVAL
    assert chain_ws(lib, dv=16) == EUNSUP
    assert chain_ws(lib, R=0) == OK


def prefix(lib, fam=0, R=2, L=2, H=2, dk=64, dv=64, mc=3, cl=A, idx=A, P_=5, pl=A, pM=0, pS=A + 0x100000,
           lo=A + 0x300000, Mo=0, So=A + 0x400000, err=0):
    return lib.hypic_compose_prefix(fam, R, L, H, dk, dv, mc, P(cl or None), P(idx or None), P_,
                                    P(pl or None), P(pM or None), P(pS or None), P(lo or None), P(Mo or None),
                                    P(So or None), P(err or None), P(None))


def test_prefix_rejects_bad_arguments(lib):
    assert prefix(lib, fam=4) == EINVAL
    assert prefix(lib, dk=48) == EUNSUP
    assert prefix(lib, lo=0) == EINVAL                 # the operator's lambda is an output
    assert prefix(lib, fam=2, pM=A + 0x200000) == EINVAL   # dense needs M_out
    assert prefix(lib, fam=0, Mo=A + 0x500000) == EINVAL   # scalar must not get one
    assert prefix(lib, fam=3, pM=0, Mo=A + 0x500000) == EINVAL   # KDA needs pool_M
    assert prefix(lib, So=A + 0x100000 + 64) == EINVAL  # S_out overlaps the pool
    assert prefix(lib, lo=A + 0x400000 + 4) == EINVAL   # lambda overlaps S_out
    assert prefix(lib, pS=A + 0x100004) == EALIGN
    assert prefix(lib, R=0) == OK


def seam(lib, fam=0, dtype=0, n=2, w=8, H=2, dk=64, dv=64, q=0, k=A, v=A, alpha=A, beta=0,
         lam=A + 0x200000, M=0, Sp=0, Sc=A + 0x400000, So=A + 0x600000, o=0):
    return lib.hypic_seam_compose(fam, dtype, n, w, H, dk, dv, P(q or None), P(k or None), P(v or None),
                                  P(alpha or None), P(beta or None), P(lam or None), P(M or None),
                                  P(Sp or None), P(Sc or None), P(So or None), P(o or None), P(None))


def test_seam_rejects_bad_arguments(lib):
    assert seam(lib, fam=4) == EINVAL
    assert seam(lib, fam=3) == EINVAL               # KDA needs M
    assert seam(lib, dtype=2) == EINVAL
    assert seam(lib, w=-1) == EINVAL
    assert seam(lib, w=5000) == EUNSUP
    assert seam(lib, dk=48) == EUNSUP
    assert seam(lib, lam=0) == EINVAL
    assert seam(lib, Sc=0) == EINVAL
    assert seam(lib, fam=2, M=0) == EINVAL
    assert seam(lib, fam=1, M=A + 0x800000) == EINVAL
    assert seam(lib, k=0) == EINVAL                   # a window needs its tokens
    assert seam(lib, o=A + 0x900000) == EINVAL       # outputs need q
    assert seam(lib, Sc=A + 0x400008) == EALIGN
    assert seam(lib, k=A + 1) == EALIGN               # bf16 rows need 2-byte alignment
    assert seam(lib, So=A + 0x400000 + 64) == EINVAL  # S_out overlaps S_C
    assert seam(lib, n=0) == OK


def test_python_binding_refuses_host_tensors():
    import torch
    import linear_attention_state_gated_gb300 as hy
    k = torch.zeros(1, 4, 1, 32)
    with pytest.raises(ValueError):
        hy.segment_scan("scalar", k, k, torch.ones(1, 4, 1), torch.tensor([0, 4]))


def test_selftest_wait_rejects_bad_arguments(lib):
    """The bounded-wait diagnostic checks its limit and pointers before any launch."""
    f = lib.hypic_selftest_wait
    assert f(-1, 0, P(A), P(A), P(None)) == EINVAL
    assert f(4_000_000_001, 0, P(A), P(A), P(None)) == EINVAL
    assert f(1000, 0, P(A + 2), P(A), P(None)) == EALIGN
    assert f(1000, 0, P(A), P(A + 4), P(None)) == EALIGN
