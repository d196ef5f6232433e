"""fp64 CPU oracle for the HYPIC segment scan and state composition.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
CUDA library and its Python binding) never imports this package, and this
package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64, token by token); this
module only compiles it on demand and marshals numpy arrays through ctypes.
Each function states the passage it follows:

* ``segment_scan`` -- xix.ai/fr HYPIC article, paragraph on linear layers:
  T_C is the product of the segment's per-token transitions and S(C|0) the
  final state from a zero start; per-token rule per family as documented in
  ``oracle.c`` (the pages print none).
* ``compose`` -- same paragraph: S(C1.C2) = T(C2) S(C1) + S(C2).
* ``compose_chain`` -- same paragraph ("under any prefix") and remio.ai/ja
  "cold requests become parallel" (the combine step folds each segment's pair
  into the running state).
* ``sequential`` -- the straight recurrence over the concatenated tokens: a
  scan with one segment.

Parity unpinned: none.  Every function is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

SCALAR, DIAG, DENSE, KDA = 0, 1, 2, 3
FAMILIES = {"scalar": SCALAR, "diag": DIAG, "dense": DENSE, "kda": KDA}
WITH_M = (DENSE, KDA)   # families whose operator is exp(lambda) * M

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile one C source of the oracle into a shared library (gcc, OpenMP)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def open_library(path: str):
    """ctypes handle with the oracle's signatures declared."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    lib.oracle_segment_scan.argtypes = [i32, i32, i32, i64, i32, i32, i32, P,
                                        P, P, P, P, P, P, P, P, P, i32]
    lib.oracle_segment_scan.restype = i32
    lib.oracle_compose.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
    lib.oracle_compose.restype = i32
    lib.oracle_compose_chain.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, i32,
                                         P, P, P, P, P, i32]
    lib.oracle_compose_chain.restype = i32
    lib.oracle_compose_prefix.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, i32, P, P, P, P, P, P]
    lib.oracle_compose_prefix.restype = i32
    lib.oracle_seam_compose.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_seam_compose.restype = i32
    lib.oracle_max_threads.restype = i32
    return lib


_override = threading.local()


def _load():
    lib = getattr(_override, "lib", None)
    if lib is not None:
        return lib
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


class using_library:
    """Context manager: route this thread's oracle calls to another build of
    the oracle (used only by the tests that plant mistakes in a copy of
    ``oracle.c`` and check that the pins catch them)."""

    def __init__(self, path: str):
        self.lib = open_library(path)

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev
        return False


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _fam(f):
    return FAMILIES[f] if isinstance(f, str) else int(f)


def segment_scan(fam, k, v, alpha, seg_offsets, beta=None, q=None, want_o=False,
                 n_threads=0):
    """Scan every (layer, segment, head) token by token in fp64.

    k [Lyr,N,H,dk], v [Lyr,N,H,dv], alpha [Lyr,N,H] or [Lyr,N,H,dk] (diag, kda),
    beta [Lyr,N,H] or None, q [Lyr,N,H,dk] (needed iff want_o),
    seg_offsets [n_seg+1] int64.  Returns dict lam, M (dense), S, o (if asked).
    """
    fam = _fam(fam)
    k, v, alpha, beta, q = _f64(k), _f64(v), _f64(alpha), _f64(beta), _f64(q)
    Lyr, N, H, dk = k.shape
    dv = v.shape[3]
    offs = np.ascontiguousarray(np.asarray(seg_offsets, dtype=np.int64))
    n_seg = offs.shape[0] - 1
    lam = np.zeros((Lyr, n_seg, H, dk) if fam == DIAG else (Lyr, n_seg, H), np.float64)
    M = np.zeros((Lyr, n_seg, H, dk, dk), np.float64) if fam in WITH_M else None
    S = np.zeros((Lyr, n_seg, H, dk, dv), np.float64)
    o = np.zeros((Lyr, N, H, dv), np.float64) if want_o else None
    rc = _load().oracle_segment_scan(fam, Lyr, n_seg, N, H, dk, dv, _ptr(offs), _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(lam),
                                     _ptr(M), _ptr(S), _ptr(o), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_segment_scan: bad arguments ({rc})")
    out = {"lam": lam, "S": S}
    if M is not None:
        out["M"] = M
    if o is not None:
        out["o"] = o
    return out


def sequential(fam, k, v, alpha, beta=None, q=None, want_o=False, n_threads=0):
    """Straight recurrence over all N tokens of each layer (one segment)."""
    N = np.asarray(k).shape[1]
    out = segment_scan(fam, k, v, alpha, [0, N], beta=beta, q=q, want_o=want_o,
                       n_threads=n_threads)
    res = {"lam": out["lam"][:, 0], "S": out["S"][:, 0]}
    if "M" in out:
        res["M"] = out["M"][:, 0]
    if "o" in out:
        res["o"] = out["o"]
    return res


def compose(fam, lam, S_C, S_prev=None, M=None, lam_prev=None, M_prev=None):
    """S = T S_prev + S_C over [n,H] items; optionally the composed operator.

    Returns dict S and, when lam_prev is given, lam_out (and M_out for dense).
    """
    fam = _fam(fam)
    lam, S_C, S_prev, M = _f64(lam), _f64(S_C), _f64(S_prev), _f64(M)
    lam_prev, M_prev = _f64(lam_prev), _f64(M_prev)
    n, H, dk, dv = S_C.shape
    S = np.zeros_like(S_C)
    lam_out = np.zeros_like(lam) if lam_prev is not None else None
    M_out = np.zeros_like(M) if (lam_prev is not None and fam in WITH_M) else None
    rc = _load().oracle_compose(fam, n, H, dk, dv, _ptr(lam), _ptr(M), _ptr(S_prev), _ptr(S_C),
                                _ptr(S), _ptr(lam_prev), _ptr(M_prev), _ptr(lam_out), _ptr(M_out))
    if rc != 0:
        raise ValueError(f"oracle_compose: bad arguments ({rc})")
    out = {"S": S}
    if lam_out is not None:
        out["lam"] = lam_out
    if M_out is not None:
        out["M"] = M_out
    return out


def compose_chain(fam, chain_len, seg_idx, pool_lam, pool_S, pool_M=None, S_init=None,
                  n_threads=0):
    """Fold pool entries seg_idx[r, :chain_len[r]] in order into each request's state.

    pool_lam [P,Lyr,H(,dk)], pool_M [P,Lyr,H,dk,dk], pool_S [P,Lyr,H,dk,dv],
    S_init [R,Lyr,H,dk,dv] or None.  Returns S [R,Lyr,H,dk,dv].
    """
    fam = _fam(fam)
    chain_len = np.ascontiguousarray(np.asarray(chain_len, dtype=np.int32))
    seg_idx = np.ascontiguousarray(np.asarray(seg_idx, dtype=np.int32))
    pool_lam, pool_S, pool_M, S_init = _f64(pool_lam), _f64(pool_S), _f64(pool_M), _f64(S_init)
    P, Lyr, H, dk, dv = pool_S.shape
    R = chain_len.shape[0]
    max_chain = seg_idx.shape[1] if seg_idx.ndim == 2 else 0
    S = np.zeros((R, Lyr, H, dk, dv), np.float64)
    rc = _load().oracle_compose_chain(fam, R, Lyr, H, dk, dv, max_chain, _ptr(chain_len),
                                      _ptr(seg_idx), P, _ptr(pool_lam), _ptr(pool_M),
                                      _ptr(pool_S), _ptr(S_init), _ptr(S), int(n_threads))
    if rc == -2:
        raise IndexError("oracle_compose_chain: pool index out of range")
    if rc != 0:
        raise ValueError(f"oracle_compose_chain: bad arguments ({rc})")
    return S


def compose_prefix(fam, chain_len, seg_idx, pool_lam, pool_S, pool_M=None):
    """The cached pair of each request's ordered pool entries (a composed prefix):
    T = T_{p_n} ... T_{p_1} as lam (and M) and S = S(C_{p_1} ... C_{p_n} | 0).
    Returns dict lam [R,Lyr,H(,dk)], M [R,Lyr,H,dk,dk] (dense, kda), S [R,Lyr,H,dk,dv]."""
    fam = _fam(fam)
    chain_len = np.ascontiguousarray(np.asarray(chain_len, dtype=np.int32))
    seg_idx = np.ascontiguousarray(np.asarray(seg_idx, dtype=np.int32))
    pool_lam, pool_S, pool_M = _f64(pool_lam), _f64(pool_S), _f64(pool_M)
    P, Lyr, H, dk, dv = pool_S.shape
    R = chain_len.shape[0]
    max_chain = seg_idx.shape[1] if seg_idx.ndim == 2 else 0
    S = np.zeros((R, Lyr, H, dk, dv), np.float64)
    lam = np.zeros((R, Lyr, H, dk) if fam == DIAG else (R, Lyr, H), np.float64)
    M = np.zeros((R, Lyr, H, dk, dk), np.float64) if fam in WITH_M else None
    rc = _load().oracle_compose_prefix(fam, R, Lyr, H, dk, dv, max_chain, _ptr(chain_len), _ptr(seg_idx), P,
                                       _ptr(pool_lam), _ptr(pool_M), _ptr(pool_S), _ptr(lam), _ptr(M), _ptr(S))
    if rc == -2:
        raise IndexError("oracle_compose_prefix: pool index out of range")
    if rc != 0:
        raise ValueError(f"oracle_compose_prefix: bad arguments ({rc})")
    out = {"lam": lam, "S": S}
    if M is not None:
        out["M"] = M
    return out


def seam_compose(fam, k, v, alpha, lam, S_C, S_prev=None, M=None, beta=None, q=None,
                 want_o=False):
    """Seam-window advance then composition, per item and head, in fp64.

    k [n,w,H,dk], v [n,w,H,dv], alpha [n,w,H] or [n,w,H,dk] (diag), beta
    [n,w,H] or None, q [n,w,H,dk] (needed iff want_o); lam [n,H] or [n,H,dk],
    M [n,H,dk,dk] (dense), S_prev (or None) and S_C [n,H,dk,dv].
    Returns dict S [n,H,dk,dv] and, if asked, o [n,w,H,dv].
    """
    fam = _fam(fam)
    k, v, alpha, beta, q = _f64(k), _f64(v), _f64(alpha), _f64(beta), _f64(q)
    lam, S_C, S_prev, M = _f64(lam), _f64(S_C), _f64(S_prev), _f64(M)
    n, H, dk, dv = S_C.shape
    w = k.shape[1]
    S = np.zeros_like(S_C)
    o = np.zeros((n, w, H, dv), np.float64) if want_o else None
    rc = _load().oracle_seam_compose(fam, n, w, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                     _ptr(beta), _ptr(lam), _ptr(M), _ptr(S_prev), _ptr(S_C), _ptr(S),
                                     _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle_seam_compose: bad arguments ({rc})")
    out = {"S": S}
    if o is not None:
        out["o"] = o
    return out


def transition(out, fam=None):
    """Materialise T_C = exp(lam) * M from a scan result (dense) or exp(lam) (scalar/diag)."""
    if "M" in out:
        return np.exp(out["lam"])[..., None, None] * out["M"]
    return np.exp(out["lam"])
