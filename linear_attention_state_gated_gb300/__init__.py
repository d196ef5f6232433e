"""GB300-native segment scan and state composition for position-independent
caching of hybrid linear-attention models (HYPIC).

Thin ctypes binding over ``libhypic.so`` (built from ``csrc/`` by
``_build.build()``).  These functions only check and marshal arguments --
device pointers of torch tensors and the current CUDA stream -- into the
C ABI declared in ``include/hypic.h``; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: if the library is not
built, or a tensor is not on a CUDA device, the call raises.

The operations (HYPIC, xix.ai/fr article, paragraph on linear layers):
  segment_scan  -- per segment C and head, T_C = product of the per-token
                   transitions (as exp(lam) * M) and S(C|0), the final state
                   from a zero start; optionally o_t = S_t^T q_t.
  compose       -- S(C1.C2) = T(C2) S(C1) + S(C2), optionally T(C2) T(C1).
  compose_chain -- fold many cached pairs in order into a running state
                   (remio.ai/ja, "cold requests become parallel": the combine step).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

SCALAR, DIAG, DENSE, KDA = 0, 1, 2, 3
FAMILIES = {"scalar": SCALAR, "diag": DIAG, "dense": DENSE, "kda": KDA}
WITH_M = (DENSE, KDA)   # families whose operator is exp(lambda) M
BF16, F32 = 0, 1
STATUS = {0: "HYPIC_OK", -1: "HYPIC_EINVAL", -2: "HYPIC_EUNSUPPORTED", -3: "HYPIC_EALIGN",
          -4: "HYPIC_ECUDA", -5: "HYPIC_EINDEX", -6: "HYPIC_ETIMEOUT"}

__all__ = ["segment_scan", "segment_scan_workspace_bytes", "segment_scan_static", "compose", "compose_chain",
           "compose_chain_workspace_bytes",
           "compose_prefix", "seam_compose", "selftest_wait", "status_string", "library", "use_library",
           "HypicError", "SCALAR", "DIAG", "DENSE", "KDA"]


class HypicError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status_string(status)})")


_lock = threading.Lock()
_lib = None

# every symbol include/hypic.h declares, with its ctypes signature
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
SIGNATURES = {
    "hypic_segment_scan": (_I32, [_I32, _I32, _I32, _I32, _I64, _I32, _I32, _I32,
                                  _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "hypic_segment_scan_ws": (_I32, [_I32, _I32, _I32, _I32, _I64, _I32, _I32, _I32,
                                     _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P]),
    "hypic_segment_scan_static": (_I32, [_I32, _I32, _I32, _I32, _I64, _I32, _I32, _I32,
                                         _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "hypic_segment_scan_workspace_bytes": (_I64, [_I32, _I32, _I32, _I32, _I64, _I32, _I32, _I32, _I32]),
    "hypic_compose": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "hypic_compose_chain": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I32,
                                   _P, _P, _P, _P, _P, _P, _P]),
    "hypic_compose_chain_workspace_bytes": (_I64, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "hypic_compose_chain_ws": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I32,
                                      _P, _P, _P, _P, _P, _P, _I64, _P, _P]),
    "hypic_compose_prefix": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I32,
                                    _P, _P, _P, _P, _P, _P, _P, _P]),
    "hypic_seam_compose": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                  _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "hypic_status_string": (ctypes.c_char_p, [_I32]),
    "hypic_version": (_I32, []),
    "hypic_selftest_wait": (_I32, [ctypes.c_longlong, _I32, _P, _P, _P]),
}


def library(path: str | None = None):
    """Load libhypic.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with "
                                   "`python -m linear_attention_state_gated_gb300._build`")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return lib
            _lib = lib
    return _lib


def use_library(path: str):
    """Route every call of this module to the library at `path` (another build
    of libhypic, e.g. with different tile sizes); returns the handle."""
    global _lib
    lib = library(path)
    with _lock:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return library().hypic_status_string(int(status)).decode()


def _fam(f):
    return FAMILIES[f] if isinstance(f, str) else int(f)


def _dev(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        raise HypicError(fn, status)


def segment_scan_workspace_bytes(family, dtype, n_layers, n_seg, total_tokens, n_heads, d_k, d_v,
                                 with_o=False):
    """Bytes of device scratch the workspace form of the scan uses for these sizes
    (0: that form needs none for this family / size)."""
    n = library().hypic_segment_scan_workspace_bytes(
        _fam(family), BF16 if dtype == torch.bfloat16 else F32, n_layers, n_seg, total_tokens, n_heads,
        d_k, d_v, int(bool(with_o)))
    if n < 0:
        raise HypicError("hypic_segment_scan_workspace_bytes", n)
    return n


def segment_scan(family, k, v, alpha, seg_offsets, beta=None, q=None, want_o=False,
                 out=None, d_err=None, stream=None, workspace="auto"):
    """(T_C, S(C|0)) for every (layer, segment, head); optionally o_t.

    k [Lyr,N,H,dk], v [Lyr,N,H,dv] (bf16 or fp32), alpha fp32 [Lyr,N,H] or
    [Lyr,N,H,dk] (diag, kda), beta fp32 [Lyr,N,H] or None, q like k (for o_t),
    seg_offsets int64 [n_seg+1] on the device.  ``out`` may hold preallocated
    ``lam``, ``M``, ``S``, ``o`` tensors.  Returns a dict with lam, S, M (dense, kda), o.

    ``workspace``: "auto" (default) allocates the device scratch the two-pass
    form needs (through torch, on the launch stream) and calls
    hypic_segment_scan_ws; a uint8 CUDA tensor is used as that scratch; None
    calls hypic_segment_scan (the single-pass kernels, no scratch).
    """
    fam = _fam(family)
    k = _dev(k, "k")
    dt = k.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("k must be bf16 or fp32")
    v = _dev(v, "v", dt)
    alpha = _dev(alpha, "alpha", torch.float32)
    beta = _dev(beta, "beta", torch.float32, allow_none=True)
    seg_offsets = _dev(seg_offsets, "seg_offsets", torch.int64)
    if want_o:
        q = _dev(q, "q", dt)
    Lyr, N, H, dk = k.shape
    dv = v.shape[-1]
    n_seg = seg_offsets.numel() - 1
    out = dict(out or {})
    dev = k.device
    lam_shape = (Lyr, n_seg, H, dk) if fam == DIAG else (Lyr, n_seg, H)
    if "lam" not in out:
        out["lam"] = torch.empty(lam_shape, dtype=torch.float32, device=dev)
    if "S" not in out:
        out["S"] = torch.empty((Lyr, n_seg, H, dk, dv), dtype=torch.float32, device=dev)
    if fam in WITH_M and "M" not in out:
        out["M"] = torch.empty((Lyr, n_seg, H, dk, dk), dtype=torch.float32, device=dev)
    if want_o and "o" not in out:
        out["o"] = torch.empty((Lyr, N, H, dv), dtype=dt, device=dev)
    args = (fam, BF16 if dt == torch.bfloat16 else F32, Lyr, n_seg, N, H, dk, dv,
            _ptr(seg_offsets), _ptr(q if want_o else None), _ptr(k), _ptr(v), _ptr(alpha),
            _ptr(beta), _ptr(out["lam"]), _ptr(out.get("M") if fam in WITH_M else None),
            _ptr(out["S"]), _ptr(out.get("o") if want_o else None))
    if workspace is None:
        st = library().hypic_segment_scan(*args, _ptr(d_err), _stream(stream))
        _check("hypic_segment_scan", st)
        return out
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        nbytes = segment_scan_workspace_bytes(fam, dt, Lyr, n_seg, N, H, dk, dv, want_o)
        if nbytes > 0:
            with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        else:
            workspace = None
    else:
        workspace = _dev(workspace, "workspace", torch.uint8)
    st = library().hypic_segment_scan_ws(*args, _ptr(workspace),
                                         0 if workspace is None else workspace.numel(),
                                         _ptr(d_err), _stream(stream))
    _check("hypic_segment_scan_ws", st)
    return out


def segment_scan_static(k, v, alpha, seg_offsets, out, beta=None, d_err=None, stream=None):
    """Dense (gated delta rule) scan through hypic_segment_scan_static: the
    library's fixed device scratch, no allocation anywhere in the call.  ``out``
    must hold caller-allocated ``lam`` [Lyr,n_seg,H], ``M`` and ``S``
    [Lyr,n_seg,H,128,128] fp32 tensors; k, v bf16 with d_k = d_v = 128."""
    k = _dev(k, "k", torch.bfloat16)
    v = _dev(v, "v", torch.bfloat16)
    alpha = _dev(alpha, "alpha", torch.float32)
    beta = _dev(beta, "beta", torch.float32, allow_none=True)
    seg_offsets = _dev(seg_offsets, "seg_offsets", torch.int64)
    lam = _dev(out.get("lam"), "out['lam']", torch.float32)
    M = _dev(out.get("M"), "out['M']", torch.float32)
    S = _dev(out.get("S"), "out['S']", torch.float32)
    Lyr, N, H, dk = k.shape
    st = library().hypic_segment_scan_static(
        DENSE, BF16, Lyr, seg_offsets.numel() - 1, N, H, dk, v.shape[-1], _ptr(seg_offsets), _ptr(k),
        _ptr(v), _ptr(alpha), _ptr(beta), _ptr(lam), _ptr(M), _ptr(S), _ptr(d_err), _stream(stream))
    _check("hypic_segment_scan_static", st)
    return out


def compose(family, lam, S_C, S_prev=None, M=None, lam_prev=None, M_prev=None, S_out=None,
            lam_out=None, M_out=None, stream=None):
    """S = exp(lam) M S_prev + S_C over [n, H] items (M = 1 / I for scalar / diag).

    With lam_prev (and M_prev for dense) also returns the composed operator
    T(C1.C2) = T(C2) T(C1) as lam (and M).  S_out may be S_prev (in place).
    """
    fam = _fam(family)
    S_C = _dev(S_C, "S_C", torch.float32)
    lam = _dev(lam, "lam", torch.float32)
    S_prev = _dev(S_prev, "S_prev", torch.float32, allow_none=True)
    M = _dev(M, "M", torch.float32, allow_none=True)
    lam_prev = _dev(lam_prev, "lam_prev", torch.float32, allow_none=True)
    M_prev = _dev(M_prev, "M_prev", torch.float32, allow_none=True)
    n, H, dk, dv = S_C.shape
    if S_out is None:
        S_out = torch.empty_like(S_C)
    want_T = lam_prev is not None
    if want_T and lam_out is None:
        lam_out = torch.empty_like(lam)
    if want_T and fam in WITH_M and M_out is None:
        M_out = torch.empty_like(M)
    st = library().hypic_compose(fam, n, H, dk, dv, _ptr(lam), _ptr(M), _ptr(S_prev), _ptr(S_C),
                                 _ptr(S_out), _ptr(lam_prev), _ptr(M_prev),
                                 _ptr(lam_out if want_T else None),
                                 _ptr(M_out if (want_T and fam in WITH_M) else None),
                                 _stream(stream))
    _check("hypic_compose", st)
    res = {"S": S_out}
    if want_T:
        res["lam"] = lam_out
        if fam in WITH_M:
            res["M"] = M_out
    return res


def compose_prefix(family, chain_len, seg_idx, pool_lam, pool_S, pool_M=None, out=None, d_err=None,
                   stream=None):
    """The cached pair of each request's ordered pool entries (hypic_compose_prefix):
    T = T_pn ... T_p1 as lam (and M) and S = S(C_p1 ... C_pn | 0).  ``out`` may hold
    preallocated ``lam``, ``M``, ``S``.  Returns a dict with lam, S and M (dense, kda)."""
    fam = _fam(family)
    chain_len = _dev(chain_len, "chain_len", torch.int32)
    seg_idx = _dev(seg_idx, "seg_idx", torch.int32)
    pool_lam = _dev(pool_lam, "pool_lam", torch.float32)
    pool_S = _dev(pool_S, "pool_S", torch.float32)
    pool_M = _dev(pool_M, "pool_M", torch.float32, allow_none=True)
    P, Lyr, H, dk, dv = pool_S.shape
    R = chain_len.numel()
    max_chain = seg_idx.shape[1] if seg_idx.dim() == 2 else 0
    out = dict(out or {})
    f = dict(dtype=torch.float32, device=pool_S.device)
    if "lam" not in out:
        out["lam"] = torch.empty((R, Lyr, H, dk) if fam == DIAG else (R, Lyr, H), **f)
    if "S" not in out:
        out["S"] = torch.empty((R, Lyr, H, dk, dv), **f)
    if fam in WITH_M and "M" not in out:
        out["M"] = torch.empty((R, Lyr, H, dk, dk), **f)
    st = library().hypic_compose_prefix(fam, R, Lyr, H, dk, dv, max_chain, _ptr(chain_len), _ptr(seg_idx), P,
                                        _ptr(pool_lam), _ptr(pool_M), _ptr(pool_S), _ptr(out["lam"]),
                                        _ptr(out.get("M") if fam in WITH_M else None), _ptr(out["S"]),
                                        _ptr(d_err), _stream(stream))
    _check("hypic_compose_prefix", st)
    return out


def seam_compose(family, k, v, alpha, lam, S_C, S_prev=None, M=None, beta=None, q=None,
                 want_o=False, S_out=None, o_out=None, stream=None):
    """Seam-window advance, then the cached rest of the segment (hypic_seam_compose).

    k [n,w,H,dk], v [n,w,H,dv] (bf16 or fp32), alpha [n,w,H] or [n,w,H,dk], beta
    [n,w,H] or None, q [n,w,H,dk] (needed iff want_o); lam [n,H] or [n,H,dk],
    M [n,H,dk,dk] (dense, kda), S_prev (or None) and S_C [n,H,dk,dv] fp32.  Returns a
    dict with S [n,H,dk,dv] and, if asked, o [n,w,H,dv] in the input dtype.
    S_out may be S_prev (in place).
    """
    fam = _fam(family)
    k = _dev(k, "k")
    dt = k.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("k must be bf16 or fp32")
    v = _dev(v, "v", dt)
    alpha = _dev(alpha, "alpha", torch.float32)
    beta = _dev(beta, "beta", torch.float32, allow_none=True)
    lam = _dev(lam, "lam", torch.float32)
    S_C = _dev(S_C, "S_C", torch.float32)
    S_prev = _dev(S_prev, "S_prev", torch.float32, allow_none=True)
    M = _dev(M, "M", torch.float32, allow_none=True)
    if want_o:
        q = _dev(q, "q", dt)
    n, w, H, dk = k.shape
    dv = v.shape[-1]
    if S_out is None:
        S_out = torch.empty_like(S_C)
    if want_o and o_out is None:
        o_out = torch.empty((n, w, H, dv), dtype=dt, device=k.device)
    st = library().hypic_seam_compose(fam, BF16 if dt == torch.bfloat16 else F32, n, w, H, dk, dv,
                                      _ptr(q if want_o else None), _ptr(k), _ptr(v), _ptr(alpha),
                                      _ptr(beta), _ptr(lam), _ptr(M), _ptr(S_prev), _ptr(S_C),
                                      _ptr(S_out), _ptr(o_out if want_o else None), _stream(stream))
    _check("hypic_seam_compose", st)
    res = {"S": S_out}
    if want_o:
        res["o"] = o_out
    return res


def compose_chain_workspace_bytes(family, n_req, n_layers, n_heads, d_k, d_v, max_chain):
    """Scratch bytes hypic_compose_chain_ws needs for this shape (0: no tree)."""
    n = library().hypic_compose_chain_workspace_bytes(_fam(family), n_req, n_layers, n_heads, d_k, d_v,
                                                      max_chain)
    if n < 0:
        raise HypicError("hypic_compose_chain_workspace_bytes", int(n))
    return int(n)


def compose_chain(family, chain_len, seg_idx, pool_lam, pool_S, pool_M=None, S_init=None,
                  S_out=None, d_err=None, stream=None, workspace=None):
    """Fold pool entries seg_idx[r, :chain_len[r]] in order: S <- T_p S + S_p.

    pool_lam [P,Lyr,H] or [P,Lyr,H,dk], pool_M [P,Lyr,H,dk,dk] (dense, kda),
    pool_S [P,Lyr,H,dk,dv], S_init [R,Lyr,H,dk,dv] or None.  Returns S [R,Lyr,H,dk,dv].
    ``workspace`` (a uint8 CUDA tensor, or "auto" to allocate one) selects
    hypic_compose_chain_ws: few long chains fold as a two-level tree.
    """
    fam = _fam(family)
    chain_len = _dev(chain_len, "chain_len", torch.int32)
    seg_idx = _dev(seg_idx, "seg_idx", torch.int32)
    pool_lam = _dev(pool_lam, "pool_lam", torch.float32)
    pool_S = _dev(pool_S, "pool_S", torch.float32)
    pool_M = _dev(pool_M, "pool_M", torch.float32, allow_none=True)
    S_init = _dev(S_init, "S_init", torch.float32, allow_none=True)
    P, Lyr, H, dk, dv = pool_S.shape
    R = chain_len.numel()
    max_chain = seg_idx.shape[1] if seg_idx.dim() == 2 else 0
    if S_out is None:
        S_out = torch.empty((R, Lyr, H, dk, dv), dtype=torch.float32, device=pool_S.device)
    if workspace is None:
        st = library().hypic_compose_chain(fam, R, Lyr, H, dk, dv, max_chain, _ptr(chain_len),
                                           _ptr(seg_idx), P, _ptr(pool_lam), _ptr(pool_M),
                                           _ptr(pool_S), _ptr(S_init), _ptr(S_out), _ptr(d_err),
                                           _stream(stream))
        _check("hypic_compose_chain", st)
        return S_out
    if isinstance(workspace, str):
        need = compose_chain_workspace_bytes(fam, R, Lyr, H, dk, dv, max_chain)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=pool_S.device)
    workspace = _dev(workspace, "workspace", torch.uint8)
    st = library().hypic_compose_chain_ws(fam, R, Lyr, H, dk, dv, max_chain, _ptr(chain_len),
                                          _ptr(seg_idx), P, _ptr(pool_lam), _ptr(pool_M), _ptr(pool_S),
                                          _ptr(S_init), _ptr(S_out), _ptr(workspace), workspace.numel(),
                                          _ptr(d_err), _stream(stream))
    _check("hypic_compose_chain_ws", st)
    return S_out


def selftest_wait(limit_cycles, arrive, d_err=None, cycles=None, stream=None):
    """Run the bounded pipeline wait on its own (hypic_selftest_wait): without
    ``arrive`` the wait gives up after ``limit_cycles`` SM cycles and writes
    HYPIC_ETIMEOUT to ``d_err`` (int32 CUDA tensor); ``cycles`` (int64 CUDA
    tensor) receives the cycles the wait took."""
    d_err = _dev(d_err, "d_err", torch.int32, allow_none=True)
    cycles = _dev(cycles, "cycles", torch.int64, allow_none=True)
    st = library().hypic_selftest_wait(int(limit_cycles), 1 if arrive else 0, _ptr(d_err), _ptr(cycles),
                                       _stream(stream))
    _check("hypic_selftest_wait", st)
