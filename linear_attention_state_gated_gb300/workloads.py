"""Seeded synthetic inputs for the segment scan and composition workloads.

This module holds no arithmetic of the method itself: it only draws random
numbers (numpy PCG64, seeded), shapes them, L2-normalises key/query rows where
a workload asks for it and rounds to bf16 (round-to-nearest-even) where the
workload's inputs are bf16.  Both the CUDA path and the fp64 oracle are fed
from here; every bf16 input is also returned as the float32 array of the
exact bf16 values, so the oracle sees precisely what the GPU sees.

Workloads (sizes as named in the HYPIC evaluation set-up; the pages run a
production RAG trace and public QA/summarisation sets, for which these seeded
draws stand in):

* ``tiny_dense``      -- gated delta rule, fp32, 1 layer, 2 heads, d=32,
                         two 64-token segments, alpha~U(0.9,1), beta~U(0,1).
* ``scalar_diag``     -- 32 heads, d=128, bf16 q/k/v, batch of equal segments;
                         scalar gate gamma_h = 1 - 2^(-5 - 6h/32) for every
                         token, or diagonal gate sigmoid(N(2,1))^(1/16).
* ``dense_stack``     -- gated delta rule on a 30-layer x 32-head x 128 stack,
                         bf16 q, v ~ N(0,1), k L2-normalised,
                         alpha = exp(-0.1 softplus(N(0,1))), beta = sigmoid(N(0,1)).
* ``rag_pool`` / ``rag_requests`` -- a pool of cached (lambda, S) pairs and
                         requests drawing distinct pool entries by truncated
                         Zipf(1.1) weights in random order;
                         ``rag_pool_lengths`` / ``scalar_diag_layer_device``
                         draw the pool's segments themselves (lengths
                         U{1024..4096}, the scalar/diagonal law) on the GPU,
                         to be scanned into the pool.
* ``long_mix``        -- one long prompt split into equal segments, some
                         cached and some not, gated delta rule.
"""
from __future__ import annotations

import os

import numpy as np

SCALAR, DIAG, DENSE, KDA = 0, 1, 2, 3


def rng(seed) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


_BLOCK = 2048          # tokens per independently seeded block
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        _POOL = cf.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 result."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    out = r.view(np.float32)
    nan = np.isnan(x)
    if nan.any():
        out = out.copy()
        out[nan] = np.nan
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _l2_rows(x):
    n = np.sqrt(np.sum(np.square(x, dtype=np.float32), axis=-1, keepdims=True, dtype=np.float32))
    n[n == 0] = 1.0
    return (x / n).astype(np.float32)


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _softplus(x):
    x = x.astype(np.float64)
    return np.where(x > 20, x, np.log1p(np.exp(np.minimum(x, 20))))


def _field(seed: int, field: int, n_layers: int, N: int, tail_shape, make, layers=None):
    """[n_layers or len(layers), N, *tail_shape] float32, filled block by block.

    Block (layer l, tokens [b*_BLOCK, ...)) draws from PCG64 seeded with
    (seed, field, l, b), so the values do not depend on the thread count and
    any layer can be regenerated on its own.  ``make(gen, shape)`` draws one block.
    """
    layers = list(range(n_layers)) if layers is None else list(layers)
    out = np.empty((len(layers), N, *tail_shape), dtype=np.float32)
    nblk = (N + _BLOCK - 1) // _BLOCK

    def job(i, b):
        l = layers[i]
        t0, t1 = b * _BLOCK, min(N, (b + 1) * _BLOCK)
        g = rng([seed, field, l, b])
        out[i, t0:t1] = make(g, (t1 - t0, *tail_shape))

    futs = [_pool().submit(job, i, b) for i in range(len(layers)) for b in range(nblk)]
    for f in futs:
        f.result()
    return out


def _unit_rows_bf16(g, shape):
    return bf16_round(_l2_rows(g.standard_normal(size=shape, dtype=np.float32)))


def _normal_bf16(g, shape):
    return bf16_round(g.standard_normal(size=shape, dtype=np.float32))


def equal_offsets(n_seg: int, length: int) -> np.ndarray:
    return np.arange(n_seg + 1, dtype=np.int64) * length


def _offsets(lengths):
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int64)


def tiny_dense(seed: int = 0, n_seg: int = 2, seg_len: int = 64, H: int = 2, d: int = 32):
    """Gated delta rule, fp32 inputs: k, q L2-normalised N(0,1), v N(0,1),
    alpha ~ U(0.9, 1), beta ~ U(0, 1)."""
    g = rng(seed)
    N = n_seg * seg_len
    k = _l2_rows(g.standard_normal((1, N, H, d), dtype=np.float32))
    q = _l2_rows(g.standard_normal((1, N, H, d), dtype=np.float32))
    v = g.standard_normal((1, N, H, d), dtype=np.float32)
    alpha = g.uniform(0.9, 1.0, size=(1, N, H)).astype(np.float32)
    beta = g.uniform(0.0, 1.0, size=(1, N, H)).astype(np.float32)
    return dict(family=DENSE, dtype="f32", q=q, k=k, v=v, alpha=alpha, beta=beta,
                seg_offsets=equal_offsets(n_seg, seg_len))


def retnet_gamma(H: int) -> np.ndarray:
    """Per-head fixed decay gamma_h = 1 - 2^(-5 - 6h/H) (RetNet-style heads)."""
    h = np.arange(H, dtype=np.float64)
    return (1.0 - np.exp2(-5.0 - 6.0 * h / H)).astype(np.float32)


def _diag_gate(g, shape):
    x = g.standard_normal(size=shape, dtype=np.float32) + np.float32(2.0)
    return (_sigmoid(x) ** np.float32(1.0 / 16.0)).astype(np.float32)


def scalar_diag(family: int, seg_len: int = 512, n_seg: int = 8, H: int = 32, d: int = 128,
                seed: int = 1, with_q: bool = False, n_layers: int = 1, lengths=None,
                layers=None):
    """Scalar (fixed gamma_h per head) or diagonal (per-channel GLA gate) workload.

    k, q: L2-normalised N(0,1) rows, v ~ N(0,1); all bf16.  No beta.
    ``lengths`` overrides the equal segment lengths (ragged batches);
    ``layers`` regenerates only those layers (same values as in the full set).
    """
    if lengths is None:
        lengths = [seg_len] * n_seg
    offs = _offsets(lengths)
    N = int(offs[-1])
    nl = n_layers if layers is None else len(layers)
    k = _field(seed, 1, n_layers, N, (H, d), _unit_rows_bf16, layers)
    v = _field(seed, 2, n_layers, N, (H, d), _normal_bf16, layers)
    q = _field(seed, 3, n_layers, N, (H, d), _unit_rows_bf16, layers) if with_q else None
    if family == SCALAR:
        alpha = np.broadcast_to(retnet_gamma(H)[None, None, :], (nl, N, H)).copy()
    elif family == DIAG:
        alpha = _field(seed, 4, n_layers, N, (H, d), _diag_gate, layers)
    else:
        raise ValueError("scalar_diag: family must be SCALAR or DIAG")
    return dict(family=family, dtype="bf16", q=q, k=k, v=v, alpha=alpha, beta=None,
                seg_offsets=offs)


def _dense_alpha(g, shape):
    return np.exp(-0.1 * _softplus(g.standard_normal(size=shape, dtype=np.float32))).astype(np.float32)


def _dense_beta(g, shape):
    return _sigmoid(g.standard_normal(size=shape, dtype=np.float32))


def dense_stack(seg_len: int = 512, n_layers: int = 30, H: int = 32, d: int = 128, seed: int = 2,
                with_q: bool = False, n_seg: int = 1, lengths=None, layers=None):
    """Gated delta rule: bf16 q, v ~ N(0,1), k L2-normalised; fp32
    alpha = exp(-0.1 softplus(N(0,1))), beta = sigmoid(N(0,1))."""
    if lengths is None:
        lengths = [seg_len] * n_seg
    offs = _offsets(lengths)
    N = int(offs[-1])
    k = _field(seed, 1, n_layers, N, (H, d), _unit_rows_bf16, layers)
    v = _field(seed, 2, n_layers, N, (H, d), _normal_bf16, layers)
    q = _field(seed, 3, n_layers, N, (H, d), _normal_bf16, layers) if with_q else None
    alpha = _field(seed, 4, n_layers, N, (H,), _dense_alpha, layers)
    beta = _field(seed, 5, n_layers, N, (H,), _dense_beta, layers)
    return dict(family=DENSE, dtype="bf16", q=q, k=k, v=v, alpha=alpha, beta=beta,
                seg_offsets=offs)


def kda_stack(seg_len: int = 512, n_layers: int = 30, H: int = 32, d: int = 128, seed: int = 7,
              with_q: bool = False, n_seg: int = 1, lengths=None, layers=None):
    """KDA-style gates: the dense stack's law (bf16 q, v ~ N(0,1), k L2-normalised,
    beta = sigmoid(N(0,1))) with alpha = exp(-0.1 softplus(N(0,1))) drawn per channel."""
    if lengths is None:
        lengths = [seg_len] * n_seg
    offs = _offsets(lengths)
    N = int(offs[-1])
    k = _field(seed, 1, n_layers, N, (H, d), _unit_rows_bf16, layers)
    v = _field(seed, 2, n_layers, N, (H, d), _normal_bf16, layers)
    q = _field(seed, 3, n_layers, N, (H, d), _normal_bf16, layers) if with_q else None
    alpha = _field(seed, 4, n_layers, N, (H, d), _dense_alpha, layers)
    beta = _field(seed, 5, n_layers, N, (H,), _dense_beta, layers)
    return dict(family=KDA, dtype="bf16", q=q, k=k, v=v, alpha=alpha, beta=beta, seg_offsets=offs)


def rag_pool(family: int, P: int = 200, n_layers: int = 30, H: int = 32, d: int = 128,
             seed: int = 3, len_lo: int = 1024, len_hi: int = 4096):
    """Pool of P cached segment pairs (lambda, S) with segment lengths ~ U{len_lo..len_hi}.

    Stands in for scanned pool segments: lambda is drawn per (entry, layer, head)
    with the magnitude a segment of that length has under the scalar/diagonal
    gates of ``scalar_diag`` (lengths x a per-head or per-channel rate), S is
    drawn N(0, 1/d) per entry.  Dense pools also get a transition factor M
    drawn N(0,1/d) and a scalar lambda.  All fp32.
    """
    g = rng(seed)
    lengths = g.integers(len_lo, len_hi + 1, size=P).astype(np.int64)
    if family == SCALAR:
        rate = np.exp2(-5.0 - 6.0 * np.arange(H) / H)
        lam = -(lengths[:, None, None] * rate[None, None, :]) * g.uniform(
            0.95, 1.05, size=(P, n_layers, H))
    elif family == DIAG:
        lam = -lengths[:, None, None, None] * g.uniform(0.005, 0.02, size=(P, n_layers, H, d))
    else:
        lam = -lengths[:, None, None] * g.uniform(0.05, 0.1, size=(P, n_layers, H))
    S = g.standard_normal((P, n_layers, H, d, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
    out = dict(family=family, lengths=lengths, lam=lam.astype(np.float32), S=S)
    if family == DENSE:
        out["M"] = g.standard_normal((P, n_layers, H, d, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
    return out


def rag_requests(R: int = 64, n: int = 20, P: int = 200, zipf_s: float = 1.1, seed: int = 3):
    """R requests, each n distinct pool indices drawn by truncated Zipf(s) weights.

    Ranks i = 1..P carry weight i^-s over a seeded permutation of the pool;
    the prompt order is the draw order.
    """
    g = rng(seed + 1000)
    perm = g.permutation(P)
    w = np.arange(1, P + 1, dtype=np.float64) ** (-zipf_s)
    idx = np.zeros((R, n), dtype=np.int32)
    for r in range(R):
        ranks = g.choice(P, size=n, replace=False, p=w / w.sum())
        idx[r] = perm[ranks]
    return np.full(R, n, dtype=np.int32), idx


def long_mix_split(n_seg: int = 64, n_uncached: int = 16, seed: int = 4):
    """Which segments of the long prompt are uncached: a seeded choice of n_uncached."""
    g = rng(seed + 1000)
    return np.sort(g.permutation(n_seg)[:n_uncached]).astype(np.int64)


def long_mix_layout(n_seg: int = 64, n_layers: int = 30, n_uncached: int = 16, seed: int = 4):
    """Pool rows of the long-context mix with its layers as requests (one chain per
    layer over all 64 segments in prompt order; n_layers = 1 in the chain call).

    The uncached segments are scanned in one call that treats every (layer,
    uncached segment) as a segment of one token array, so their pairs land at rows
    l * n_uncached + u; cached segment c's pairs (one scan call each) at rows
    n_layers * n_uncached + c * n_layers + l.  Returns (uncached, cached, rows) with
    rows[l, s] the pool row of segment s at layer l (int32, the chains' seg_idx).
    """
    unc = [int(x) for x in long_mix_split(n_seg=n_seg, n_uncached=n_uncached, seed=seed)]
    cached = [s for s in range(n_seg) if s not in unc]
    rows = np.empty((n_layers, n_seg), np.int32)
    for u, s in enumerate(unc):
        rows[:, s] = np.arange(n_layers) * len(unc) + u
    for c, s in enumerate(cached):
        rows[:, s] = n_layers * len(unc) + c * n_layers + np.arange(n_layers)
    return unc, cached, rows


def long_mix_uncached_flat(unc, seg_len: int = 2048, n_layers: int = 30, H: int = 32, d: int = 128,
                           seed: int = 4, device="cuda"):
    """The uncached segments' inputs (same draws as ``long_mix_segment_device``) as
    one token array for a single scan call: tokens ordered (layer, uncached segment,
    token), shapes [1, n_layers * len(unc) * seg_len, H, d] (bf16 q, k, v) and
    [1, ..., H] (fp32 alpha, beta); offsets of the n_layers * len(unc) segments."""
    import torch
    n = n_layers * len(unc) * seg_len
    flat = {"k": torch.empty((1, n, H, d), dtype=torch.bfloat16, device=device),
            "v": torch.empty((1, n, H, d), dtype=torch.bfloat16, device=device),
            "q": torch.empty((1, n, H, d), dtype=torch.bfloat16, device=device),
            "alpha": torch.empty((1, n, H), dtype=torch.float32, device=device),
            "beta": torch.empty((1, n, H), dtype=torch.float32, device=device)}
    for u, s in enumerate(unc):
        w = long_mix_segment_device(s, seg_len=seg_len, n_layers=n_layers, H=H, d=d, seed=seed, with_q=True,
                                    device=device)
        for l in range(n_layers):
            a = (l * len(unc) + u) * seg_len
            for key in flat:
                flat[key][0, a:a + seg_len] = w[key][l]
        del w
    offs = np.arange(n_layers * len(unc) + 1, dtype=np.int64) * seg_len
    return flat, offs


def _seed_key(*parts) -> int:
    x = 0
    for p in parts:
        x = (x * 1000003 + int(p)) % (2 ** 63)
    return x


def _dense_layer_device(g, seg_len, H, d, device, with_q):
    """One layer of the gated delta rule's law, drawn from torch generator ``g``."""
    import torch
    k = torch.randn((seg_len, H, d), generator=g, device=device)
    k = (k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(torch.bfloat16)
    v = torch.randn((seg_len, H, d), generator=g, device=device).to(torch.bfloat16)
    q = torch.randn((seg_len, H, d), generator=g, device=device)
    a = torch.randn((seg_len, H), generator=g, device=device)
    alpha = torch.exp(-0.1 * torch.nn.functional.softplus(a))
    beta = torch.sigmoid(torch.randn((seg_len, H), generator=g, device=device))
    return k, v, (q.to(torch.bfloat16) if with_q else None), alpha, beta


def long_mix_segment_device(seg: int, seg_len: int = 2048, n_layers: int = 30, H: int = 32,
                            d: int = 128, seed: int = 4, with_q: bool = True, device="cuda",
                            layers=None, heads=None):
    """One segment of the long-context mix, drawn on the GPU (torch's seeded
    generator; the full prompt is ~72 GB of inputs, too much to draw on the host).

    Gate law of ``dense_stack``: bf16 q, v ~ N(0,1), k L2-normalised N(0,1);
    alpha = exp(-0.1 softplus(N(0,1))), beta = sigmoid(N(0,1)).  Layer l draws
    from a generator seeded with (seed, segment, layer), so any layer (and head
    slice) can be drawn again alone.  Tensors: q, k, v [Lyr, L, H, d] bf16,
    alpha, beta [Lyr, L, H] fp32, contiguous per segment.
    """
    import torch
    layers = list(range(n_layers)) if layers is None else list(layers)
    nl = len(layers)
    out = {"k": torch.empty((nl, seg_len, H, d), dtype=torch.bfloat16, device=device),
           "v": torch.empty((nl, seg_len, H, d), dtype=torch.bfloat16, device=device),
           "alpha": torch.empty((nl, seg_len, H), dtype=torch.float32, device=device),
           "beta": torch.empty((nl, seg_len, H), dtype=torch.float32, device=device)}
    if with_q:
        out["q"] = torch.empty((nl, seg_len, H, d), dtype=torch.bfloat16, device=device)
    for i, l in enumerate(layers):
        g = torch.Generator(device=device)
        g.manual_seed(_seed_key(seed, seg, l))
        k, v, q, alpha, beta = _dense_layer_device(g, seg_len, H, d, device, with_q)
        out["k"][i], out["v"][i], out["alpha"][i], out["beta"][i] = k, v, alpha, beta
        if with_q:
            out["q"][i] = q
    if heads is not None:
        out = {key: t[:, :, heads].contiguous() for key, t in out.items()}
    return out


def dense_stack_device(seg_len: int, n_layers: int = 30, H: int = 32, d: int = 128, seed: int = 2,
                       device="cuda"):
    """The dense stack's law (``dense_stack``) drawn on the GPU, one segment of
    ``seg_len`` tokens per layer, for lengths whose host draw would take minutes
    (30 layers x 32768 tokens x 32 heads x 128 is 4 G values a tensor).  Layer l
    draws from a generator seeded with (seed, 0, l)."""
    return long_mix_segment_device(0, seg_len=seg_len, n_layers=n_layers, H=H, d=d, seed=seed + 1000,
                                   with_q=False, device=device)


def rag_pool_lengths(P: int = 200, len_lo: int = 1024, len_hi: int = 4096, seed: int = 3) -> np.ndarray:
    """Segment lengths of the RAG pool: P seeded draws from U{len_lo..len_hi}."""
    return rng(seed + 2000).integers(len_lo, len_hi + 1, size=P).astype(np.int64)


def scalar_diag_layer_device(family: int, lengths, layer: int, H: int = 32, d: int = 128, seed: int = 3,
                             device="cuda", heads=None):
    """One layer of a packed batch of segments under the scalar/diagonal law of
    ``scalar_diag`` (k L2-normalised N(0,1), v ~ N(0,1), bf16; gamma_h per token,
    or sigmoid(N(2,1))^(1/16) per channel), drawn on the GPU from a generator
    seeded with (seed, family, layer).  Returns k, v [1, N, H, d] bf16, alpha
    [1, N, H] or [1, N, H, d] fp32 and the int64 segment offsets (host)."""
    import torch
    offs = _offsets(list(lengths))
    N = int(offs[-1])
    g = torch.Generator(device=device)
    g.manual_seed(_seed_key(seed, family, layer))
    k = torch.randn((N, H, d), generator=g, device=device)
    k = (k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(torch.bfloat16)
    v = torch.randn((N, H, d), generator=g, device=device).to(torch.bfloat16)
    if family == SCALAR:
        alpha = torch.from_numpy(retnet_gamma(H)).to(device)[None, :].expand(N, H).contiguous()
    elif family == DIAG:
        alpha = torch.sigmoid(torch.randn((N, H, d), generator=g, device=device) + 2.0) ** (1.0 / 16.0)
    else:
        raise ValueError("scalar_diag_layer_device: family must be SCALAR or DIAG")
    if heads is not None:
        k, v, alpha = k[:, heads].contiguous(), v[:, heads].contiguous(), alpha[:, heads].contiguous()
    return k[None], v[None], alpha[None], offs
