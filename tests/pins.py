"""Pins for the fp64 oracle: each check compares the oracle with something
other than itself -- a value the HYPIC pages print, a closed form, a textbook
special case, a library routine, or exact rational arithmetic on tiny inputs.

Each check raises AssertionError on failure.  ``test_oracle.py`` runs them
one by one; ``test_oracle_mutants.py`` runs them against copies of the oracle
with a planted mistake and expects at least one to fail for every mistake.

Pages cited: [xix-fr] = xix.ai/fr HYPIC article, paragraph on linear layers
("opérateurs de transition"); [remio-ja] = remio.ai/ja HYPIC article, section
"how HYPIC composes states".
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle

SCALAR, DIAG, DENSE, KDA = oracle.SCALAR, oracle.DIAG, oracle.DENSE, oracle.KDA
FAMS = (SCALAR, DIAG, DENSE, KDA)
PER_CH = (DIAG, KDA)      # a gate per channel
WITH_M = (DENSE, KDA)     # operator kept as exp(lambda) * M
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

TOL = 1e-12


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def _inputs(fam, Lyr, N, H, dk, dv, seed, beta=True, q=False, alpha_lo=0.8):
    g = np.random.default_rng(seed)
    k = g.standard_normal((Lyr, N, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = g.standard_normal((Lyr, N, H, dv))
    ash = (Lyr, N, H, dk) if fam in PER_CH else (Lyr, N, H)
    alpha = g.uniform(alpha_lo, 1.0, size=ash)
    b = g.uniform(0.1, 1.0, size=(Lyr, N, H)) if beta else None
    qq = g.standard_normal((Lyr, N, H, dk)) if q else None
    return k, v, alpha, b, qq


def token_T(fam, a, b, k):
    """Per-token transition matrix: alpha I, diag(alpha), alpha (I - beta k k^T) or
    diag(alpha) (I - beta k k^T)."""
    d = k.shape[0]
    if fam == SCALAR:
        return a * np.eye(d)
    if fam == DIAG:
        return np.diag(a)
    if fam == KDA:
        return np.diag(a) @ (np.eye(d) - b * np.outer(k, k))
    return a * (np.eye(d) - b * np.outer(k, k))


def _head(arr, l, h):
    return None if arr is None else arr[l, :, h]


def unrolled(fam, k, v, alpha, beta):
    """Definition written out for one head (arrays over tokens):
    T_C = T_L ... T_1 (ordered product) and
    S_t = sum_{s<=t} (T_t ... T_{s+1}) beta_s k_s v_s^T for every t."""
    L, dk = k.shape
    beta = np.ones(L) if beta is None else beta
    Ts = [token_T(fam, alpha[t], beta[t], k[t]) for t in range(L)]
    T = np.eye(dk)
    for t in range(L):
        T = Ts[t] @ T
    states = []
    for t in range(L):
        St = np.zeros((dk, v.shape[1]))
        for s in range(t + 1):
            P = np.eye(dk)
            for r in range(s + 1, t + 1):
                P = Ts[r] @ P
            St += P @ (beta[s] * np.outer(k[s], v[s]))
        states.append(St)
    return T, states


# ---------------------------------------------------------------- pins ----

def check_transition_is_ordered_product():
    """[xix-fr]: T_C is the product of the per-token transitions of the segment."""
    for fam in FAMS:
        k, v, alpha, beta, _ = _inputs(fam, 1, 13, 2, 6, 4, seed=10 + fam)
        out = oracle.sequential(fam, k, v, alpha, beta)
        for h in range(2):
            T, _ = unrolled(fam, k[0, :, h], v[0, :, h], _head(alpha, 0, h), _head(beta, 0, h))
            if fam in WITH_M:
                Tg = np.exp(out["lam"][0, h]) * out["M"][0, h]
                assert rel(Tg, T) < TOL, ("T_C", rel(Tg, T))
                assert abs(np.max(np.abs(out["M"][0, h])) - 1.0) < 1e-15
            elif fam == DIAG:
                assert rel(np.diag(np.exp(out["lam"][0, h])), T) < TOL
            else:
                assert rel(np.exp(out["lam"][0, h]) * np.eye(6), T) < TOL


def check_state_and_output_unrolled():
    """S(C|0) and o_t = S_t^T q_t against the unrolled sum definition."""
    for fam in FAMS:
        k, v, alpha, beta, q = _inputs(fam, 1, 11, 2, 5, 3, seed=20 + fam, q=True)
        out = oracle.sequential(fam, k, v, alpha, beta, q=q, want_o=True)
        for h in range(2):
            _, states = unrolled(fam, k[0, :, h], v[0, :, h], _head(alpha, 0, h), _head(beta, 0, h))
            assert rel(out["S"][0, h], states[-1]) < TOL, ("S", fam)
            o_ref = np.stack([states[t].T @ q[0, t, h] for t in range(11)])
            assert rel(out["o"][0, :, h], o_ref) < TOL, ("o", fam)


def check_composition_identity():
    """[xix-fr]: S(C1.C2) = T(C2) S(C1) + S(C2) equals the straight recurrence;
    T(C1.C2) = T(C2) T(C1).  Ragged segments, non-square state."""
    for fam in FAMS:
        n1, n2 = 7, 12
        k, v, alpha, beta, _ = _inputs(fam, 2, n1 + n2, 3, 6, 4, seed=30 + fam)
        seg = oracle.segment_scan(fam, k, v, alpha, [0, n1, n1 + n2], beta)
        whole = oracle.sequential(fam, k, v, alpha, beta)
        c1 = {key: a[:, 0] for key, a in seg.items()}
        c2 = {key: a[:, 1] for key, a in seg.items()}
        comp = oracle.compose(fam, c2["lam"], c2["S"], S_prev=c1["S"], M=c2.get("M"),
                              lam_prev=c1["lam"], M_prev=c1.get("M"))
        assert rel(comp["S"], whole["S"]) < TOL, ("S", fam, rel(comp["S"], whole["S"]))
        if fam in WITH_M:
            Tg = np.exp(comp["lam"])[..., None, None] * comp["M"]
            Tw = np.exp(whole["lam"])[..., None, None] * whole["M"]
            assert rel(Tg, Tw) < TOL
        else:
            assert np.max(np.abs(comp["lam"] - whole["lam"])) < TOL * 100


def check_scalar_closed_form():
    """Scalar family collapses to a product of decays: lambda = L log gamma,
    T_C = gamma^L, S = K^T diag(beta_s gamma^(L-s)) V (numpy matmul)."""
    g = np.random.default_rng(40)
    L, dk, dv = 37, 8, 5
    gamma = 1.0 - 2.0 ** -6
    k = g.standard_normal((1, L, 1, dk))
    v = g.standard_normal((1, L, 1, dv))
    beta = g.uniform(0, 1, size=(1, L, 1))
    alpha = np.full((1, L, 1), gamma)
    out = oracle.sequential(SCALAR, k, v, alpha, beta)
    assert abs(out["lam"][0, 0] - L * np.log(gamma)) < 1e-12
    assert abs(np.exp(out["lam"][0, 0]) - gamma ** L) < 1e-14
    w = beta[0, :, 0] * gamma ** (L - 1 - np.arange(L))
    S_ref = k[0, :, 0].T @ (w[:, None] * v[0, :, 0])
    assert rel(out["S"][0, 0], S_ref) < TOL


def check_diag_closed_form():
    """Diagonal gates act per key channel: S[i,:] = sum_s prod_{r>s} alpha_{r,i}
    beta_s k_{s,i} v_s; lambda_i = sum_t log alpha_{t,i}.  Equal channels give the
    scalar family."""
    k, v, alpha, beta, _ = _inputs(DIAG, 1, 15, 1, 6, 4, seed=50)
    out = oracle.sequential(DIAG, k, v, alpha, beta)
    a = alpha[0, :, 0]                                     # [L, dk]
    logs = np.log(a)
    suffix = np.cumsum(logs[::-1], axis=0)[::-1] - logs   # sum_{r>s} log alpha_r
    w = np.exp(suffix) * beta[0, :, 0][:, None]           # [L, dk]
    S_ref = np.einsum("si,si,sj->ij", w, k[0, :, 0], v[0, :, 0])
    assert rel(out["S"][0, 0], S_ref) < TOL
    assert np.max(np.abs(out["lam"][0, 0] - logs.sum(0))) < 1e-12
    # equal channels == scalar
    a_s = alpha[..., 0]
    eq = np.repeat(a_s[..., None], 6, axis=-1)
    o_d = oracle.sequential(DIAG, k, v, eq, beta)
    o_s = oracle.sequential(SCALAR, k, v, a_s, beta)
    assert rel(o_d["S"], o_s["S"]) < TOL
    assert np.max(np.abs(o_d["lam"][..., 0] - o_s["lam"])) < 1e-12


def check_beta_zero_is_pure_decay():
    """beta = 0 turns the delta rule into pure decay: M = I, lambda = sum log alpha, S = 0."""
    k, v, alpha, _, _ = _inputs(DENSE, 1, 9, 2, 5, 3, seed=60)
    beta = np.zeros((1, 9, 2))
    out = oracle.sequential(DENSE, k, v, alpha, beta)
    assert np.max(np.abs(out["M"] - np.eye(5))) == 0.0
    assert np.max(np.abs(out["lam"][0] - np.log(alpha[0]).sum(0))) < 1e-12
    assert np.max(np.abs(out["S"])) == 0.0


def check_naive_add_plain_linear_attention():
    """[xix-fr]: adding zero-start states is valid for plain linear attention
    (no decay, no delta); then S = K^T V (numpy matmul)."""
    g = np.random.default_rng(70)
    n1, n2, dk, dv = 10, 14, 6, 4
    k = g.standard_normal((1, n1 + n2, 2, dk))
    v = g.standard_normal((1, n1 + n2, 2, dv))
    alpha = np.ones((1, n1 + n2, 2))
    seg = oracle.segment_scan(SCALAR, k, v, alpha, [0, n1, n1 + n2])
    whole = oracle.sequential(SCALAR, k, v, alpha)
    assert rel(seg["S"][:, 0] + seg["S"][:, 1], whole["S"]) < TOL
    for h in range(2):
        assert rel(whole["S"][0, h], k[0, :, h].T @ v[0, :, h]) < TOL
    assert np.max(np.abs(whole["lam"])) == 0.0


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(None, 1)
            vals[key] = float(val)
    return vals


def check_naive_add_retnet_22_percent():
    """[xix-fr]: omitting T(C2) costs 22 % of the state norm after 256 tokens on a
    slow-decay RetNet head.  With gamma = 1 - 2^-10 the error is exactly
    (1 - gamma^256) ||S(C1)||; the pages print it rounded to 0.22."""
    gd = read_golden("naive_add_retnet.txt")
    gamma, n2 = gd["gamma"], int(gd["c2_tokens"])
    g = np.random.default_rng(80)
    n1, dk, dv = 300, 16, 16
    N = n1 + n2
    k = g.standard_normal((1, N, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = g.standard_normal((1, N, 1, dv))
    alpha = np.full((1, N, 1), gamma)
    seg = oracle.segment_scan(SCALAR, k, v, alpha, [0, n1, N])
    whole = oracle.sequential(SCALAR, k, v, alpha)
    naive = seg["S"][:, 0] + seg["S"][:, 1]
    err = np.linalg.norm(naive - whole["S"]) / np.linalg.norm(seg["S"][:, 0])
    assert abs(err - (1.0 - gamma ** n2)) < 1e-12, err
    assert abs(err - gd["relative_error"]) <= gd["rounding"], err


def check_associativity_and_linearity():
    """Composition is associative (with T composed as T(C2) T(C1)) and affine in S_prev."""
    for fam in FAMS:
        n = [5, 8, 6]
        offs = np.concatenate([[0], np.cumsum(n)])
        k, v, alpha, beta, _ = _inputs(fam, 1, sum(n), 2, 5, 3, seed=90 + fam)
        seg = oracle.segment_scan(fam, k, v, alpha, offs, beta)
        A, B, C = ({key: a[:, i] for key, a in seg.items()} for i in range(3))

        def comp(x, y):   # x then y
            r = oracle.compose(fam, y["lam"], y["S"], S_prev=x["S"], M=y.get("M"),
                               lam_prev=x["lam"], M_prev=x.get("M"))
            return r

        left = comp(comp(A, B), C)
        right = comp(A, comp(B, C))
        assert rel(left["S"], right["S"]) < TOL
        if fam in WITH_M:
            tl = np.exp(left["lam"])[..., None, None] * left["M"]
            tr = np.exp(right["lam"])[..., None, None] * right["M"]
            assert rel(tl, tr) < TOL
        g = np.random.default_rng(99)
        X = g.standard_normal(A["S"].shape)
        Y = g.standard_normal(A["S"].shape)
        a, b = 0.7, -1.9

        def app(Sp):
            return oracle.compose(fam, B["lam"], B["S"], S_prev=Sp, M=B.get("M"))["S"]

        lhs = app(a * X + b * Y) - B["S"]
        rhs = a * (app(X) - B["S"]) + b * (app(Y) - B["S"])
        assert rel(lhs, rhs) < 1e-12
        zero = oracle.compose(fam, B["lam"], B["S"], S_prev=None, M=B.get("M"))["S"]
        assert np.array_equal(zero, B["S"])


def check_one_token():
    """One token: T = alpha (I - beta k k^T), S = beta k v^T (dense)."""
    g = np.random.default_rng(100)
    dk, dv = 7, 3
    k = g.standard_normal((1, 1, 1, dk))
    k /= np.linalg.norm(k)
    v = g.standard_normal((1, 1, 1, dv))
    alpha, beta = np.array([[[0.93]]]), np.array([[[0.41]]])
    out = oracle.sequential(DENSE, k, v, alpha, beta)
    T = np.exp(out["lam"][0, 0]) * out["M"][0, 0]
    kk = k[0, 0, 0]
    assert rel(T, 0.93 * (np.eye(dk) - 0.41 * np.outer(kk, kk))) < TOL
    assert rel(out["S"][0, 0], 0.41 * np.outer(kk, v[0, 0, 0])) < TOL


def check_delta_rule_textbook():
    """Delta rule with alpha = beta = 1: reading the state at the key just
    written returns its value (S_t^T k_t = v_t); with orthonormal keys the
    erasures annihilate, prod (I - k k^T) = 0, and S = K^T V."""
    g = np.random.default_rng(110)
    dk, dv = 6, 4
    Q, _ = np.linalg.qr(g.standard_normal((dk, dk)))
    keys = Q.T                                    # rows orthonormal
    k = keys[None, :, None, :]
    v = g.standard_normal((1, dk, 1, dv))
    ones = np.ones((1, dk, 1))
    out = oracle.sequential(DENSE, k, v, ones, ones, q=k, want_o=True)
    assert rel(out["o"][0, :, 0], v[0, :, 0]) < 1e-12
    T = np.exp(out["lam"][0, 0]) * out["M"][0, 0]
    assert np.max(np.abs(T)) < 1e-12
    assert rel(out["S"][0, 0], keys.T @ v[0, :, 0]) < 1e-12
    # random (non-orthogonal) unit keys: read-back still returns the value just written
    k2 = g.standard_normal((1, 20, 1, dk))
    k2 /= np.linalg.norm(k2, axis=-1, keepdims=True)
    v2 = g.standard_normal((1, 20, 1, dv))
    o2 = oracle.sequential(DENSE, k2, v2, np.ones((1, 20, 1)), np.ones((1, 20, 1)),
                           q=k2, want_o=True)
    assert rel(o2["o"][0, :, 0], v2[0, :, 0]) < 1e-12


def check_causal_linear_attention_textbook():
    """Scalar family with alpha = 1: o = tril(Q K^T) V (causal linear attention)."""
    g = np.random.default_rng(120)
    L, dk, dv = 17, 5, 6
    k = g.standard_normal((1, L, 1, dk))
    v = g.standard_normal((1, L, 1, dv))
    q = g.standard_normal((1, L, 1, dk))
    out = oracle.sequential(SCALAR, k, v, np.ones((1, L, 1)), q=q, want_o=True)
    A = np.tril(q[0, :, 0] @ k[0, :, 0].T)
    assert rel(out["o"][0, :, 0], A @ v[0, :, 0]) < TOL


def _frac_unrolled(fam, k, v, alpha, beta, q):
    """Exact rational arithmetic: T_C = T_L...T_1, S_t by the unrolled sum, o_t = S_t^T q_t."""
    L, dk, dv = len(k), len(k[0]), len(v[0])

    def eye():
        return [[Fraction(int(i == j)) for j in range(dk)] for i in range(dk)]

    def mm(A, B):
        return [[sum((A[i][r] * B[r][j] for r in range(len(B))), Fraction(0))
                 for j in range(len(B[0]))] for i in range(len(A))]

    def tok(t):
        if fam == SCALAR:
            return [[alpha[t] if i == j else Fraction(0) for j in range(dk)] for i in range(dk)]
        if fam == DIAG:
            return [[alpha[t][i] if i == j else Fraction(0) for j in range(dk)] for i in range(dk)]
        if fam == KDA:
            return [[alpha[t][i] * (Fraction(int(i == j)) - beta[t] * k[t][i] * k[t][j])
                     for j in range(dk)] for i in range(dk)]
        return [[alpha[t] * (Fraction(int(i == j)) - beta[t] * k[t][i] * k[t][j])
                 for j in range(dk)] for i in range(dk)]

    Ts = [tok(t) for t in range(L)]
    T = eye()
    for t in range(L):
        T = mm(Ts[t], T)
    outs = []
    S = None
    for t in range(L):
        S = [[Fraction(0)] * dv for _ in range(dk)]
        for s in range(t + 1):
            P = eye()
            for r in range(s + 1, t + 1):
                P = mm(Ts[r], P)
            kv = [[beta[s] * k[s][i] * v[s][j] for j in range(dv)] for i in range(dk)]
            PK = mm(P, kv)
            S = [[S[i][j] + PK[i][j] for j in range(dv)] for i in range(dk)]
        outs.append([sum((S[i][j] * q[t][i] for i in range(dk)), Fraction(0)) for j in range(dv)])
    return T, S, outs


def check_brute_force_rational():
    """Tiny inputs in exact rational arithmetic (Python fractions), all families."""
    g = np.random.default_rng(130)
    L, dk, dv = 6, 3, 2

    def rnd(lo, hi):
        return Fraction(int(g.integers(lo, hi)), 16)

    for fam in FAMS:
        k = [[rnd(-16, 17) for _ in range(dk)] for _ in range(L)]
        v = [[rnd(-32, 33) for _ in range(dv)] for _ in range(L)]
        q = [[rnd(-16, 17) for _ in range(dk)] for _ in range(L)]
        beta = [rnd(1, 17) for _ in range(L)]
        if fam in PER_CH:
            alpha = [[rnd(8, 17) for _ in range(dk)] for _ in range(L)]
        else:
            alpha = [rnd(8, 17) for _ in range(L)]
        T, S, o = _frac_unrolled(fam, k, v, alpha, beta, q)
        f = lambda x: np.array(x, dtype=np.float64)  # noqa: E731
        kk, vv, qq = f(k)[None, :, None], f(v)[None, :, None], f(q)[None, :, None]
        aa = f(alpha)[None, :, None]
        bb = f(beta)[None, :, None]
        out = oracle.sequential(fam, kk, vv, aa, bb, q=qq, want_o=True)
        Tref = np.array([[float(x) for x in row] for row in T])
        if fam in WITH_M:
            Tg = np.exp(out["lam"][0, 0]) * out["M"][0, 0]
        elif fam == DIAG:
            Tg = np.diag(np.exp(out["lam"][0, 0]))
        else:
            Tg = np.exp(out["lam"][0, 0]) * np.eye(dk)
        assert rel(Tg, Tref) < TOL, ("T", fam)
        assert rel(out["S"][0, 0], np.array([[float(x) for x in r] for r in S])) < TOL
        assert rel(out["o"][0, :, 0], np.array([[float(x) for x in r] for r in o])) < TOL


def check_chain_equals_sequential():
    """[xix-fr] "under any prefix" / [remio-ja] combine: folding cached pairs in
    any order equals the straight recurrence over the tokens in that order."""
    for fam in FAMS:
        lens = [4, 9, 6, 3, 7]
        P = len(lens)
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        Lyr, H, dk, dv = 2, 2, 5, 3
        k, v, alpha, beta, _ = _inputs(fam, Lyr, int(offs[-1]), H, dk, dv, seed=140 + fam)
        pool = oracle.segment_scan(fam, k, v, alpha, offs, beta)
        # pool arrays [Lyr, P, ...] -> [P, Lyr, ...]
        pl = np.moveaxis(pool["lam"], 1, 0)
        pS = np.moveaxis(pool["S"], 1, 0)
        pM = np.moveaxis(pool["M"], 1, 0) if fam in WITH_M else None
        orders = np.array([[3, 0, 4, 1], [2, 2, 1, 0], [4, 3, 0, 0]], dtype=np.int32)
        chain_len = np.array([4, 3, 2], dtype=np.int32)
        # request 1 starts from the state of a prefix (segment 1 scanned alone)
        S_init = np.zeros((3, Lyr, H, dk, dv))
        S_init[1] = pS[1]
        got = oracle.compose_chain(fam, chain_len, orders, pl, pS, pool_M=pM, S_init=S_init)
        for r in range(3):
            segs = ([1] if r == 1 else []) + list(orders[r, :chain_len[r]])
            idx = np.concatenate([np.arange(offs[s], offs[s + 1]) for s in segs])
            kk, vv = k[:, idx], v[:, idx]
            aa = alpha[:, idx]
            bb = None if beta is None else beta[:, idx]
            ref = oracle.sequential(fam, kk, vv, aa, bb)
            assert rel(got[r], ref["S"]) < TOL, (fam, r, rel(got[r], ref["S"]))


def check_segment_independence():
    """[xix-fr]: T_C and S(C|0) depend only on the segment's own tokens -- scanning
    a segment alone or inside a batch gives the same bits."""
    for fam in FAMS:
        lens = [5, 0, 8, 3]
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        k, v, alpha, beta, _ = _inputs(fam, 1, int(offs[-1]), 2, 4, 3, seed=150 + fam)
        batch = oracle.segment_scan(fam, k, v, alpha, offs, beta)
        for s in range(len(lens)):
            sl = slice(offs[s], offs[s + 1])
            alone = oracle.segment_scan(fam, k[:, sl], v[:, sl], alpha[:, sl], [0, lens[s]],
                                        None if beta is None else beta[:, sl])
            for key in alone:
                assert np.array_equal(alone[key][:, 0], batch[key][:, s]), (fam, s, key)
        # the empty segment: lambda = 0, M = I, S = 0
        assert np.all(batch["S"][:, 1] == 0) and np.all(batch["lam"][:, 1] == 0)
        if fam in WITH_M:
            assert np.array_equal(batch["M"][0, 1, 0], np.eye(4))


def _seam_inputs(fam, n_pre, w, n_body, H, dk, dv, seed):
    """One layer of tokens laid out as prefix | seam window | rest of the segment."""
    N = n_pre + w + n_body
    k, v, alpha, beta, q = _inputs(fam, 1, N, H, dk, dv, seed=seed, q=True)
    return k, v, alpha, beta, q, slice(0, n_pre), slice(n_pre, n_pre + w), slice(n_pre + w, N)


def check_seam_window_equals_sequential():
    """[xix-fr], paragraph on full-attention layers: the first w tokens of a
    reused segment are recomputed at reuse under the full prefix -- the linear
    layers advance the running state through them and hand up each one's
    output -- and the rest of the segment enters by its cached pair.  State
    after the segment and seam outputs equal the straight recurrence over
    prefix + segment; the outputs also equal the unrolled definition."""
    for fam in FAMS:
        n_pre, w, n_body, H, dk, dv = 5, 3, 6, 2, 5, 4
        k, v, alpha, beta, q, pre, seam, body = _seam_inputs(fam, n_pre, w, n_body, H, dk, dv, 170 + fam)
        whole = oracle.sequential(fam, k, v, alpha, beta, q=q, want_o=True)
        S_prev = oracle.sequential(fam, k[:, pre], v[:, pre], alpha[:, pre], beta[:, pre])["S"]
        cached = oracle.sequential(fam, k[:, body], v[:, body], alpha[:, body], beta[:, body])
        got = oracle.seam_compose(fam, k[:, seam], v[:, seam], alpha[:, seam], cached["lam"], cached["S"],
                                  S_prev=S_prev, M=cached.get("M"), beta=beta[:, seam], q=q[:, seam],
                                  want_o=True)
        assert rel(got["S"], whole["S"]) < TOL, ("S", fam, rel(got["S"], whole["S"]))
        assert rel(got["o"], whole["o"][:, seam]) < TOL, ("o", fam)
        for h in range(H):
            idx = slice(0, n_pre + w)
            _, states = unrolled(fam, k[0, idx, h], v[0, idx, h], _head(alpha, 0, h)[idx],
                                 _head(beta, 0, h)[idx])
            o_ref = np.stack([states[n_pre + t].T @ q[0, n_pre + t, h] for t in range(w)])
            assert rel(got["o"][0, :, h], o_ref) < TOL, ("o unrolled", fam, h)
        # no seam window: plain composition; no previous state: the window from zero
        plain = oracle.seam_compose(fam, k[:, :0], v[:, :0], alpha[:, :0], cached["lam"], cached["S"],
                                    S_prev=S_prev, M=cached.get("M"))
        ref = oracle.compose(fam, cached["lam"], cached["S"], S_prev=S_prev, M=cached.get("M"))
        assert rel(plain["S"], ref["S"]) < TOL, ("w = 0", fam)


def check_seam_window_pure_decay_closed_form():
    """beta = 0 inside the window: the state only decays, S_t = (prod_{s<=t} alpha_s) S_prev,
    so o_t = (prod alpha) S_prev^T q_t and S_out = T_body (prod alpha) S_prev + S_body,
    written out with numpy products."""
    g = np.random.default_rng(181)
    n, w, H, dk, dv = 2, 4, 2, 5, 3
    for fam in FAMS:
        k = g.standard_normal((n, w, H, dk))
        v = g.standard_normal((n, w, H, dv))
        q = g.standard_normal((n, w, H, dk))
        alpha = g.uniform(0.7, 1.0, size=(n, w, H, dk) if fam in PER_CH else (n, w, H))
        beta = np.zeros((n, w, H))
        S_prev = g.standard_normal((n, H, dk, dv))
        S_C = g.standard_normal((n, H, dk, dv))
        lam = -g.uniform(0.0, 2.0, size=(n, H, dk) if fam == DIAG else (n, H))
        M = g.standard_normal((n, H, dk, dk)) if fam in WITH_M else None
        got = oracle.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M, beta=beta, q=q,
                                  want_o=True)
        for i in range(n):
            for h in range(H):
                S = S_prev[i, h].copy()
                for t in range(w):
                    a = alpha[i, t, h]
                    S = (a[:, None] if fam in PER_CH else a) * S
                    assert rel(got["o"][i, t, h], S.T @ q[i, t, h]) < TOL, ("o", fam, i, t, h)
                if fam in WITH_M:
                    Sref = np.exp(lam[i, h]) * (M[i, h] @ S) + S_C[i, h]
                elif fam == DIAG:
                    Sref = np.exp(lam[i, h])[:, None] * S + S_C[i, h]
                else:
                    Sref = np.exp(lam[i, h]) * S + S_C[i, h]
                assert rel(got["S"][i, h], Sref) < TOL, ("S", fam, i, h)


def check_kda_with_one_gate_is_dense():
    """KDA (a gate per channel) with every channel's gate equal to one value is the
    gated delta rule: same state, outputs and operator as the dense family."""
    k, v, alpha, beta, q = _inputs(KDA, 1, 17, 2, 6, 4, seed=190, q=True)
    one = np.ascontiguousarray(alpha[..., 0])
    same = np.repeat(one[..., None], 6, axis=-1)
    kda = oracle.sequential(KDA, k, v, same, beta, q=q, want_o=True)
    dense = oracle.sequential(DENSE, k, v, one, beta, q=q, want_o=True)
    assert rel(kda["S"], dense["S"]) < TOL and rel(kda["o"], dense["o"]) < TOL
    Tk = np.exp(kda["lam"])[..., None, None] * kda["M"]
    Td = np.exp(dense["lam"])[..., None, None] * dense["M"]
    assert rel(Tk, Td) < TOL


def check_kda_without_erasure_is_per_channel_decay():
    """beta = 0: nothing is written or erased, and T_C is diag(prod_t alpha_t), the
    diagonal family's operator (closed form)."""
    k, v, alpha, _, _ = _inputs(KDA, 1, 12, 2, 5, 3, seed=191)
    beta = np.zeros(alpha.shape[:3])
    out = oracle.sequential(KDA, k, v, alpha, beta)
    assert np.all(out["S"] == 0)
    T = np.exp(out["lam"])[..., None, None] * out["M"]
    for h in range(2):
        assert rel(T[0, h], np.diag(np.prod(alpha[0, :, h], axis=0))) < TOL


def _operator(fam, out, dk):
    """T = exp(lambda) M (dense, kda), diag(exp(lambda)) or exp(lambda) I, per (.., head)."""
    if fam in WITH_M:
        return np.exp(out["lam"])[..., None, None] * out["M"]
    if fam == DIAG:
        return np.exp(out["lam"])[..., :, None] * np.eye(dk)
    return np.exp(out["lam"])[..., None, None] * np.eye(dk)


def check_composed_prefix_equals_concatenation():
    """[xix-fr] T(C1.C2) = T(C2) T(C1): an ordered group of cached pairs composes
    into the pair of the concatenated tokens (operator and zero-start state), and
    that pair, cached, stands in for its members in later chains."""
    for fam in FAMS:
        lens = [5, 8, 3, 6]
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        Lyr, H, dk, dv = 2, 2, 4, 3
        k, v, alpha, beta, _ = _inputs(fam, Lyr, int(offs[-1]), H, dk, dv, seed=200 + fam)
        pool = oracle.segment_scan(fam, k, v, alpha, offs, beta)
        pl, pS = np.moveaxis(pool["lam"], 1, 0), np.moveaxis(pool["S"], 1, 0)
        pM = np.moveaxis(pool["M"], 1, 0) if fam in WITH_M else None
        groups = np.array([[2, 0, 3], [1, 1, 0], [3, 0, 0]], dtype=np.int32)
        glen = np.array([3, 2, 0], dtype=np.int32)
        got = oracle.compose_prefix(fam, glen, groups, pl, pS, pool_M=pM)
        for r in range(3):
            idx = [i for s in groups[r, :glen[r]] for i in range(offs[s], offs[s + 1])]
            ref = oracle.sequential(fam, k[:, idx], v[:, idx], alpha[:, idx],
                                    None if beta is None else beta[:, idx])
            assert rel(got["S"][r], ref["S"]) < TOL, (fam, r)
            Tg = _operator(fam, {key: a[r] for key, a in got.items()}, dk)
            Tw = _operator(fam, ref, dk)
            assert rel(Tg, Tw) < TOL, (fam, r, "T")
        # the cached prefix of group 0 as a pool entry: [prefix, 1] == [2, 0, 3, 1]
        P = pS.shape[0]
        ext = lambda a, b: np.concatenate([a, b[None]], axis=0)   # noqa: E731
        pl2, pS2 = ext(pl, got["lam"][0]), ext(pS, got["S"][0])
        pM2 = ext(pM, got["M"][0]) if fam in WITH_M else None
        S_a = oracle.compose_chain(fam, [2], [[P, 1]], pl2, pS2, pool_M=pM2)
        S_b = oracle.compose_chain(fam, [4], [[2, 0, 3, 1]], pl, pS, pool_M=pM)
        assert rel(S_a, S_b) < TOL, (fam, "reuse")


ALL_CHECKS = [
    check_transition_is_ordered_product,
    check_state_and_output_unrolled,
    check_composition_identity,
    check_scalar_closed_form,
    check_diag_closed_form,
    check_beta_zero_is_pure_decay,
    check_naive_add_plain_linear_attention,
    check_naive_add_retnet_22_percent,
    check_associativity_and_linearity,
    check_one_token,
    check_delta_rule_textbook,
    check_causal_linear_attention_textbook,
    check_brute_force_rational,
    check_chain_equals_sequential,
    check_segment_independence,
    check_seam_window_equals_sequential,
    check_seam_window_pure_decay_closed_form,
    check_kda_with_one_gate_is_dense,
    check_kda_without_erasure_is_per_channel_decay,
    check_composed_prefix_equals_concatenation,
]
