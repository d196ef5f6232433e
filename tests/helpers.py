"""Comparison metrics and device marshalling shared by the tests.

Error metrics (per (layer, segment, head) matrix, as the parity contract
states them):
  * state S: relative Frobenius error  ||S_g - S_o||_F / ||S_o||_F
  * transition T_C = exp(lambda) M: relative Frobenius error of the operator
    itself, evaluated without materialising exp(lambda) (which underflows):
      scalar : |exp(lam_g - lam_o) - 1|
      diag   : ||exp(lam_g - m) - exp(lam_o - m)|| / ||exp(lam_o - m)||, m = max lam_o
      dense  : ||exp(lam_g - lam_o) M_g - M_o||_F / ||M_o||_F
"""
from __future__ import annotations

import numpy as np

TOL_SCAN_BF16 = 1e-3     # T_C, S(C|0) from bf16 inputs
TOL_F32 = 1e-5           # fp32 inputs / fp32 composition on identical inputs
# o_t is written in the input dtype: bf16 output rounding alone has rms relative
# error ~1.7e-3 (8-bit significand, round to nearest even); 4e-3 leaves room
# for the fp32 path's own <= 1e-3.
TOL_O_BF16 = 4e-3


def rel_fro(g, o, axes=(-2, -1)):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    num = np.sqrt(np.sum((g - o) ** 2, axis=axes))
    den = np.sqrt(np.sum(o ** 2, axis=axes))
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def t_err(fam, lam_g, lam_o, M_g=None, M_o=None):
    lam_g = np.asarray(lam_g, np.float64)
    lam_o = np.asarray(lam_o, np.float64)
    if fam == 0:
        return np.abs(np.expm1(lam_g - lam_o))
    if fam == 1:
        m = lam_o.max(axis=-1, keepdims=True)
        eo = np.exp(lam_o - m)
        eg = np.exp(lam_g - m)
        return np.sqrt(np.sum((eg - eo) ** 2, -1) / np.sum(eo ** 2, -1))
    sc = np.exp(lam_g - lam_o)[..., None, None]
    return rel_fro(sc * np.asarray(M_g, np.float64), M_o)


def to_dev(x, dtype="f32"):
    import torch
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def to_host(t):
    import torch
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy().astype(np.float64)
