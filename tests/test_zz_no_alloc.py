"""hypic_segment_scan_static: the two-pass dense scan out of the library's fixed
device scratch (no allocation inside the call).  Its results must equal the
caller-workspace form, hypic_segment_scan_ws, bit for bit, on two calls in a
row (the second call finds the first one's records in the scratch), and the
calls must leave both the caller's allocator and the device's free memory
untouched; a problem larger than the scratch, or another family or input type,
is refused before any launch; a batch of empty segments needs no scratch."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _inputs(lengths, n_layers, H, seed):
    import torch
    from linear_attention_state_gated_gb300 import workloads as wl
    w = wl.dense_stack(lengths=lengths, n_layers=n_layers, H=H, d=128, seed=seed)
    dev = torch.device("cuda")
    return (torch.from_numpy(w["k"]).to(torch.bfloat16).to(dev),
            torch.from_numpy(w["v"]).to(torch.bfloat16).to(dev),
            torch.from_numpy(w["alpha"]).to(dev), torch.from_numpy(w["beta"]).to(dev),
            torch.from_numpy(w["seg_offsets"]).to(dev))


def _nan_out(Lyr, n_seg, H):
    import torch
    f = dict(dtype=torch.float32, device="cuda")
    return {"lam": torch.full((Lyr, n_seg, H), float("nan"), **f),
            "M": torch.full((Lyr, n_seg, H, 128, 128), float("nan"), **f),
            "S": torch.full((Lyr, n_seg, H, 128, 128), float("nan"), **f)}


def test_static_scratch_equals_workspace_form_on_two_calls_in_a_row():
    import torch
    import linear_attention_state_gated_gb300 as hy
    lengths, Lyr, H = [2048, 700, 129], 2, 4
    k, v, a, b, offs = _inputs(lengths, Lyr, H, seed=31)
    need = hy.segment_scan_workspace_bytes("dense", torch.bfloat16, Lyr, len(lengths), k.shape[1], H, 128, 128)
    assert 0 < need <= 64 << 20
    ref = hy.segment_scan("dense", k, v, a, offs, beta=b, workspace="auto")
    outs = [_nan_out(Lyr, len(lengths), H) for _ in range(2)]
    torch.cuda.synchronize()
    allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for out in outs:
        hy.segment_scan_static(k, v, a, offs, out, beta=b)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    hy.segment_scan_static(k, v, a, offs, outs[1], beta=b)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
    assert torch.cuda.mem_get_info()[0] == free1
    for out in outs:
        for key in ("lam", "M", "S"):
            assert torch.equal(out[key], ref[key]), key


def test_static_scratch_refuses_a_problem_beyond_its_size():
    import torch
    import linear_attention_state_gated_gb300 as hy
    Lyr, H, L = 1, 32, 8192           # 32 x 129 records of 49424 bytes: 204.0 MB > 64 MiB
    k, v, a, b, offs = _inputs([L], Lyr, H, seed=32)
    out = _nan_out(Lyr, 1, H)
    with pytest.raises(hy.HypicError) as e:
        hy.segment_scan_static(k, v, a, offs, out, beta=b)
    assert e.value.status == -2
    torch.cuda.synchronize()
    assert torch.isnan(out["S"]).all() and torch.isnan(out["lam"]).all()


def test_static_scratch_refuses_other_families_and_types():
    import torch
    import linear_attention_state_gated_gb300 as hy
    lib = hy.library()
    k, v, a, b, offs = _inputs([256], 1, 2, seed=33)
    out = _nan_out(1, 1, 2)
    P = hy._ptr
    for fam, dt in ((hy.SCALAR, hy.BF16), (hy.DIAG, hy.BF16), (hy.KDA, hy.BF16), (hy.DENSE, hy.F32)):
        M = out["M"] if fam in (hy.DENSE, hy.KDA) else None
        st = lib.hypic_segment_scan_static(fam, dt, 1, 1, k.shape[1], 2, 128, 128, P(offs), P(k), P(v), P(a),
                                           P(b), P(out["lam"]), P(M), P(out["S"]), P(None), P(None))
        assert st == -2, (fam, dt)
    torch.cuda.synchronize()
    assert torch.isnan(out["S"]).all() and torch.isnan(out["lam"]).all()


def test_static_scratch_empty_segments_need_no_scratch():
    import torch
    import linear_attention_state_gated_gb300 as hy
    k, v, a, b, _ = _inputs([64], 1, 2, seed=34)
    offs = torch.zeros(4, dtype=torch.int64, device="cuda")      # three empty segments
    out = _nan_out(1, 3, 2)
    hy.segment_scan_static(k[:, :0], v[:, :0], a[:, :0], offs, out, beta=b[:, :0])
    torch.cuda.synchronize()
    eye = torch.eye(128, device="cuda").expand(1, 3, 2, 128, 128)
    assert torch.equal(out["lam"], torch.zeros_like(out["lam"]))
    assert torch.equal(out["M"], eye) and torch.equal(out["S"], torch.zeros_like(out["S"]))
