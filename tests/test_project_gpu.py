"""The fused input projections (kda_project_inputs, one tcgen05 GEMM) against the fp64 definition x W^T.

Bar, per element: |y_gpu - y| <= 2^-8 |y| + 2 * 2 K 2^-24 sum_k |x_k w_k|.  The first term is the bf16
rounding of the result (unit roundoff 2^-8); the second bounds the fp32 accumulation error of a K-term sum
in any order ((K-1) 2^-24 sum |terms|), doubled, and doubled again for the rounding of that error.  Then
projections feeding the prefill kernels reproduce the oracle's layer output within the prefill bars.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.kda_testutil import S_TOL, Y_TOL, bf16_dev_to_f64, s_err, to_dev_bf16, y_err

pytestmark = pytest.mark.gpu


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


def _run(kda, x_bits, w_bits, H, dk, dv, with_z=True):
    T = x_bits.shape[0]
    x, w = to_dev_bf16(x_bits), to_dev_bf16(w_bits)
    e = lambda *s: torch.full(s, -7.0, dtype=torch.bfloat16, device="cuda")  # noqa: E731  (poisoned)
    out = dict(q=e(T, H, dk), k=e(T, H, dk), v=e(T, H, dv), a=e(T, H, dk), z=e(T, H, dv) if with_z else None,
               b=e(T, H))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_project_inputs(x, w, H, dk, dv, out["q"], out["k"], out["v"], out["a"], out["b"], out["z"], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {k: (bf16_dev_to_f64(v) if v is not None else None) for k, v in out.items()}


def _check(got, x_bits, w_bits, H, dk, dv, rows=None):
    xf = ki.bf16_bits_to_f64(x_bits if rows is None else x_bits[rows])
    wf = ki.bf16_bits_to_f64(w_bits)
    ref = oracle.project(xf, wf, H, dk, dv)
    mag = oracle.project(np.abs(xf), np.abs(wf), H, dk, dv)  # sum_k |x_k w_k| per output
    K = xf.shape[1]
    for name in ("q", "k", "v", "a", "z", "b"):
        if got[name] is None:
            continue
        g = got[name] if rows is None else got[name][rows]
        tol = 2.0 ** -8 * np.abs(ref[name]) + 4.0 * K * 2.0 ** -24 * mag[name]
        bad = np.abs(g - ref[name]) > tol
        assert not bad.any(), (name, int(bad.sum()), float(np.abs(g - ref[name]).max()))


@pytest.mark.parametrize("T,hidden,H,dk,dv,with_z", [
    (333, 320, 3, 16, 16, True),      # hidden not a multiple of the 64-wide K step; ragged M and N tiles
    (200, 512, 4, 128, 128, True),    # the production head shape
    (129, 256, 2, 32, 16, False),     # dk != dv, no output gate: those columns are computed and dropped
    (1, 64, 1, 16, 32, True),         # one token, one head
])
def test_projection_matches_fp64(T, hidden, H, dk, dv, with_z):
    kda = _kda()
    N = kda.projection_width(H, dk, dv)
    x, w = ki.projection_inputs(T + hidden + H, T, hidden, N)
    got = _run(kda, x, w, H, dk, dv, with_z)
    _check(got, x, w, H, dk, dv)


def test_projection_full_size_sampled_rows():
    """The benchmark's projection: 22528 tokens, hidden 4096, H = 32, d = 128 (20512 features); every output
    of 12 sampled token rows (across all M tiles' positions) against fp64."""
    kda = _kda()
    T, hidden, H, D = 22528, 4096, 32, 128
    N = kda.projection_width(H, D, D)
    x, w = ki.projection_inputs(3, T, hidden, N)
    got = _run(kda, x, w, H, D, D)
    rows = np.array([0, 1, 127, 128, 5000, 11111, 12800, 17407, 20000, 22400, 22526, 22527])
    _check(got, x, w, H, D, D, rows=rows)


def test_projected_inputs_drive_the_prefill():
    """Hidden states -> projections -> chunked prefill on the GPU, against the oracle run on the fp64
    projections rounded to bf16 (the inputs the layer consumes)."""
    kda = _kda()
    T, hidden, H, D, C = 300, 256, 2, 128, 64
    N = kda.projection_width(H, D, D)
    x, w = ki.projection_inputs(77, T, hidden, N)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    out = {n: torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda") for n in ("q", "k", "v", "a", "z")}
    out["b"] = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_project_inputs(xd, wd, H, D, D, out["q"], out["k"], out["v"], out["a"], out["b"], out["z"], st)
    pool = kda.StatePool.empty(4, H, D, D)
    wts = ki.layer_weights(78, H, D, D)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    y = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, 1, T, C), dtype=torch.uint8, device="cuda")
    t = lambda a, dt: torch.tensor(a, dtype=dt, device="cuda")  # noqa: E731
    kda.kda_prefill_chunked(pool, prm, t([0, T], torch.int32), t([0], torch.int64), t([-1], torch.int32),
                            t([1], torch.int32), C, 0, t([0, 0], torch.int32), t([0], torch.int32), out["q"],
                            out["k"], out["v"], out["a"], out["b"], out["z"], y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_p = oracle.project(ki.bf16_bits_to_f64(x), ki.bf16_bits_to_f64(w), H, D, D)
    f = {k: oracle.round_to_bf16(v) for k, v in ref_p.items()}
    ref = oracle.forward(oracle.Cfg(H=H, dk=D, dv=D), [0, T], [0], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                         wts["conv_w"], wts["norm_w"], np.zeros((1, H, D, D)), np.zeros((1, H, 3, 3 * D)))
    assert y_err(bf16_dev_to_f64(y), ref["y"]) <= Y_TOL
    assert s_err(pool.S[1].cpu().numpy()[None], ref["S"]) <= S_TOL
