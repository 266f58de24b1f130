"""Pins for the fp64 oracle, checked against things other than the oracle itself.

The pages print no worked numeric example for the KDA layer, so every pin here comes from the
mathematics of the recurrence (gated delta rule with channel-wise decay, as used by Kimi Linear):
a brute force written with library routines and the dense matrix form of the update, exact rational
arithmetic, closed forms, invariants, and agreement of the oracle's two independent evaluation orders
(token by token vs chunked WY/UT).  Shapes use dk != dv so that a transposed operand fails.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import kda_inputs as ki

RNG = np.random.default_rng(1234)


def _rand_case(H=2, dk=4, dv=3, W=4, lens=(7, 5), starts=(0, 3), with_z=True, seed=0, a_shift=3.0):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    Cc = 2 * dk + dv
    d = dict(
        q=rng.standard_normal((T, H, dk)), k=rng.standard_normal((T, H, dk)), v=rng.standard_normal((T, H, dv)),
        a=rng.standard_normal((T, H, dk)) + a_shift, b=rng.standard_normal((T, H)),
        z=rng.standard_normal((T, H, dv)) if with_z else None,
        conv_w=rng.standard_normal((H, Cc, W)) / math.sqrt(W), norm_w=1 + 0.1 * rng.standard_normal(dv),
        S0=0.3 * rng.standard_normal((N, H, dk, dv)), conv0=rng.standard_normal((N, H, W - 1, Cc)),
        cu=cu, sp=np.array(starts, dtype=np.int64))
    return d


def _run(cfg, d, interval=0, chunk=0, **over):
    d = {**d, **over}
    return oracle.forward(cfg, d["cu"], d["sp"], d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], d["conv_w"],
                          d["norm_w"], d["S0"], d["conv0"], interval=interval, chunk=chunk)


def _brute(cfg, d, interval):
    """Library routines (torch fp64 conv1d / silu / sigmoid / normalize / rms_norm) and the dense
    matrix update S <- (I - beta k k^T) Diag(alpha) S + beta k v^T."""
    H, dk, dv, W = cfg.H, cfg.dk, cfg.dv, cfg.W
    Cc = cfg.Cc
    cu, sp = d["cu"], d["sp"]
    T = int(cu[-1])
    y = np.zeros((T, H, dv))
    o_all = np.zeros((T, H, dv))
    S_fin, C_fin, cks = [], [], []
    for n in range(len(sp)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        Sn, Cn = [], []
        for h in range(H):
            x = np.concatenate([d["q"][t0:t1, h], d["k"][t0:t1, h], d["v"][t0:t1, h]], axis=1)  # [L, Cc]
            full = np.concatenate([d["conv0"][n, h], x], axis=0)                                 # [W-1+L, Cc]
            xt = torch.tensor(full.T[None], dtype=torch.float64)
            wt = torch.tensor(d["conv_w"][h][:, None, :], dtype=torch.float64)
            conv = F.conv1d(xt, wt, groups=Cc)[0].T                                               # [L, Cc]
            if cfg.conv_silu:
                conv = F.silu(conv)
            qh = F.normalize(conv[:, :dk], dim=-1, eps=1e-300)
            kh = F.normalize(conv[:, dk:2 * dk], dim=-1, eps=1e-300)
            vh = conv[:, 2 * dk:]
            al = torch.sigmoid(torch.tensor(d["a"][t0:t1, h]))
            be = torch.sigmoid(torch.tensor(d["b"][t0:t1, h]))
            S = torch.tensor(d["S0"][n, h])
            hc = []
            for i in range(t1 - t0):
                M = (torch.eye(dk, dtype=torch.float64) - be[i] * torch.outer(kh[i], kh[i])) @ torch.diag(al[i])
                S = M @ S + be[i] * torch.outer(kh[i], vh[i])
                o = cfg.scale * (S.T @ qh[i])
                yy = F.rms_norm(o[None], (dv,), weight=torch.tensor(d["norm_w"]), eps=cfg.rms_eps)[0]
                if d["z"] is not None:
                    yy = yy * torch.sigmoid(torch.tensor(d["z"][t0 + i, h]))
                y[t0 + i, h] = yy.numpy()
                o_all[t0 + i, h] = o.numpy()
                p = int(sp[n]) + i + 1
                if interval and p % interval == 0:
                    hc.append((p, S.numpy().copy(), full[i + 1:i + W].copy()))
            Sn.append(S.numpy())
            Cn.append(full[-(W - 1):] if W > 1 else np.zeros((0, Cc)))
            cks.append((n, h, hc))
        S_fin.append(Sn)
        C_fin.append(Cn)
    return dict(y=y, o=o_all, S=np.array(S_fin), conv=np.array(C_fin), cks=cks)


@pytest.mark.parametrize("silu,with_z,scale", [(True, True, 1.0), (False, False, 0.25), (True, False, 0.5)])
def test_oracle_matches_library_brute_force(silu, with_z, scale):
    cfg = oracle.Cfg(H=2, dk=4, dv=3, W=4, conv_silu=silu, l2_eps=0.0, rms_eps=1e-6, scale=scale)
    d = _rand_case(with_z=with_z, seed=7, lens=(9, 6, 1), starts=(0, 5, 11))
    r = _run(cfg, d, interval=3)
    b = _brute(cfg, d, interval=3)
    np.testing.assert_allclose(r["y"], b["y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["o"], b["o"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["S"], b["S"], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(r["conv"], b["conv"])
    # checkpoints: positions and contents
    j = 0
    for n in range(3):
        per_h = [c for c in b["cks"] if c[0] == n]
        npos = len(per_h[0][2])
        for m in range(npos):
            assert r["ckpt_seq"][j] == n and r["ckpt_pos"][j] == per_h[0][2][m][0]
            for h in range(2):
                np.testing.assert_allclose(r["ckpt_S"][j, h], per_h[h][2][m][1], rtol=1e-11, atol=1e-12)
                np.testing.assert_array_equal(r["ckpt_conv"][j, h], per_h[h][2][m][2])
            j += 1
    assert j == len(r["ckpt_pos"])


def _pyth_vectors():
    """Integer 4-vectors with integer norms (tests/golden/pythagorean_vectors.txt)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "pythagorean_vectors.txt")
    out = []
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            vals = [int(x) for x in line.split()]
            assert sum(x * x for x in vals[:4]) == vals[4] ** 2
            out.append((vals[:4], vals[4]))
    return out


def test_oracle_exact_rational_arithmetic():
    """d=4, T=8: q, k with integer norms (so the normalised vectors are rational), identity conv, no
    activation, l2_eps = 0; alpha and beta are the exact binary fractions of the fp64 sigmoids.  The
    recurrence is then evaluated in exact rational arithmetic with the dense matrix form."""
    vecs = _pyth_vectors()
    rng = np.random.default_rng(5)
    dk, dv, T, H, W = 4, 3, 8, 1, 4
    q = np.zeros((T, H, dk)); k = np.zeros((T, H, dk)); qn = []; kn = []
    for t in range(T):
        for arr, nl in ((q, qn), (k, kn)):
            vec, nrm = vecs[rng.integers(len(vecs))]
            perm = rng.permutation(4)
            sgn = rng.choice([-1, 1], 4)
            arr[t, 0] = np.array(vec)[perm] * sgn
            nl.append(nrm)
    v = rng.integers(-4, 5, (T, H, dv)).astype(np.float64)
    a = np.round(rng.standard_normal((T, H, dk)) + 2, 3)
    b = np.round(rng.standard_normal((T, H)), 3)
    conv_w = np.zeros((H, 2 * dk + dv, W)); conv_w[..., -1] = 1.0
    S0 = rng.integers(-3, 4, (1, H, dk, dv)).astype(np.float64) / 4
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv, W=W, conv_silu=False, l2_eps=0.0, rms_eps=0.0, scale=1.0)
    r = oracle.forward(cfg, [0, T], [0], q, k, v, a, b, None, conv_w, np.ones(dv), S0, np.zeros((1, H, W - 1, 11)))
    S = [[Fraction(int(x * 4), 4) for x in row] for row in S0[0, 0]]
    for t in range(T):
        kh = [Fraction(int(x), kn[t]) for x in k[t, 0]]
        qh = [Fraction(int(x), qn[t]) for x in q[t, 0]]
        al = [Fraction(1.0 / (1.0 + math.exp(-float(x)))) for x in a[t, 0]]
        be = Fraction(1.0 / (1.0 + math.exp(-float(b[t, 0]))))
        M = [[(1 if i == j else 0) * al[j] - be * kh[i] * kh[j] * al[j] for j in range(dk)] for i in range(dk)]
        S = [[sum(M[i][m] * S[m][j] for m in range(dk)) + be * kh[i] * Fraction(int(v[t, 0, j])) for j in range(dv)]
             for i in range(dk)]
        o = [sum(S[i][j] * qh[i] for i in range(dk)) for j in range(dv)]
        np.testing.assert_allclose(r["o"][t, 0], [float(x) for x in o], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["S"][0, 0], [[float(x) for x in row] for row in S], rtol=1e-13, atol=1e-14)


def _ident_cfg(**kw):
    base = dict(H=2, dk=5, dv=3, W=4, conv_silu=False, l2_eps=0.0, rms_eps=0.0, scale=1.0)
    base.update(kw)
    return oracle.Cfg(**base)


def _ident_conv(cfg):
    w = np.zeros((cfg.H, cfg.Cc, cfg.W)); w[..., -1] = 1.0
    return w


def test_pin_identity_step_alpha1_beta0():
    """alpha = 1, beta = 0 leaves S unchanged exactly and o = S_0^T q^."""
    cfg = _ident_cfg()
    d = _rand_case(H=2, dk=5, dv=3, lens=(6,), starts=(0,), seed=3)
    d["a"][:] = 40.0     # sigmoid(40) == 1.0 in fp64
    d["b"][:] = -1000.0  # sigmoid(-1000) == 0.0
    r = _run(cfg, d, conv_w=_ident_conv(cfg))
    np.testing.assert_array_equal(r["S"], d["S0"])
    for t in range(6):
        for h in range(2):
            qh = F.normalize(torch.tensor(d["q"][t, h]), dim=0, eps=1e-300).numpy()
            np.testing.assert_allclose(r["o"][t, h], d["S0"][0, h].T @ qh, rtol=1e-13, atol=1e-14)


def test_pin_beta0_closed_form_decay():
    """beta = 0: S_T = Diag(prod_t alpha_t) S_0."""
    cfg = _ident_cfg()
    d = _rand_case(H=2, dk=5, dv=3, lens=(9,), starts=(0,), seed=4)
    d["b"][:] = -1000.0
    r = _run(cfg, d, conv_w=_ident_conv(cfg))
    prod = torch.sigmoid(torch.tensor(d["a"])).prod(dim=0).numpy()  # [H, dk]
    np.testing.assert_allclose(r["S"][0], prod[:, :, None] * d["S0"][0], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("b_logit", [1000.0, 0.7, -0.4])
def test_pin_delta_rule_invariant(b_logit):
    """With |k^| = 1: S_1^T k^ = (1 - beta) (Diag(alpha) S_0)^T k^ + beta v; at beta = 1 the new
    value is stored exactly under its key."""
    cfg = _ident_cfg()
    d = _rand_case(H=2, dk=5, dv=3, lens=(1,), starts=(0,), seed=11)
    d["b"][:] = b_logit
    r = _run(cfg, d, conv_w=_ident_conv(cfg))
    for h in range(2):
        kh = F.normalize(torch.tensor(d["k"][0, h]), dim=0, eps=1e-300).numpy()
        al = torch.sigmoid(torch.tensor(d["a"][0, h])).numpy()
        be = float(torch.sigmoid(torch.tensor(b_logit, dtype=torch.float64)))
        lhs = r["S"][0, h].T @ kh
        rhs = (1 - be) * (al[:, None] * d["S0"][0, h]).T @ kh + be * d["v"][0, h]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)


def test_pin_single_token_from_zero_state():
    """S_0 = 0, one token: S_1 = beta k^ v^T and o = scale beta (q^ . k^) v."""
    cfg = _ident_cfg(scale=0.37)
    d = _rand_case(H=2, dk=5, dv=3, lens=(1,), starts=(0,), seed=12)
    d["S0"][:] = 0.0
    r = _run(cfg, d, conv_w=_ident_conv(cfg))
    for h in range(2):
        qh = F.normalize(torch.tensor(d["q"][0, h]), dim=0, eps=1e-300).numpy()
        kh = F.normalize(torch.tensor(d["k"][0, h]), dim=0, eps=1e-300).numpy()
        be = float(torch.sigmoid(torch.tensor(d["b"][0, h])))
        np.testing.assert_allclose(r["S"][0, h], be * np.outer(kh, d["v"][0, h]), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(r["o"][0, h], 0.37 * be * (qh @ kh) * d["v"][0, h], rtol=1e-12, atol=1e-14)


def test_pin_linearity_in_state_and_values():
    """Given q, k, alpha, beta (and a linear conv), (S_0, V, v-window) -> (S_T, O) is linear."""
    cfg = oracle.Cfg(H=2, dk=5, dv=3, W=4, conv_silu=False, l2_eps=1e-6, rms_eps=1e-6)
    d1 = _rand_case(H=2, dk=5, dv=3, lens=(8,), starts=(2,), seed=20)
    d2 = _rand_case(H=2, dk=5, dv=3, lens=(8,), starts=(2,), seed=21)
    d2.update({key: d1[key] for key in ("q", "k", "a", "b", "conv_w", "z")})
    c2 = d2["conv0"].copy(); c2[..., :10] = d1["conv0"][..., :10]; d2["conv0"] = c2  # same q,k windows
    ds = dict(d1); ds["S0"] = d1["S0"] + d2["S0"]; ds["v"] = d1["v"] + d2["v"]
    cs = d1["conv0"].copy(); cs[..., 10:] = d1["conv0"][..., 10:] + d2["conv0"][..., 10:]; ds["conv0"] = cs
    r1, r2, rs = _run(cfg, d1), _run(cfg, d2), _run(cfg, ds)
    np.testing.assert_allclose(rs["S"], r1["S"] + r2["S"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(rs["o"], r1["o"] + r2["o"], rtol=1e-11, atol=1e-12)


def test_pin_conv_constant_input_and_window_shift():
    """Constant raw input c with a window full of c gives v^ = c * sum_j w_j (no activation); the
    stored window holds the last W-1 raw inputs, oldest first."""
    cfg = _ident_cfg(H=1, dk=2, dv=3)
    d = _rand_case(H=1, dk=2, dv=3, lens=(1,), starts=(0,), seed=30)
    cw = d["conv_w"].copy()
    cw[0, :4] = 0.0
    cw[0, :4, -1] = 1.0          # identity taps on the q and k channels
    c = 0.75
    d["v"][:] = c
    d["conv0"][..., 4:] = c
    d["S0"][:] = 0.0
    d["b"][:] = 1000.0           # beta = 1: S_1 = k^ v^^T, so S_1^T k^ = v^ (|k^| = 1)
    r = _run(cfg, d, conv_w=cw)
    kh = F.normalize(torch.tensor(d["k"][0, 0]), dim=0, eps=1e-300).numpy()
    np.testing.assert_allclose(r["S"][0, 0].T @ kh, c * cw[0, 4:].sum(-1), rtol=1e-12)
    for L in (1, 2, 5):
        d = _rand_case(H=1, dk=2, dv=3, lens=(L,), starts=(0,), seed=31)
        r = _run(cfg, d)
        raw = np.concatenate([d["conv0"][0, 0], np.concatenate([d["q"][:, 0], d["k"][:, 0], d["v"][:, 0]], 1)], 0)
        np.testing.assert_array_equal(r["conv"][0, 0], raw[-3:])


def test_pin_rmsnorm_unit_rms():
    cfg = oracle.Cfg(H=2, dk=4, dv=6, W=4, rms_eps=0.0)
    d = _rand_case(H=2, dk=4, dv=6, lens=(5, 3), starts=(0, 0), with_z=False, seed=40)
    r = _run(cfg, d, norm_w=np.ones(6))
    np.testing.assert_allclose((r["y"] ** 2).mean(-1), 1.0, rtol=1e-13)


def test_pin_l2_eps_placement():
    """q^ = q / sqrt(|q|^2 + eps): a zero vector stays zero, a one-hot c e_0 maps to c / sqrt(c^2+eps)."""
    cfg = oracle.Cfg(H=1, dk=3, dv=2, W=4, conv_silu=False, l2_eps=0.5)
    d = _rand_case(H=1, dk=3, dv=2, lens=(1,), starts=(0,), seed=50)
    conv_w = np.zeros((1, 8, 4)); conv_w[..., -1] = 1.0
    d["q"][:] = 0.0; d["q"][0, 0, 0] = 2.0
    d["k"][:] = 0.0; d["k"][0, 0, 1] = 2.0
    d["S0"][:] = 0.0
    d["b"][:] = 1000.0
    r = _run(cfg, d, conv_w=conv_w)
    kh = 2.0 / math.sqrt(4.5)
    np.testing.assert_allclose(r["S"][0, 0][1], kh * d["v"][0, 0], rtol=1e-14)
    assert np.all(r["S"][0, 0][[0, 2]] == 0.0)
    assert np.all(r["o"] == 0.0)  # q^ is orthogonal to k^
    d["q"][:] = 0.0; d["q"][0, 0, 1] = 2.0  # now parallel: o = (q^ . k^) v = (4 / 4.5) v
    r = _run(cfg, d, conv_w=conv_w)
    np.testing.assert_allclose(r["o"][0, 0], kh * kh * d["v"][0, 0], rtol=1e-14)
    d["k"][:] = 0.0
    r = _run(cfg, d, conv_w=conv_w)
    assert np.all(r["S"] == 0.0) and np.all(np.isfinite(r["y"]))


@pytest.mark.parametrize("chunk", [4, 16, 64])
def test_pin_chunked_form_equals_recurrence(chunk):
    """The chunked WY/UT form (chunks aligned to absolute positions, ragged first and last chunks)
    reproduces the token-by-token recurrence."""
    cfg = oracle.Cfg(H=2, dk=8, dv=6, W=4)
    d = _rand_case(H=2, dk=8, dv=6, lens=(70, 33, 5), starts=(0, chunk * 3 - 7 if chunk > 7 else 5, 2), seed=60)
    interval = chunk * 2
    r0 = _run(cfg, d, interval=interval)
    r1 = _run(cfg, d, interval=interval, chunk=chunk)
    for key in ("y", "o", "S", "ckpt_S"):
        np.testing.assert_allclose(r1[key], r0[key], rtol=1e-10, atol=1e-11)
    for key in ("conv", "ckpt_conv", "ckpt_pos", "ckpt_seq"):
        np.testing.assert_array_equal(r1[key], r0[key])


def test_pin_chunked_form_stress_small_alpha_large_v():
    """alpha down to 1e-3 (decay logits near -7) and |v| ~ 100."""
    cfg = oracle.Cfg(H=1, dk=8, dv=4, W=4)
    d = _rand_case(H=1, dk=8, dv=4, lens=(50,), starts=(3,), seed=70, a_shift=0.0)
    d["a"] = np.where(RNG.random(d["a"].shape) < 0.3, -6.9, d["a"])
    d["v"] *= 100.0
    r0 = _run(cfg, d)
    r1 = _run(cfg, d, chunk=16)
    np.testing.assert_allclose(r1["S"], r0["S"], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(r1["y"], r0["y"], rtol=1e-9, atol=1e-10)


def test_pin_resume_equals_replay_bitwise():
    """Resuming from the checkpoint at a boundary gives bit-for-bit the same outputs and final state
    as replaying the whole sequence (same operation order)."""
    cfg = oracle.Cfg(H=2, dk=6, dv=5, W=4)
    d = _rand_case(H=2, dk=6, dv=5, lens=(40,), starts=(0,), seed=80)
    full = _run(cfg, d, interval=16)
    b = 32
    j = list(full["ckpt_pos"]).index(b)
    tail = {key: (d[key][b:] if key in ("q", "k", "v", "a", "b", "z") else d[key]) for key in d}
    tail.update(cu=np.array([0, 40 - b]), sp=np.array([b]), S0=full["ckpt_S"][j][None],
                conv0=full["ckpt_conv"][j][None])
    res = _run(cfg, tail)
    np.testing.assert_array_equal(res["S"], full["S"])
    np.testing.assert_array_equal(res["conv"], full["conv"])
    np.testing.assert_array_equal(res["y"], full["y"][b:])


@pytest.mark.parametrize("start,length,interval", [(0, 64, 32), (5, 64, 32), (32, 32, 32), (31, 1, 32),
                                                   (0, 0, 128), (127, 129, 128), (32768, 1024, 128)])
def test_checkpoint_count_matches_scan(start, length, interval):
    scan = [p for p in range(start + 1, start + length + 1) if p % interval == 0]
    assert oracle.ckpt_positions(start, length, interval) == scan


def test_generator_bf16_rounding_and_determinism():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e38, np.inf, -0.0], dtype=np.float32)
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 1.5*2^-8 rounds up to 1 + 2^-7
    np.testing.assert_array_equal(ki.bf16_bits_to_f32(ki.f32_to_bf16_bits(x))[:4],
                                  np.array([1.0, 1.0, 1.0078125, -2.5], dtype=np.float32))
    a = ki.normal(1, 2, (1000,))
    b = ki.normal(1, 2, (10,), offset=500)
    np.testing.assert_array_equal(a[500:510], b)
    assert abs(float(a.mean())) < 0.1 and abs(float(a.std()) - 1) < 0.1


def test_golden_tiny_regression_anchor():
    """The oracle + generator still reproduce tests/golden/tiny_kda.json (written by make_golden.py)."""
    import json
    import os
    from tests.golden import make_golden
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_kda.json")
    ref = json.load(open(path))
    now = make_golden.compute()
    for key, val in now.items():
        np.testing.assert_allclose(np.asarray(val, dtype=np.float64), np.asarray(ref[key], dtype=np.float64),
                                   rtol=1e-12, atol=1e-14, err_msg=key)


def test_bf16_pool_rounding_is_nearest_even():
    """The oracle's bf16-pool storage rounds to nearest even: a tie goes to the even neighbour, a value
    just above a tie rounds up, and values already representable in bf16 are unchanged."""
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.5, 0.0])
    want = np.array([1.0, 1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -2.5, 0.0])
    np.testing.assert_array_equal(oracle.round_to_bf16(x), want)
    vals = ki.bf16_bits_to_f64(ki.f32_to_bf16_bits(RNG.standard_normal(1000).astype(np.float32)))
    np.testing.assert_array_equal(oracle.round_to_bf16(vals), vals)


def test_multi_token_decode_equals_chained_single_steps():
    """The multi-token decode helper (per-position retention) against L single-token oracle steps chained
    through the pool: outputs, every kept state and window bit for bit; positions marked -1 write nothing;
    a request whose src is also its last kept slot updates in place."""
    H, dk, dv, L, n, slots = 2, 4, 3, 4, 3, 16
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
    rng = np.random.default_rng(77)
    Cc = 2 * dk + dv
    pool_S = 0.3 * rng.standard_normal((slots, H, dk, dv))
    pool_C = rng.standard_normal((slots, H, 3, Cc))
    tok = dict(q=rng.standard_normal((n * L, H, dk)), k=rng.standard_normal((n * L, H, dk)),
               v=rng.standard_normal((n * L, H, dv)), a=rng.standard_normal((n * L, H, dk)) + 3.0,
               b=rng.standard_normal((n * L, H)), z=rng.standard_normal((n * L, H, dv)))
    conv_w = rng.standard_normal((H, Cc, 4)) / 2.0
    norm_w = 1 + 0.1 * rng.standard_normal(dv)
    src = [3, -1, 9]
    dst = [[4, 5, -1, 6], [7, -1, -1, 8], [10, 11, 12, 9]]
    r = oracle.decode_multi_pool(cfg, pool_S, pool_C, L, src, np.array(dst).reshape(-1), tok["q"], tok["k"],
                                 tok["v"], tok["a"], tok["b"], tok["z"], conv_w, norm_w)
    scratch = [13, 14, 15]  # chain the single steps through spare slots
    S, C = pool_S.copy(), pool_C.copy()
    S[scratch] = 0.0
    C[scratch] = 0.0
    cur = list(src)
    for j in range(L):
        rows = [i * L + j for i in range(n)]
        step = oracle.decode_pool(cfg, S, C, cur, scratch, *(tok[x][rows] for x in ("q", "k", "v", "a", "b", "z")),
                                  conv_w, norm_w)
        S, C = step["pool_S"], step["pool_conv"]
        np.testing.assert_array_equal(r["y"][rows], step["y"])
        for i in range(n):
            np.testing.assert_array_equal(r["pos_S"][i * L + j], S[scratch[i]])
            if dst[i][j] >= 0:
                np.testing.assert_array_equal(r["pool_S"][dst[i][j]], S[scratch[i]])
                np.testing.assert_array_equal(r["pool_conv"][dst[i][j]], C[scratch[i]])
        cur = list(scratch)
    kept = {d for row in dst for d in row if d >= 0}
    for s_ in range(slots):
        if s_ not in kept:
            np.testing.assert_array_equal(r["pool_S"][s_], pool_S[s_])
    # a bf16 pool stores the rounding of the fp64 chain, which itself is never rounded between tokens
    rb = oracle.decode_multi_pool(cfg, pool_S, pool_C, L, src, np.array(dst).reshape(-1), tok["q"], tok["k"],
                                  tok["v"], tok["a"], tok["b"], tok["z"], conv_w, norm_w, state_bf16=True)
    np.testing.assert_array_equal(rb["y"], r["y"])
    np.testing.assert_array_equal(rb["pool_S"][8], oracle.round_to_bf16(r["pool_S"][8]))


def test_projection_definition_by_explicit_loops():
    """oracle.project against explicit sums on a tiny case: the row order of the packed weight (q, k, v, a,
    z, b) and the [T, H, d] split of each block."""
    H, dk, dv, hidden, T = 2, 3, 2, 5, 4
    rng = np.random.default_rng(5)
    N = H * (3 * dk + 2 * dv) + H
    x = rng.standard_normal((T, hidden))
    w = rng.standard_normal((N, hidden))
    got = oracle.project(x, w, H, dk, dv)
    row = 0
    for name, d in (("q", dk), ("k", dk), ("v", dv), ("a", dk), ("z", dv), ("b", None)):
        for h in range(H):
            for c in range(d or 1):
                for t in range(T):
                    want = sum(x[t, i] * w[row, i] for i in range(hidden))
                    val = got[name][t, h] if d is None else got[name][t, h, c]
                    assert abs(val - want) <= 1e-12 * (1 + abs(want)), (name, h, c, t)
                row += 1
    assert row == N
