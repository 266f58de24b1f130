"""Output precision of the tensor-core prefill where it is hardest, against the fp64 oracle.

A token's attention output can be far smaller than the terms that form it; the gated RMSNorm then scales
the residual up to unit size, so the per-token output bar (2e-2 of the vector's largest element) sees the
operand rounding of those terms.  The plainest such token is a sequence's first one from an empty state:
its output is the single term scale * (q^ . k^) * beta * v^, and when q^ and k^ are nearly orthogonal the
dot product is a sum of 128 terms that cancel.  These tests build that token on purpose (the conv output
of its raw q and k solved for a chosen q^ . k^), and sweep many seeds of the prefill workload's shapes.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.kda_testutil import S_TOL, Y_TOL, bf16_dev_to_f64, s_err, to_dev_bf16, y_err

D, C, W = 128, 64, 4
SILU_MIN_X = -1.2784645427610738  # argmin of x * sigmoid(x)


def _silu(x):
    return x / (1.0 + np.exp(-x))


def _silu_inverse(y):
    """The x >= SILU_MIN_X with silu(x) = y (bisection), or None below silu's minimum."""
    if y <= _silu(SILU_MIN_X):
        return None
    lo, hi = SILU_MIN_X, max(1.0, y + 2.0)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if _silu(mid) < y:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _bf16(x):
    return float(ki.bf16_bits_to_f64(ki.f32_to_bf16_bits(np.array([x], dtype=np.float32)))[0])


def _unit_dot(xq, xk, eps=1e-6):
    return float(xq @ xk / np.sqrt((xq @ xq + eps) * (xk @ xk + eps)))


def near_orthogonal_k(q_raw, k_raw, wq, wk, target):
    """Raw bf16 key values k' (fp64 array) such that, for a first token from an empty window (only the conv's
    last tap sees an input), the L2-normalised conv outputs satisfy q^ . k'^ ~= target.  Channels taken in
    order of q's conv output move the key's conv output (kept within [-0.25, 4]) until the remaining dot
    product is small; one reserved channel, set to a small value where bf16 is fine-grained, absorbs the
    rest.  Returns None if that does not converge."""
    xq = _silu(wq * q_raw)
    order = [int(c) for c in np.argsort(-np.abs(xq)) if abs(wk[c]) >= 0.05]
    c2 = order[1]
    k = k_raw.copy()

    def resid(k_):
        xk = _silu(wk * k_)
        return target * np.sqrt((xq @ xq + 1e-6) * (xk @ xk + 1e-6)) - xq @ xk, xk

    for _ in range(8):
        k[c2] = 0.0
        for c in order:
            if c == c2:
                continue
            r, xk = resid(k)
            if abs(r) <= 0.1 * abs(xq[c2]):
                break
            k[c] = _bf16(_silu_inverse(float(np.clip(xk[c] + r / xq[c], -0.25, 4.0))) / wk[c])
        r, _ = resid(k)
        u = _silu_inverse(r / xq[c2])
        if u is None:
            return None
        k[c2] = _bf16(u / wk[c2])
        if abs(_unit_dot(xq, _silu(wk * k)) - target) <= 0.05 * abs(target):
            return k
    return None


def test_near_orthogonal_construction_reaches_its_target():
    """The input construction itself (CPU): the fp64 conv + SiLU + L2 norm of the built key gives the asked-for
    q^ . k^ to within 10%, for targets down to 3e-5, on the workload's distributions."""
    wts = ki.layer_weights(90, 1, D, D)
    tok = ki.token_inputs(90, 8, 1, D, D)
    q = ki.bf16_bits_to_f64(tok["q"])[:, 0]
    k = ki.bf16_bits_to_f64(tok["k"])[:, 0]
    wq, wk = wts["conv_w"][0, :D, W - 1], wts["conv_w"][0, D:2 * D, W - 1]
    for r, target in enumerate([1e-3, -3e-4, 1e-4, -1e-4, 3e-5, 2e-4]):
        kk = near_orthogonal_k(q[r], k[r], wq, wk, target)
        assert kk is not None
        got = _unit_dot(_silu(wq * q[r]), _silu(wk * kk))
        assert abs(got - target) <= 0.1 * abs(target), (target, got)
        # the built key is a bf16 vector and keeps most of the drawn channels
        assert np.array_equal(kk, ki.bf16_bits_to_f64(ki.f32_to_bf16_bits(kk.astype(np.float32))))
        assert int((kk != k[r]).sum()) <= 24


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


def _run(kda, H, lens, starts, tok, conv_w, norm_w, interval, num_slots):
    """One prefill call from empty states (src = -1) into slots 0.., checkpoints after them; returns y and the
    pool tensors."""
    N, T = len(lens), int(sum(lens))
    pool = kda.StatePool.empty(num_slots, H, D, D)
    prm = kda.LayerParams(torch.from_numpy(conv_w).cuda(), torch.from_numpy(norm_w).cuda())
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    counts = [oracle.ckpt_count(s, l, interval) if interval else 0 for s, l in zip(starts, lens)]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ck = np.arange(N, N + int(offs[-1]), dtype=np.int32)
    assert N + len(ck) <= num_slots
    i32 = lambda a: torch.tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa: E731
    d = {k_: to_dev_bf16(v) for k_, v in tok.items()}
    y = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, N, T, C), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill_chunked(pool, prm, i32(cu), torch.tensor(starts, dtype=torch.int64, device="cuda"),
                            i32([-1] * N), i32(list(range(N))), C, interval, i32(offs), i32(ck if len(ck) else [0]),
                            d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, pool, cu, ck


@pytest.mark.gpu
def test_near_orthogonal_first_tokens_match_the_oracle():
    """Eight sequences (some starting mid-chunk) whose first token has q^ . k^ between 3e-5 and 1e-3 in
    every head, from empty states: outputs at every token within 2e-2 and states within 1e-3 of the oracle.
    The first token's output here is a single near-cancelling dot product scaled to unit size by the norm."""
    kda = _kda()
    H = 4
    lens = [130, 64, 200, 97, 64, 150, 70, 129]
    starts = [0, 0, 37, 0, 5, 0, 63, 0]
    targets = [1e-4, -1e-4, 3e-4, 3e-5, -3e-5, 1e-3, 1e-4, -3e-4]
    T = int(sum(lens))
    wts = ki.layer_weights(91, H, D, D)
    tok = ki.token_inputs(91, T, H, D, D)
    q = ki.bf16_bits_to_f64(tok["q"])
    k = ki.bf16_bits_to_f64(tok["k"]).copy()
    cu = np.concatenate([[0], np.cumsum(lens)])
    built = 0
    for n, target in enumerate(targets):
        t0 = int(cu[n])
        for h in range(H):
            wq, wk = wts["conv_w"][h, :D, W - 1], wts["conv_w"][h, D:2 * D, W - 1]
            kk = near_orthogonal_k(q[t0, h], k[t0, h], wq, wk, target)
            if kk is None:
                continue
            k[t0, h] = kk
            got = _unit_dot(_silu(wq * q[t0, h]), _silu(wk * kk))
            assert abs(got - target) <= 0.1 * abs(target)
            built += 1
    assert built >= 28  # nearly every (sequence, head) got its near-orthogonal first token
    tok["k"] = ki.f32_to_bf16_bits(k.astype(np.float32))
    y, pool, cu32, ck = _run(kda, H, lens, starts, tok, wts["conv_w"], wts["norm_w"], 128, 32)
    f = {k_: ki.bf16_bits_to_f64(v) for k_, v in tok.items()}
    N = len(lens)
    ref = oracle.forward(oracle.Cfg(H=H, dk=D, dv=D, W=W), cu32, np.array(starts, dtype=np.int64), f["q"], f["k"],
                         f["v"], f["a"], f["b"], f["z"], wts["conv_w"], wts["norm_w"], np.zeros((N, H, D, D)),
                         np.zeros((N, H, W - 1, 3 * D)), interval=128)
    yg = bf16_dev_to_f64(y)
    first = cu32[:-1]
    e_first = y_err(yg[first], ref["y"][first])
    e_all = y_err(yg, ref["y"])
    e_S = s_err(pool.S[:N].cpu().numpy(), ref["S"])
    print(f"near-orthogonal first tokens: output error {e_all:.3e} (first tokens {e_first:.3e}), state {e_S:.3e}")
    assert e_all <= Y_TOL and e_S <= S_TOL
    if len(ck):
        assert s_err(pool.S[ck].cpu().numpy(), ref["ckpt_S"]) <= S_TOL


@pytest.mark.gpu
def test_sixteen_seed_sweep_matches_the_oracle():
    """Sixteen seeds of the prefill workload's distributions, four heads each (64 heads in one call: heads
    4s..4s+3 take seed s's tokens and conv weights), 8192 tokens from an empty state, chunk 64, checkpoints
    every 1024 tokens: every output element and every state against the oracle."""
    kda = _kda()
    S_, Hs, T, I = 16, 4, 8192, 1024
    H = S_ * Hs
    parts = [ki.token_inputs(100 + s, T, Hs, D, D) for s in range(S_)]
    tok = {k_: np.ascontiguousarray(np.concatenate([p[k_] for p in parts], axis=1)) for k_ in parts[0]}
    conv_w = np.concatenate([ki.layer_weights(100 + s, Hs, D, D)["conv_w"] for s in range(S_)])
    norm_w = ki.layer_weights(100, Hs, D, D)["norm_w"]
    y, pool, cu32, ck = _run(kda, H, [T], [0], tok, conv_w, norm_w, I, 1 + T // I)
    f = {k_: ki.bf16_bits_to_f64(v) for k_, v in tok.items()}
    ref = oracle.forward(oracle.Cfg(H=H, dk=D, dv=D, W=W), cu32, np.zeros(1, dtype=np.int64), f["q"], f["k"],
                         f["v"], f["a"], f["b"], f["z"], conv_w, norm_w, np.zeros((1, H, D, D)),
                         np.zeros((1, H, W - 1, 3 * D)), interval=I)
    yg = bf16_dev_to_f64(y)
    Sf = pool.S[0].cpu().numpy()
    Sc = pool.S[ck].cpu().numpy()
    worst = []
    for s in range(S_):
        hs = slice(Hs * s, Hs * (s + 1))
        ey = y_err(yg[:, hs], ref["y"][:, hs])
        es = max(s_err(Sf[hs], ref["S"][0, hs]), s_err(Sc[:, hs], ref["ckpt_S"][:, hs]))
        worst.append((ey, es))
    ey = np.array([w[0] for w in worst])
    es = np.array([w[1] for w in worst])
    print("sixteen-seed sweep: output error per seed " + " ".join(f"{e:.2e}" for e in ey))
    print(f"sixteen-seed sweep: worst output {ey.max():.3e} (median {np.median(ey):.3e}), worst state {es.max():.3e}")
    assert ey.max() <= Y_TOL and es.max() <= S_TOL
