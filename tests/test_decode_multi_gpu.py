"""Multi-token decode (speculative verification, per-position state retention) on the GPU through the C ABI,
against the fp64 oracle and against the single-token kernel.

Bars as for decode: bf16 outputs within 2e-2 (max over (token, head) of max|y - y_ref| / max|y_ref|), states
within 1e-3 relative Frobenius per (request, head) (1e-3 + 2^-9 for a bf16 pool), conv windows and untouched
slots bit-exact; L = 1 and the resume-after-rejection path bit-for-bit against the kernels' own results.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.kda_testutil import (S_TOL, S_TOL_BF16, Y_TOL, bf16_dev_bits, bf16_dev_to_f64, fill_pool, pool_unit_host,
                                s_err, to_dev_bf16, y_err)

pytestmark = pytest.mark.gpu


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


class Multi:
    def __init__(self, kda, H, dk, dv, L, src, dst, num_slots, seed, sbf16=False, with_z=True):
        self.kda, self.H, self.dk, self.dv, self.L, self.sbf16 = kda, H, dk, dv, L, sbf16
        self.src, self.dst = list(src), np.asarray(dst, dtype=np.int32).reshape(-1)
        self.n = len(src)
        self.pool = kda.StatePool.empty(num_slots, H, dk, dv,
                                        state_dtype=torch.bfloat16 if sbf16 else torch.float32)
        self.S_h, self.C_h = fill_pool(self.pool, seed)
        self.wts = ki.layer_weights(seed, H, dk, dv)
        self.prm = kda.LayerParams(torch.from_numpy(self.wts["conv_w"]).cuda(),
                                   torch.from_numpy(self.wts["norm_w"]).cuda())
        self.tok = ki.token_inputs(seed, self.n * L, H, dk, dv, with_z=with_z)
        self.d = {k: (to_dev_bf16(v) if v is not None else None) for k, v in self.tok.items()}
        self.st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self):
        self.y = torch.empty(self.n * self.L, self.H, self.dv, dtype=torch.bfloat16, device="cuda")
        d = self.d
        self.kda.kda_decode_multi(self.pool, self.prm, self.L, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], self.y,
                                  torch.tensor(self.src, dtype=torch.int32, device="cuda"),
                                  torch.from_numpy(self.dst).cuda(), self.st)
        torch.cuda.synchronize()
        return int(self.st.item())

    def reference(self):
        H, dk, dv = self.H, self.dk, self.dv
        cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
        S0 = np.zeros((self.n, H, dk, dv))
        C0 = np.zeros((self.n, H, 3, 2 * dk + dv))
        for i, s in enumerate(self.src):
            if s >= 0:
                S0[i], C0[i] = pool_unit_host(self.S_h, self.C_h, s, H)
                if self.sbf16:
                    S0[i] = oracle.round_to_bf16(S0[i])
        f = {k: (ki.bf16_bits_to_f64(v) if v is not None else None) for k, v in self.tok.items()}
        return oracle.forward(cfg, np.arange(self.n + 1) * self.L, np.zeros(self.n, dtype=np.int64), f["q"], f["k"],
                              f["v"], f["a"], f["b"], f["z"], self.wts["conv_w"], self.wts["norm_w"], S0, C0,
                              interval=1)

    def check(self, ref):
        stol = S_TOL_BF16 if self.sbf16 else S_TOL
        assert y_err(bf16_dev_to_f64(self.y), ref["y"]) <= Y_TOL
        for i, slot in enumerate(self.dst):
            if slot < 0:
                continue
            Sg = self.pool.S[int(slot)].float().cpu().numpy()
            assert s_err(Sg, ref["ckpt_S"][i]) <= stol, (i, int(slot))
            np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(self.pool.conv[int(slot)])),
                                          ref["ckpt_conv"][i])


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 16), (16, 32), (64, 64), (128, 128)])
@pytest.mark.parametrize("L", [2, 5, 8])
def test_multi_matches_oracle(dk, dv, L):
    """Fresh, moved and in-place requests; some positions not kept; untouched slots bit-exact."""
    kda = _kda()
    src = [3, -1, 20, 7]
    free = iter(s for s in range(8, 60) if s not in (20,))
    dst = []
    for r in range(4):
        row = [next(free) if (j % 3 != 1 or j == L - 1) else -1 for j in range(L)]
        dst.append(row)
    dst[2][L - 1] = 20  # the third request ends in place
    m = Multi(kda, 3, dk, dv, L, src, dst, 64, seed=dk * 3 + dv + L)
    S_before, C_before = m.pool.S.clone(), m.pool.conv.clone()
    assert m.run() == 0
    m.check(m.reference())
    written = set(int(x) for x in m.dst if x >= 0)
    keep = [s for s in range(64) if s not in written]
    assert torch.equal(m.pool.S[keep], S_before[keep])
    assert torch.equal(m.pool.conv[keep].view(torch.int16), C_before[keep].view(torch.int16))


@pytest.mark.parametrize("sbf16", [False, True])
def test_multi_L1_equals_single_token_decode_bitwise(sbf16):
    kda = _kda()
    n, H = 16, 8
    src = list(range(0, 2 * n, 2))
    dst = list(range(1, 2 * n, 2))
    a = Multi(kda, H, 128, 128, 1, src, dst, 2 * n, seed=5, sbf16=sbf16)
    b = Multi(kda, H, 128, 128, 1, src, dst, 2 * n, seed=5, sbf16=sbf16)
    assert a.run() == 0
    y = torch.empty(n, H, 128, dtype=torch.bfloat16, device="cuda")
    d = b.d
    t = lambda x: torch.tensor(x, dtype=torch.int32, device="cuda")  # noqa: E731
    kda.kda_decode_step(b.pool, b.prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, t(src), t(dst), b.st)
    torch.cuda.synchronize()
    assert int(b.st.item()) == 0
    assert torch.equal(a.y.view(torch.int16), y.view(torch.int16))
    assert torch.equal(a.pool.S.view(torch.int16), b.pool.S.view(torch.int16))
    assert torch.equal(a.pool.conv.view(torch.int16), b.pool.conv.view(torch.int16))


def test_multi_bf16_pool_matches_oracle():
    kda = _kda()
    L = 5
    src = [1, 2, -1, 3]
    dst = [[10 + 5 * r + j for j in range(L)] for r in range(4)]
    m = Multi(kda, 4, 128, 128, L, src, dst, 40, seed=9, sbf16=True)
    assert m.run() == 0
    m.check(m.reference())


def test_rejection_resumes_from_the_last_accepted_position():
    """Verify 5 draft tokens keeping every position; accept a different prefix per request; continue with one
    more token from the kept slot.  The continued state equals, bit for bit, a verify call of exactly the
    accepted length followed by the same token, and the oracle within the bars."""
    kda = _kda()
    H, L, n = 4, 5, 6
    accept = [1, 2, 3, 4, 5, 3]
    src = list(range(n))
    dst = [[8 + r * L + j for j in range(L)] for r in range(n)]
    m = Multi(kda, H, 128, 128, L, src, dst, 64, seed=21)
    assert m.run() == 0
    # next token per request from the slot of its last accepted position, into a fresh slot
    nxt = ki.token_inputs(99, n, H, 128, 128)
    dn = {k: to_dev_bf16(v) for k, v in nxt.items()}
    resume = [dst[r][accept[r] - 1] for r in range(n)]
    out = [40 + r for r in range(n)]
    y1 = torch.empty(n, H, 128, dtype=torch.bfloat16, device="cuda")
    t = lambda x: torch.tensor(x, dtype=torch.int32, device="cuda")  # noqa: E731
    kda.kda_decode_step(m.pool, m.prm, dn["q"], dn["k"], dn["v"], dn["a"], dn["b"], dn["z"], y1, t(resume), t(out), m.st)
    torch.cuda.synchronize()
    assert int(m.st.item()) == 0
    # replay: per request, a verify call of exactly the accepted tokens, then the same next token
    for r in range(n):
        Lr = accept[r]
        rep = Multi(kda, H, 128, 128, Lr, [src[r]], [[50 + j for j in range(Lr)]], 64, seed=21)
        rows = list(range(r * L, r * L + Lr))
        rep.tok = {k: v[rows] for k, v in m.tok.items()}
        rep.d = {k: to_dev_bf16(v) for k, v in rep.tok.items()}
        assert rep.run() == 0
        assert torch.equal(rep.y.view(torch.int16), m.y[rows].view(torch.int16))
        assert torch.equal(rep.pool.S[50 + Lr - 1], m.pool.S[resume[r]])
        y2 = torch.empty(1, H, 128, dtype=torch.bfloat16, device="cuda")
        d1 = {k: v[r:r + 1].contiguous() for k, v in dn.items()}
        kda.kda_decode_step(rep.pool, rep.prm, d1["q"], d1["k"], d1["v"], d1["a"], d1["b"], d1["z"], y2,
                            t([50 + Lr - 1]), t([60]), rep.st)
        torch.cuda.synchronize()
        assert int(rep.st.item()) == 0
        assert torch.equal(y2.view(torch.int16), y1[r:r + 1].view(torch.int16))
        assert torch.equal(rep.pool.S[60], m.pool.S[out[r]])
        # oracle: the accepted tokens then the next one, from the request's initial state
        cfg = oracle.Cfg(H=H, dk=128, dv=128)
        S0, C0 = pool_unit_host(m.S_h, m.C_h, src[r], H)
        f = {k: np.concatenate([ki.bf16_bits_to_f64(m.tok[k][rows]), ki.bf16_bits_to_f64(nxt[k][r:r + 1])])
             for k in m.tok}
        ref = oracle.forward(cfg, [0, Lr + 1], [0], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                             m.wts["conv_w"], m.wts["norm_w"], S0[None], C0[None])
        assert y_err(bf16_dev_to_f64(y2), ref["y"][Lr:]) <= Y_TOL
        assert s_err(m.pool.S[out[r]].cpu().numpy()[None], ref["S"]) <= S_TOL


def test_multi_bad_slot_is_reported_and_isolated():
    kda = _kda()
    L = 3
    src = [0, 1, 2]
    dst = [[3, 4, 5], [6, 999, 7], [8, 9, 10]]  # request 1 keeps a position outside the pool
    m = Multi(kda, 2, 64, 64, L, src, dst, 16, seed=3)
    S_before = m.pool.S.clone()
    assert m.run() == kda.KDA_DEV_BAD_SLOT
    assert not bool(m.y[L:2 * L].float().abs().sum())  # its outputs are zero
    assert torch.equal(m.pool.S[[6, 7]], S_before[[6, 7]])  # and it writes nothing
    ref = m.reference()
    good = list(range(0, L)) + list(range(2 * L, 3 * L))
    assert y_err(bf16_dev_to_f64(m.y[good]), ref["y"][good]) <= Y_TOL


def test_multi_full_size_sampled():
    """The benchmark's verify configuration: 64 requests x 5 tokens, H = 32, d = 128, every position kept, on a
    4096-slot pool; the oracle checks sampled requests (all heads)."""
    kda = _kda()
    n, H, L, slots = 64, 32, 5, 4096
    perm = ki.permutation(17, ki.STREAM["slots"], slots)
    src = [int(x) for x in perm[:n]]
    dst = np.asarray(perm[n:n + n * L], dtype=np.int32).reshape(n, L)
    m = Multi(kda, H, 128, 128, L, src, dst, slots, seed=17)
    assert m.run() == 0
    cfg = oracle.Cfg(H=H, dk=128, dv=128)
    for r in (0, 29, 63):
        rows = list(range(r * L, (r + 1) * L))
        S0, C0 = pool_unit_host(m.S_h, m.C_h, src[r], H)
        f = {k: ki.bf16_bits_to_f64(v[rows]) for k, v in m.tok.items()}
        ref = oracle.forward(cfg, [0, L], [0], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"], m.wts["conv_w"],
                             m.wts["norm_w"], S0[None], C0[None], interval=1)
        assert y_err(bf16_dev_to_f64(m.y[rows]), ref["y"]) <= Y_TOL
        for j in range(L):
            assert s_err(m.pool.S[int(dst[r, j])].cpu().numpy(), ref["ckpt_S"][j]) <= S_TOL
