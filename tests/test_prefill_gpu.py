"""Chunked prefill with checkpoint emission on the GPU (through the C ABI) against the fp64 oracle.

Bars: bf16 outputs within 2e-2 (max over (token, head) of max|y - y_ref| / max|y_ref|); fp32 states
(final and every checkpoint) within 1e-3 relative Frobenius per (sequence, head); conv windows, slot
placement and every untouched slot bit-exact; resume == replay bit-exact GPU against GPU.
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


class Problem:
    """A varlen prefill call: sequences, start positions, slots, checkpoint table, inputs."""

    def __init__(self, kda, H, dk, dv, lens, starts, src, dst, chunk, interval, num_slots, seed, with_z=True,
                 fill=True, ckpt_skip=(), sbf16=False):
        self.kda, self.H, self.dk, self.dv, self.sbf16 = kda, H, dk, dv, sbf16
        self.lens, self.starts, self.src, self.dst = list(lens), list(starts), list(src), list(dst)
        self.chunk, self.interval, self.num_slots = chunk, interval, num_slots
        self.T = int(sum(lens))
        self.cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        self.pool = kda.StatePool.empty(num_slots, H, dk, dv,
                                        state_dtype=torch.bfloat16 if sbf16 else torch.float32)
        self.S_h, self.C_h = fill_pool(self.pool, seed) if fill else (None, None)
        self.wts = ki.layer_weights(seed, H, dk, dv)
        self.prm = kda.LayerParams(torch.from_numpy(self.wts["conv_w"]).cuda(),
                                   torch.from_numpy(self.wts["norm_w"]).cuda())
        self.tok = ki.token_inputs(seed, self.T, H, dk, dv, with_z=with_z)
        counts = [oracle.ckpt_count(s, l, interval) if interval else 0 for s, l in zip(starts, lens)]
        self.offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        used = set(x for x in src if x >= 0) | set(dst)
        free = [s for s in range(num_slots) if s not in used]
        nck = int(self.offs[-1])
        assert len(free) >= nck
        self.ck = np.array(free[:nck], dtype=np.int32)
        for j in ckpt_skip:
            self.ck[j] = -1

    def run(self, status=None):
        kda = self.kda
        d = {k: (to_dev_bf16(v) if v is not None else None) for k, v in self.tok.items()}
        self.y = torch.empty(self.T, self.H, self.dv, dtype=torch.bfloat16, device="cuda")
        nbytes = kda.kda_prefill_workspace_bytes(self.pool, len(self.lens), self.T, self.chunk)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        ws.fill_(0xAB)  # contents need not be initialised
        self.status = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
        t = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device="cuda")  # noqa: E731
        kda.kda_prefill_chunked(self.pool, self.prm, t(self.cu, torch.int32), t(self.starts, torch.int64),
                                t(self.src, torch.int32), t(self.dst, torch.int32), self.chunk, self.interval,
                                t(self.offs, torch.int32), t(self.ck if len(self.ck) else [0], torch.int32),
                                d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], self.y, ws, self.status)
        torch.cuda.synchronize()
        return int(self.status.item())

    def reference(self, heads=None):
        """fp64 oracle over all sequences for the given heads (all by default)."""
        heads = list(range(self.H)) if heads is None else list(heads)
        Hs, dk, dv = len(heads), self.dk, self.dv
        cfg = oracle.Cfg(H=Hs, dk=dk, dv=dv)
        N = len(self.lens)
        S0 = np.zeros((N, Hs, dk, dv))
        C0 = np.zeros((N, Hs, 3, 2 * dk + dv))
        for n, s in enumerate(self.src):
            if s >= 0:
                Sa, Ca = pool_unit_host(self.S_h, self.C_h, s, self.H)
                S0[n], C0[n] = Sa[heads], Ca[heads]
                if self.sbf16:  # the pool holds the bf16 rounding of the generated states
                    S0[n] = oracle.round_to_bf16(S0[n])
        f = {k: (ki.bf16_bits_to_f64(v)[:, heads] if v is not None else None) for k, v in self.tok.items()}
        return oracle.forward(cfg, self.cu, np.array(self.starts, dtype=np.int64), f["q"], f["k"], f["v"], f["a"],
                              f["b"], f["z"], self.wts["conv_w"][heads], self.wts["norm_w"], S0, C0,
                              interval=self.interval)

    def check(self, ref, heads=None):
        """Asserts the bars; returns the measured worst output error, final-state error and checkpoint error."""
        heads = list(range(self.H)) if heads is None else list(heads)
        stol = S_TOL_BF16 if self.sbf16 else S_TOL
        yg = bf16_dev_to_f64(self.y)[:, heads]
        ey = y_err(yg, ref["y"])
        assert ey <= Y_TOL
        es, ec = 0.0, 0.0
        for n, d in enumerate(self.dst):
            Sg = self.pool.S[d].float().cpu().numpy()[heads]
            e = s_err(Sg, ref["S"][n])
            assert e <= stol, ("final", n)
            es = max(es, e)
            np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(self.pool.conv[d]))[heads],
                                          ref["conv"][n])
        for j, slot in enumerate(self.ck):
            if slot < 0:
                continue
            Sg = self.pool.S[int(slot)].float().cpu().numpy()[heads]
            e = s_err(Sg, ref["ckpt_S"][j])
            assert e <= stol, ("ckpt", j, int(ref["ckpt_pos"][j]))
            ec = max(ec, e)
            np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(self.pool.conv[int(slot)]))[heads],
                                          ref["ckpt_conv"][j])
        return ey, es, ec


SHAPES = [(16, 16), (32, 16), (16, 32), (64, 64), (128, 128)]


@pytest.mark.parametrize("dk,dv", SHAPES)
@pytest.mark.parametrize("chunk", [16, 64])
def test_prefill_matches_oracle_varlen(dk, dv, chunk):
    """Ragged sequences, non-zero start positions (resumed states), fresh and moved slots, checkpoints
    (one skipped), a zero-length sequence; every slot that is neither a destination nor a checkpoint
    is bit-for-bit unchanged."""
    kda = _kda()
    interval = 2 * chunk
    lens = [3 * chunk + 5, 1, chunk - 3, 0, 2 * chunk]
    starts = [0, 7, 2 * chunk + 1, 5, interval]
    src = [-1, 3, 4, 6, 9]
    dst = [2, 3, 5, 7, 10]
    p = Problem(kda, 3, dk, dv, lens, starts, src, dst, chunk, interval, 40, seed=dk * 7 + dv + chunk,
                ckpt_skip=(1,))
    before_S, before_C = p.pool.S.clone(), p.pool.conv.clone()
    assert p.run() == 0
    p.check(p.reference())
    written = set(dst) | set(int(x) for x in p.ck if x >= 0)
    keep = [s for s in range(40) if s not in written]
    assert torch.equal(p.pool.S[keep], before_S[keep])
    assert torch.equal(p.pool.conv[keep].view(torch.int16), before_C[keep].view(torch.int16))


@pytest.mark.parametrize("dk,dv,chunk,H", [(16, 16, 16, 2), (128, 128, 64, 1)])
def test_prefill_more_sequences_than_one_table_block(dk, dv, chunk, H):
    """1500 sequences of 0 to 3 tokens at scattered start positions, a third of them resumed from stored
    states, checkpoints at every chunk boundary they cross: more sequences than the table kernel's block
    takes at once, on both paths, against the oracle (outputs, final states, windows, checkpoints)."""
    kda = _kda()
    rng = np.random.default_rng(7)
    N = 1500
    lens = rng.integers(0, 4, N).tolist()
    starts = rng.integers(0, 200, N).tolist()
    src = [N + i if i % 3 == 0 else -1 for i in range(N)]
    p = Problem(kda, H, dk, dv, lens, starts, src, list(range(N)), chunk, chunk, 2 * N + 64, seed=dk + H)
    assert len(p.ck) > 0
    assert p.run() == 0
    p.check(p.reference())


@pytest.mark.parametrize("dk,dv,chunk", [(16, 16, 16), (128, 128, 64)])
def test_prefill_of_empty_sequences_only(dk, dv, chunk):
    """A call whose sequences are all empty (no tokens at all): each destination receives its source state and
    window unchanged (zeros for a fresh one), and no other slot changes."""
    kda = _kda()
    src, dst = [3, -1, 5, 1], [2, 4, 6, 7]
    p = Problem(kda, 2, dk, dv, [0, 0, 0, 0], [0, 9, 64, 100], src, dst, chunk, chunk, 12, seed=dk)
    before_S, before_C = p.pool.S.clone(), p.pool.conv.clone()
    assert p.run() == 0
    for s_, d_ in zip(src, dst):
        if s_ >= 0:
            assert torch.equal(p.pool.S[d_], before_S[s_])
            assert torch.equal(p.pool.conv[d_].view(torch.int16), before_C[s_].view(torch.int16))
        else:
            assert not p.pool.S[d_].any() and not p.pool.conv[d_].view(torch.int16).any()
    keep = [x for x in range(12) if x not in dst]
    assert torch.equal(p.pool.S[keep], before_S[keep])


def test_prefill_no_gate_and_no_checkpoints():
    kda = _kda()
    p = Problem(kda, 2, 128, 128, [100, 37], [0, 64], [-1, 1], [0, 1], 64, 0, 8, seed=5, with_z=False)
    assert p.run() == 0
    p.check(p.reference())


def test_tiny_configuration_end_to_end():
    """The tiny configuration: H=2, dk=dv=16, a 64-token prefill from an empty prefix (chunk 16,
    checkpoints every 32 tokens), 8 decode steps from the final state, and a resume from the checkpoint
    at 32 replayed to 64 -- all against the oracle; resume vs replay bit-exact on the GPU."""
    kda = _kda()
    H, D, T = 2, 16, 64
    p = Problem(kda, H, D, D, [T], [0], [-1], [0], 16, 32, 8, seed=1)
    assert p.run() == 0
    ref = p.reference()
    p.check(ref)
    assert list(ref["ckpt_pos"]) == [32, 64]
    ck32, ck64 = int(p.ck[0]), int(p.ck[1])
    # 8 decode steps from slot 0
    tok = ki.token_inputs(11, 8, H, D, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for s in range(8):
        d = {k: to_dev_bf16(np.ascontiguousarray(v[s:s + 1])) for k, v in tok.items()}
        y = torch.empty(1, H, D, dtype=torch.bfloat16, device="cuda")
        sl = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.kda_decode_step(p.pool, p.prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, sl, sl, status)
        ys.append(bf16_dev_to_f64(y)[0])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    f = {k: ki.bf16_bits_to_f64(v) for k, v in tok.items()}
    cfg = oracle.Cfg(H=H, dk=D, dv=D)
    dec = oracle.forward(cfg, [0, 8], [T], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"], p.wts["conv_w"],
                         p.wts["norm_w"], ref["S"], ref["conv"])
    assert y_err(np.array(ys), dec["y"]) <= Y_TOL
    assert s_err(p.pool.S[0].cpu().numpy(), dec["S"][0]) <= S_TOL
    # resume from the checkpoint at 32 into a private slot, replay tokens 32..63
    kda.kda_resume_from_slot(p.pool, torch.tensor([ck32], dtype=torch.int32, device="cuda"),
                             torch.tensor([5], dtype=torch.int32, device="cuda"), status)
    q = Problem.__new__(Problem)
    q.__dict__.update(p.__dict__)
    q.lens, q.starts, q.src, q.dst, q.T = [32], [32], [5], [5], 32
    q.cu = np.array([0, 32], dtype=np.int32)
    q.tok = {k: np.ascontiguousarray(v[32:]) for k, v in p.tok.items()}
    q.offs = np.array([0, 1], dtype=np.int32)
    q.ck = np.array([6], dtype=np.int32)
    y_full = p.y.clone()
    assert q.run() == 0
    assert torch.equal(q.y.view(torch.int16), y_full[32:].view(torch.int16))
    assert torch.equal(p.pool.S[6], p.pool.S[ck64]) and torch.equal(p.pool.S[5], p.pool.S[ck64])
    assert torch.equal(p.pool.conv[5].view(torch.int16), p.pool.conv[ck64].view(torch.int16))


def test_resume_equals_replay_bitwise_shared_prefix():
    """Several requests share one prefix: each resumes from the prefix's last checkpoint (copy-on-write
    into a private slot) and prefills its own suffix; each result equals, bit for bit, a full replay of
    prefix + suffix, and the shared checkpoint slot is left untouched."""
    kda = _kda()
    H, D, C, I, P, R, L = 4, 128, 64, 128, 1024 + 40, 3, 200
    b = (P // I) * I  # largest checkpoint boundary inside the shared prefix
    base = ki.token_inputs(41, P, H, D, D)
    full = Problem(kda, H, D, D, [P], [0], [-1], [0], C, I, 64, seed=41)
    full.tok = base
    assert full.run() == 0
    j = list(oracle.ckpt_positions(0, P, I)).index(b)
    shared = int(full.ck[j])
    shared_before = (full.pool.S[shared].clone(), full.pool.conv[shared].clone())
    suffixes = [ki.token_inputs(100 + r, L, H, D, D) for r in range(R)]
    # resumed: copy-on-write into private slots 50.., then one varlen call for all suffixes (tokens b.. P+L)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    priv = list(range(50, 50 + R))
    kda.kda_resume_from_slot(full.pool, torch.tensor([shared] * R, dtype=torch.int32, device="cuda"),
                             torch.tensor(priv, dtype=torch.int32, device="cuda"), status)
    res = Problem.__new__(Problem)
    res.__dict__.update(full.__dict__)
    seg = [{k: np.concatenate([base[k][b:], suffixes[r][k]]) for k in base} for r in range(R)]
    res.lens, res.starts, res.src, res.dst = [P - b + L] * R, [b] * R, priv, priv
    res.T = R * (P - b + L)
    res.cu = np.arange(R + 1, dtype=np.int32) * (P - b + L)
    res.tok = {k: np.concatenate([s[k] for s in seg]) for k in base}
    res.offs = np.zeros(R + 1, dtype=np.int32)
    res.ck = np.zeros(0, dtype=np.int32)
    res.interval = 0
    assert res.run() == 0
    y_res = res.y.clone()
    assert torch.equal(full.pool.S[shared], shared_before[0])
    assert torch.equal(full.pool.conv[shared].view(torch.int16), shared_before[1].view(torch.int16))
    # full replays of prefix + suffix, one call each
    for r in range(R):
        rep = Problem.__new__(Problem)
        rep.__dict__.update(full.__dict__)
        rep.lens, rep.starts, rep.src, rep.dst = [P + L], [0], [-1], [60 + r]
        rep.T = P + L
        rep.cu = np.array([0, P + L], dtype=np.int32)
        rep.tok = {k: np.concatenate([base[k], suffixes[r][k]]) for k in base}
        rep.offs = np.zeros(2, dtype=np.int32)
        rep.ck = np.zeros(0, dtype=np.int32)
        rep.interval = 0
        assert rep.run() == 0
        seg_len = P - b + L
        assert torch.equal(rep.y[b:].view(torch.int16), y_res[r * seg_len:(r + 1) * seg_len].view(torch.int16))
        assert torch.equal(full.pool.S[60 + r], full.pool.S[priv[r]])
        assert torch.equal(full.pool.conv[60 + r].view(torch.int16), full.pool.conv[priv[r]].view(torch.int16))
    # and the resumed results match the oracle
    f_ref = rep.reference(heads=[0, 3])  # the last replay, oracle
    yg = bf16_dev_to_f64(y_res[(R - 1) * (P - b + L):])[:, [0, 3]]
    assert y_err(yg, f_ref["y"][b:]) <= Y_TOL


@pytest.mark.parametrize("dk,dv,chunk", [(128, 128, 64), (16, 16, 16), (32, 16, 16)])
def test_in_place_resume_equals_moved_resume_bitwise(dk, dv, chunk):
    """Resumed sequences prefilled in place (src == dst, the plan the prefix index makes) give, bit for bit,
    what the same call gives with the destinations moved to other slots.  With one head, the items of a
    sequence's first and last chunks are adjacent and run in the same wave, on different CTAs; sequences of
    1 and 2 tokens write a destination window made partly of source rows; one sequence is empty."""
    kda = _kda()
    lens = [chunk - 37 % chunk + 7, 1, 2, 0, 2 * chunk + 3]
    starts = [37, 64, 5, 9, 130]
    src = [3, 4, 5, 6, 7]
    moved = [12, 13, 14, 15, 16]
    seed = 4 * dk + dv + chunk
    p_in = Problem(kda, 1, dk, dv, lens, starts, src, src, chunk, chunk, 40, seed=seed)
    p_mv = Problem(kda, 1, dk, dv, lens, starts, src, moved, chunk, chunk, 40, seed=seed)
    p_in.ck = p_mv.ck = np.arange(20, 20 + len(p_in.ck), dtype=np.int32)
    assert p_mv.run() == 0
    assert p_in.run() == 0
    assert torch.equal(p_in.y.view(torch.int16), p_mv.y.view(torch.int16))
    for a_, b_ in zip(src, moved):
        assert torch.equal(p_in.pool.S[a_], p_mv.pool.S[b_])
        assert torch.equal(p_in.pool.conv[a_].view(torch.int16), p_mv.pool.conv[b_].view(torch.int16))
    for c_ in p_in.ck:
        assert torch.equal(p_in.pool.S[c_], p_mv.pool.S[c_])
        assert torch.equal(p_in.pool.conv[c_].view(torch.int16), p_mv.pool.conv[c_].view(torch.int16))
    p_mv.check(p_mv.reference())


def test_prefill_bad_tables_flag_status():
    kda = _kda()
    # checkpoint offsets that do not match the boundary count: flagged, no checkpoint written
    p = Problem(kda, 2, 16, 16, [40, 20], [0, 0], [-1, -1], [0, 1], 16, 16, 16, seed=3)
    p.offs = np.array([0, 1, 2], dtype=np.int32)  # should be [0, 2, 3]: sequence 0 is inconsistent
    before = p.pool.S.clone()
    st = p.run()
    assert st & kda.KDA_DEV_BAD_CKPT
    untouched = [s for s in range(16) if s not in (0, 1, int(p.ck[1]))]  # seq 1's entry is consistent
    assert torch.equal(p.pool.S[untouched], before[untouched])
    # a destination slot out of range: that sequence is skipped, the other one is computed
    p2 = Problem(kda, 2, 16, 16, [40, 20], [0, 0], [-1, -1], [0, 99], 16, 0, 16, seed=3)
    st = p2.run()
    assert st & kda.KDA_DEV_BAD_SLOT
    ref = p2.reference()
    assert y_err(bf16_dev_to_f64(p2.y)[:40], ref["y"][:40]) <= Y_TOL
    # cu_seqlens not ending at total_tokens
    p3 = Problem(kda, 2, 16, 16, [40, 20], [0, 0], [-1, -1], [0, 1], 16, 0, 16, seed=3)
    p3.cu = np.array([0, 40, 50], dtype=np.int32)
    assert p3.run() & kda.KDA_DEV_BAD_SEQLENS


def test_prefill_full_size_sampled_heads():
    """The chunked-prefill workload at full size (4 sequences of 2048/4096/8192/8192 tokens, H=32,
    dk=dv=128, chunk 64, checkpoints every 128 tokens: 176 boundaries), in the launch configuration the
    benchmark times; two heads against the oracle at every output, every checkpoint and the final states."""
    kda = _kda()
    lens = [2048, 4096, 8192, 8192]
    p = Problem(kda, 32, 128, 128, lens, [0] * 4, [-1] * 4, [0, 1, 2, 3], 64, 128, 256, seed=3, fill=False)
    assert p.run() == 0
    assert len(p.ck) == 176
    heads = [0, 21]
    ref = p.reference(heads)
    ey, es, ec = p.check(ref, heads)
    print(f"prefill workload (heads {heads}): output {ey:.3e}, final state {es:.3e}, checkpoints {ec:.3e}")


def test_prefill_wide_decay_range_and_large_values():
    """Decay logits near -8 (alpha ~ 3e-4) on runs of consecutive tokens in some channels, and values
    scaled by 50: the chunk's cumulative log-decay spans far more than the range one reference point
    can carry in fp32, so the intra-chunk products take the exact pairwise form."""
    kda = _kda()
    p = Problem(kda, 2, 128, 128, [200, 90], [0, 37], [-1, 3], [0, 3], 64, 128, 16, seed=13)
    a = ki.bf16_bits_to_f32(p.tok["a"]).copy()
    a[10:70, :, :16] = -8.0                  # channels 0..15 decay almost fully for 60 tokens
    a[150:160, 1, 40:60] = -6.0
    p.tok["a"] = ki.f32_to_bf16_bits(a)
    v = ki.bf16_bits_to_f32(p.tok["v"]) * 50.0
    p.tok["v"] = ki.f32_to_bf16_bits(v)
    assert p.run() == 0
    p.check(p.reference())


def test_prefix_resume_workload_full_size():
    """The prefix-resume workload at full size: one 32768-token prefix prefilled with checkpoints every 128
    tokens; 16 requests copy-on-write the checkpoint at 32768 into private slots and prefill 1024
    distinct tokens each in one varlen call.  Each result equals, bit for bit, a full replay of its
    33792 tokens; two heads of one request also match the oracle."""
    kda = _kda()
    H, D, C, I, P, R, L = 32, 128, 64, 128, 32768, 16, 1024
    pre = Problem(kda, H, D, D, [P], [0], [-1], [0], C, I, 320, seed=50, fill=False)
    assert pre.run() == 0
    shared = int(pre.ck[-1])  # the boundary at 32768
    assert oracle.ckpt_positions(0, P, I)[-1] == P
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    priv = list(range(300, 300 + R))
    kda.kda_resume_from_slot(pre.pool, torch.tensor([shared] * R, dtype=torch.int32, device="cuda"),
                             torch.tensor(priv, dtype=torch.int32, device="cuda"), status)
    suffix = [ki.token_inputs(500 + r, L, H, D, D) for r in range(R)]
    res = Problem.__new__(Problem)
    res.__dict__.update(pre.__dict__)
    res.lens, res.starts, res.src, res.dst, res.T = [L] * R, [P] * R, priv, priv, R * L
    res.cu = np.arange(R + 1, dtype=np.int32) * L
    res.tok = {k: np.concatenate([s[k] for s in suffix]) for k in suffix[0]}
    res.interval, res.offs, res.ck = 0, np.zeros(R + 1, dtype=np.int32), np.zeros(0, dtype=np.int32)
    assert res.run() == 0
    y_res = res.y.clone()
    for r in (0, 7, 15):  # full replays of three of the requests
        rep = Problem.__new__(Problem)
        rep.__dict__.update(pre.__dict__)
        rep.lens, rep.starts, rep.src, rep.dst, rep.T = [P + L], [0], [-1], [310], P + L
        rep.cu = np.array([0, P + L], dtype=np.int32)
        rep.tok = {k: np.concatenate([pre.tok[k], suffix[r][k]]) for k in suffix[0]}
        rep.interval, rep.offs, rep.ck = 0, np.zeros(2, dtype=np.int32), np.zeros(0, dtype=np.int32)
        assert rep.run() == 0
        assert torch.equal(rep.y[P:].view(torch.int16), y_res[r * L:(r + 1) * L].view(torch.int16))
        assert torch.equal(pre.pool.S[310], pre.pool.S[priv[r]])
        assert torch.equal(pre.pool.conv[310].view(torch.int16), pre.pool.conv[priv[r]].view(torch.int16))
        if r == 15:
            ref = rep.reference(heads=[3, 30])
            ey = y_err(bf16_dev_to_f64(y_res[r * L:(r + 1) * L])[:, [3, 30]], ref["y"][P:])
            es = s_err(pre.pool.S[priv[r]].cpu().numpy()[[3, 30]], ref["S"][0])
            print(f"prefix-resume workload (request 15, heads [3, 30]): resumed output {ey:.3e}, state {es:.3e}")
            assert ey <= Y_TOL and es <= S_TOL


def test_long_context_workload_full_size():
    """The long-context workload: one 131072-token prefill (H=32, dk=dv=128, chunk 64, checkpoints every
    32768 tokens), then a batch-256 decode step in which one request continues this sequence from its
    final state and 255 use random slots.  Two heads against the oracle at every output, checkpoint,
    the final state and the decode step."""
    kda = _kda()
    H, D, T, I = 32, 128, 131072, 32768
    p = Problem(kda, H, D, D, [T], [0], [-1], [0], 64, I, 512, seed=60, fill=False)
    assert p.run() == 0
    assert len(p.ck) == 4
    heads = [5, 26]
    ref = p.reference(heads)
    ey, es, ec = p.check(ref, heads)
    print(f"long-context prefill (heads {heads}): output {ey:.3e}, final state {es:.3e}, checkpoints {ec:.3e}")
    # decode at batch 256: request 0 continues slot 0, the others use random slots (zero states here)
    N = 256
    slots = [0] + [int(s) for s in ki.random_slots(61, 512, N + 8)[1:] if int(s) not in p.ck and s != 0][:N - 1]
    tok = ki.token_inputs(62, N, H, D, D)
    dev = {k: to_dev_bf16(v) for k, v in tok.items()}
    y = torch.empty(N, H, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    kda.kda_decode_step(p.pool, p.prm, dev["q"], dev["k"], dev["v"], dev["a"], dev["b"], dev["z"], y, sl, sl, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cfg = oracle.Cfg(H=len(heads), dk=D, dv=D)
    f = {k: ki.bf16_bits_to_f64(v)[:1, heads] for k, v in tok.items()}
    dec = oracle.forward(cfg, [0, 1], [T], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                         p.wts["conv_w"][heads], p.wts["norm_w"], ref["S"], ref["conv"])
    ey = y_err(bf16_dev_to_f64(y[:1])[:, heads], dec["y"])
    es = s_err(p.pool.S[0].cpu().numpy()[heads], dec["S"][0])
    print(f"long-context decode step after the prefill: output {ey:.3e}, state {es:.3e}")
    assert ey <= Y_TOL and es <= S_TOL
