"""Host prefix index (kda_prefix_* in the C ABI): chained match-unit hashes, interval and second-hit
retention, copy-on-write private slots, deferred same-step reuse, LRU eviction under pins, slot accounting.

The CPU tests need no GPU: the index is host code.  One of them drives the fp64 oracle through the plans the
index hands out (resume from the cached slot, prefill from the boundary with the ckpt_slots table) and checks
that every resumed output equals the from-scratch recurrence bit for bit.  The GPU test drives the kernels
through the same plans.
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle


def _kda():
    from hybrid_linear_attention_decode_gb300 import build as kbuild
    import hybrid_linear_attention_decode_gb300 as kda
    kbuild.build()
    kda.load_library()
    return kda


def toks(*segs):
    """Token ids of a prompt made of (segment id, length) pieces; equal pieces give equal ids."""
    return np.concatenate([np.int32(sid) * 100000 + np.arange(n, dtype=np.int32) for sid, n in segs]
                          ).astype(np.int32)


# ---------------------------------------------------------------------------------------------------- logic


def test_interval_policy_places_checkpoints_and_hits_the_longest_prefix():
    kda = _kda()
    ix = kda.PrefixIndex(16, match_unit=128, policy=kda.KDA_RETAIN_INTERVAL, interval=256)
    a = toks((1, 1000))
    p = ix.plan(a)
    assert p.src_slot == -1 and p.start_pos == 0
    # boundaries 128..896: kept at multiples of 256 and at the prompt's last boundary (896)
    kept = [128 * (j + 1) for j, s in enumerate(p.ckpt_slots) if s >= 0]
    assert len(p.ckpt_slots) == 7 and kept == [256, 512, 768, 896]
    assert len(set(s for s in p.ckpt_slots if s >= 0) | {p.private_slot}) == 5
    ix.commit(p)
    # same first 600 tokens, then a different tail: the longest cached prefix inside 600 is 512
    b = np.concatenate([a[:600], toks((2, 400))])
    q = ix.plan(b)
    assert q.start_pos == 512 and q.src_slot == p.ckpt_slots[3]
    assert len(q.ckpt_slots) == (1000 // 128) - 4  # boundaries 640..896
    ix.commit(q)
    # the whole of `a` plus more: hits the last boundary of `a`
    c = np.concatenate([a, toks((3, 50))])
    r = ix.plan(c)
    assert r.start_pos == 896 and r.src_slot == p.ckpt_slots[6]
    # a prompt equal to a cached prefix keeps at least one token to prefill
    d = a[:512]
    s = ix.plan(d)
    assert s.start_pos == 256 and s.src_slot == p.ckpt_slots[1]


def test_hashes_chain_over_the_whole_prefix():
    """A block with the same tokens after a different prefix is a different prefix."""
    kda = _kda()
    ix = kda.PrefixIndex(8, match_unit=16, interval=16)
    p = ix.plan(np.concatenate([toks((1, 16)), toks((2, 16)), toks((9, 5))]))
    ix.commit(p)
    q = ix.plan(np.concatenate([toks((3, 16)), toks((2, 16)), toks((9, 5))]))
    assert q.src_slot == -1 and q.start_pos == 0
    r = ix.plan(np.concatenate([toks((1, 16)), toks((2, 16)), toks((8, 5))]))
    assert r.start_pos == 32


def test_deferred_same_step_reuse():
    """Entries of an uncommitted plan are invisible: a second request of the same step starts from scratch
    and does not write the boundary state again; after the commit a third request resumes."""
    kda = _kda()
    ix = kda.PrefixIndex(8, match_unit=16, interval=16)
    prompt = toks((1, 40))
    p1 = ix.plan(prompt)
    assert p1.ckpt_slots[0] >= 0 and p1.ckpt_slots[1] >= 0
    p2 = ix.plan(prompt)
    assert p2.src_slot == -1 and p2.start_pos == 0 and p2.ckpt_slots == [-1, -1]
    ix.commit(p2)
    ix.commit(p1)
    p3 = ix.plan(prompt)
    assert p3.src_slot == p1.ckpt_slots[1] and p3.start_pos == 32


def test_second_hit_retention_keeps_only_prefixes_seen_twice():
    kda = _kda()
    ix = kda.PrefixIndex(8, match_unit=16, policy=kda.KDA_RETAIN_SECOND_HIT)
    sys_prompt = toks((1, 48))
    p1 = ix.plan(np.concatenate([sys_prompt, toks((2, 20))]))
    assert p1.ckpt_slots == [-1] * 4  # first sight: nothing kept
    ix.commit(p1)
    p2 = ix.plan(np.concatenate([sys_prompt, toks((3, 30))]))
    assert p2.src_slot == -1
    # boundaries 16..64; seen before: 16, 32, 48 (the shared prompt); only the longest shared one is kept
    assert [s >= 0 for s in p2.ckpt_slots] == [False, False, True, False]
    ix.commit(p2)
    p3 = ix.plan(np.concatenate([sys_prompt, toks((4, 20))]))
    assert p3.start_pos == 48 and p3.src_slot == p2.ckpt_slots[2]
    assert p3.ckpt_slots == [-1]  # boundary 64 of this prompt: first sight


def test_second_hit_with_interval_keeps_seen_interval_boundaries():
    kda = _kda()
    ix = kda.PrefixIndex(8, match_unit=16, policy=kda.KDA_RETAIN_SECOND_HIT, interval=32)
    base = toks((1, 100))
    ix.commit(ix.plan(base))
    p = ix.plan(np.concatenate([base[:70], toks((2, 30))]))
    # seen boundaries 16, 32, 48, 64: keep the interval ones (32, 64) and the longest shared one (64)
    assert [16 * (j + 1) for j, s in enumerate(p.ckpt_slots) if s >= 0] == [32, 64]


def test_lru_eviction_skips_pinned_states_and_reports_exhaustion():
    kda = _kda()
    ix = kda.PrefixIndex(4, match_unit=16, interval=0)
    # three prompts, each keeps its last boundary: 3 cached states + 3 private slots > 4 slots
    plans = []
    for sid in (1, 2):
        p = ix.plan(toks((sid, 20)))
        ix.commit(p)
        ix.release_slot(p.private_slot)
        plans.append(p)
    assert ix.free_slots() == 2
    # a hit pins prompt 1's state; then new prompts evict prompt 2's (least recently used, unpinned)
    h = ix.plan(np.concatenate([toks((1, 16)), toks((7, 3))]))
    assert h.src_slot == plans[0].ckpt_slots[0]
    n1 = ix.plan(toks((3, 20)))  # takes the last free slot (private) + evicts prompt 2 for its checkpoint
    assert n1.ckpt_slots[0] == plans[1].ckpt_slots[0]
    assert ix.free_slots() == 0
    # everything is now pinned or pending: no private slot can be found
    with pytest.raises(kda.KdaError) as e:
        ix.plan(toks((4, 20)))
    assert e.value.rc == kda.KDA_ERR_WORKSPACE
    # prompt 2 was evicted: it misses
    ix.commit(h)
    ix.commit(n1)
    ix.release_slot(h.private_slot)
    m = ix.plan(np.concatenate([toks((2, 16)), toks((5, 1))]))
    assert m.src_slot == -1


def test_abort_returns_slots_and_restores_ghosts():
    kda = _kda()
    ix = kda.PrefixIndex(6, match_unit=16, policy=kda.KDA_RETAIN_SECOND_HIT)
    ix.commit(ix.plan(toks((1, 40))))
    assert ix.free_slots() == 5  # the first request's private slot is still held
    p = ix.plan(toks((1, 40)))  # second sight: keeps boundary 32
    assert p.ckpt_slots == [-1, 0 + p.ckpt_slots[1]] and p.ckpt_slots[1] >= 0
    assert ix.free_slots() == 3
    ix.abort(p)
    assert ix.free_slots() == 5
    q = ix.plan(toks((1, 40)))  # the ghosts survived the abort: still a second sight
    assert q.ckpt_slots[1] >= 0
    with pytest.raises(kda.KdaError):
        ix.commit(p)  # an aborted plan is gone


def test_slot_accounting_and_invalid_arguments():
    kda = _kda()
    with pytest.raises(kda.KdaError):
        kda.PrefixIndex(4, match_unit=16, interval=24)  # interval not a multiple of the match unit
    with pytest.raises(kda.KdaError):
        kda.PrefixIndex(0)
    ix = kda.PrefixIndex(4, match_unit=16, interval=16)
    p = ix.plan(toks((1, 40)))
    cached = [s for s in p.ckpt_slots if s >= 0]
    assert ix.free_slots() == 4 - 1 - len(cached)
    ix.commit(p)
    with pytest.raises(kda.KdaError):
        ix.release_slot(cached[0])  # cached states leave by eviction only
    ix.release_slot(p.private_slot)
    with pytest.raises(kda.KdaError):
        ix.release_slot(p.private_slot)  # double release
    with pytest.raises(kda.KdaError):
        ix.release_slot(99)
    assert ix.free_slots() == 4 - len(cached)
    e = ix.plan(np.zeros(0, dtype=np.int32))  # an empty prompt: a fresh private slot, no checkpoints
    assert e.src_slot == -1 and e.ckpt_slots == []
    short = ix.plan(toks((5, 10)))  # shorter than one match unit
    assert short.ckpt_slots == [] and short.start_pos == 0


def test_many_requests_keep_the_pool_consistent():
    """Random traffic: every slot is always exactly one of free, private or cached."""
    kda = _kda()
    rng = np.random.default_rng(3)
    for policy in (kda.KDA_RETAIN_INTERVAL, kda.KDA_RETAIN_SECOND_HIT):
        ix = kda.PrefixIndex(24, match_unit=16, policy=policy, interval=32)
        cached, live = {}, []
        for step in range(300):
            prefix = int(rng.integers(0, 4))
            prompt = np.concatenate([toks((prefix + 1, int(rng.integers(0, 70)))),
                                     toks((100 + step, int(rng.integers(1, 40))))])
            try:
                p = ix.plan(prompt)
            except kda.KdaError:
                for s in live:
                    ix.release_slot(s)
                live = []
                continue
            if p.src_slot >= 0:
                assert p.src_slot in cached.values()
                assert p.start_pos % 16 == 0 and 0 < p.start_pos < len(prompt)
            assert p.private_slot not in live
            if rng.random() < 0.1:
                ix.abort(p)  # the private slot and the new checkpoints return to the free list
                continue
            for j, s in enumerate(p.ckpt_slots):
                if s >= 0:
                    assert s not in live and s != p.private_slot
                    cached[(step, j)] = s
            ix.commit(p)
            live.append(p.private_slot)
            if len(live) > 3:
                ix.release_slot(live.pop(0))
            assert len(set(live)) == len(live)
            assert ix.free_slots() + len(live) <= 24


# --------------------------------------------------------------------------- plans driving the fp64 oracle


class Requests:
    """Prompts built from (segment, length) pieces; layer inputs of a piece depend only on the piece, so equal
    token prefixes have equal inputs (as the inputs of a layer deep in a model would)."""

    def __init__(self, H, dk, dv, seed):
        self.H, self.dk, self.dv, self.seed = H, dk, dv, seed

    def build(self, segs):
        parts = [ki.token_inputs(self.seed * 1000 + sid, n, self.H, self.dk, self.dv) for sid, n in segs]
        inp = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
        return toks(*segs), inp


def _oracle_serve(ix, pools, cfg, wts, segs, req, U):
    tokens, inp = req.build(segs)
    L = len(tokens)
    p = ix.plan(tokens)
    S, C = pools
    if p.src_slot >= 0:  # copy-on-write into the private slot, then prefill from the boundary
        r = oracle.resume_pool(S, C, [p.src_slot], [p.private_slot])
        S, C = r["pool_S"], r["pool_conv"]
    s = p.start_pos
    f = {k: ki.bf16_bits_to_f64(v[s:]) for k, v in inp.items()}
    r = oracle.prefill_pool(cfg, S, C, [0, L - s], [s], [p.private_slot if p.src_slot >= 0 else -1],
                            [p.private_slot], U, p.ckpt_slots, f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                            wts["conv_w"], wts["norm_w"])
    ix.commit(p)
    return p, r, (r["pool_S"], r["pool_conv"]), inp


def _scratch(cfg, wts, inp):
    f = {k: ki.bf16_bits_to_f64(v) for k, v in inp.items()}
    T = f["q"].shape[0]
    return oracle.forward(cfg, [0, T], [0], f["q"], f["k"], f["v"], f["a"], f["b"], f["z"], wts["conv_w"],
                          wts["norm_w"], np.zeros((1, cfg.H, cfg.dk, cfg.dv)),
                          np.zeros((1, cfg.H, cfg.W - 1, cfg.Cc)))


@pytest.mark.parametrize("policy", [0, 1])
def test_plans_drive_the_oracle_to_the_from_scratch_result(policy):
    kda = _kda()
    H, dk, dv, U = 2, 16, 16, 16
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
    wts = ki.layer_weights(11, H, dk, dv)
    req = Requests(H, dk, dv, seed=7)
    ix = kda.PrefixIndex(12, match_unit=U, policy=policy, interval=32)
    pools = (np.zeros((12, H, dk, dv)), np.zeros((12, H, 3, 2 * dk + dv)))
    traffic = [[(1, 40), (2, 30)], [(1, 40), (3, 25)], [(1, 40), (2, 30), (4, 20)], [(1, 40), (5, 9)],
               [(1, 40), (3, 25), (6, 33)]]
    resumed = 0
    for segs in traffic:
        p, r, pools, inp = _oracle_serve(ix, pools, cfg, wts, segs, req, U)
        ref = _scratch(cfg, wts, inp)
        s = p.start_pos
        resumed += s > 0
        np.testing.assert_array_equal(r["y"], ref["y"][s:])
        np.testing.assert_array_equal(pools[0][p.private_slot], ref["S"][0])
        np.testing.assert_array_equal(pools[1][p.private_slot], ref["conv"][0])
        for j, slot in enumerate(p.ckpt_slots):  # a kept checkpoint is the from-scratch state at its boundary
            if slot >= 0:
                b = (s // U + 1 + j) * U
                fb = {k: v[:b] for k, v in inp.items()}
                np.testing.assert_array_equal(pools[0][slot], _scratch(cfg, wts, fb)["S"][0])
        ix.release_slot(p.private_slot)
    assert resumed >= 3


# --------------------------------------------------------------------------- plans driving the GPU kernels


@pytest.mark.gpu
def test_plans_drive_the_kernels():
    """The same traffic through the kernels (dk = dv = 128, chunk 64, match unit 128): outputs and states
    within the parity bars of the from-scratch oracle, and every resumed output equal bit for bit to the
    kernels' own from-scratch prefill (chunks are aligned to absolute positions)."""
    import torch
    from tests.kda_testutil import S_TOL, Y_TOL, bf16_dev_to_f64, s_err, to_dev_bf16, y_err
    kda = _kda()
    H, dk, dv, U, chunk, NS = 4, 128, 128, 128, 64, 16
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
    wts = ki.layer_weights(13, H, dk, dv)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    req = Requests(H, dk, dv, seed=9)
    pool = kda.StatePool.empty(NS + 1, H, dk, dv)
    pool.S.zero_()
    pool.conv.zero_()
    ix = kda.PrefixIndex(NS, match_unit=U, interval=256)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device="cuda")  # noqa: E731

    def prefill(inp, s, src, dst, ck_slots, interval):
        L = inp["q"].shape[0]
        d = {k: to_dev_bf16(v[s:]) for k, v in inp.items()}
        y = torch.empty(L - s, H, dv, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(kda.kda_prefill_workspace_bytes(pool, 1, L - s, chunk), 16), dtype=torch.uint8,
                         device="cuda")
        n = len(ck_slots)
        kda.kda_prefill_chunked(pool, prm, t([0, L - s], torch.int32), t([s], torch.int64), t([src], torch.int32),
                                t([dst], torch.int32), chunk, interval, t([0, n], torch.int32),
                                t(ck_slots if n else [0], torch.int32), d["q"], d["k"], d["v"], d["a"], d["b"],
                                d["z"], y, ws, st)
        return y

    traffic = [[(1, 600), (2, 150)], [(1, 600), (3, 77)], [(1, 600), (2, 150), (4, 300)], [(1, 600), (5, 1)]]
    resumed = 0
    for segs in traffic:
        tokens, inp = req.build(segs)
        p = ix.plan(tokens)
        if p.src_slot >= 0:
            kda.kda_resume_from_slot(pool, t([p.src_slot], torch.int32), t([p.private_slot], torch.int32), st)
        s = p.start_pos
        y = prefill(inp, s, p.private_slot if p.src_slot >= 0 else -1, p.private_slot, p.ckpt_slots, U)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ix.commit(p)
        resumed += s > 0
        ref = _scratch(cfg, wts, inp)
        assert y_err(bf16_dev_to_f64(y), ref["y"][s:]) <= Y_TOL
        assert s_err(pool.S[p.private_slot].cpu().numpy(), ref["S"][0]) <= S_TOL
        # replay from scratch on the kernels into the spare slot NS: the resumed tail is identical
        y_full = prefill(inp, 0, -1, NS, [], 0)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_full[s:].view(torch.int16))
        assert torch.equal(pool.S[p.private_slot], pool.S[NS])
        ix.release_slot(p.private_slot)
    assert resumed >= 3
