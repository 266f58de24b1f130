"""Failure detection on the GPU without a fault: a bounded wait that runs out reports KDA_DEV_TIMEOUT and
leaves the context usable; a NaN injected into one request or sequence stays in it (every other request's
output and state are bit-for-bit those of a clean run)."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
from tests.kda_testutil import fill_pool, to_dev_bf16

pytestmark = pytest.mark.gpu

BF16_NAN = np.uint16(0x7FC0)


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


def test_bounded_wait_gives_up_and_the_context_survives():
    kda = _kda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_selftest_wait_timeout(50_000_000, st)  # 50 ms
    torch.cuda.synchronize()
    assert int(st.item()) == kda.KDA_DEV_TIMEOUT
    # the context still works: a decode step right after it succeeds
    H, dk, dv = 2, 128, 128
    pool = kda.StatePool.empty(4, H, dk, dv)
    wts = ki.layer_weights(1, H, dk, dv)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    d = {k: to_dev_bf16(v) for k, v in ki.token_inputs(1, 2, H, dk, dv).items()}
    y = torch.empty(2, H, dv, dtype=torch.bfloat16, device="cuda")
    st.zero_()
    s = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, s, s, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and bool(torch.isfinite(y.float()).all())


def _decode_once(kda, seed, tok, n, H, dk, dv, slots):
    pool = kda.StatePool.empty(2 * n, H, dk, dv)
    fill_pool(pool, seed)
    wts = ki.layer_weights(seed, H, dk, dv)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    d = {k: to_dev_bf16(v) for k, v in tok.items()}
    y = torch.empty(n, H, dv, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.tensor(slots, dtype=torch.int32, device="cuda")
    kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, s, s, st)
    torch.cuda.synchronize()
    return y, pool, int(st.item())


@pytest.mark.parametrize("field", ["q", "k", "v", "a", "b", "z"])
def test_nan_in_one_decode_request_stays_in_it(field):
    kda = _kda()
    n, H, dk, dv, seed, bad = 8, 4, 128, 128, 31, 3
    slots = [1, 3, 5, 7, 9, 11, 13, 15]
    tok = ki.token_inputs(seed, n, H, dk, dv)
    y0, p0, st0 = _decode_once(kda, seed, tok, n, H, dk, dv, slots)
    t2 = {k: v.copy() for k, v in tok.items()}
    t2[field][bad].reshape(-1)[0] = BF16_NAN  # one element of request 3, head 0
    y1, p1, st1 = _decode_once(kda, seed, t2, n, H, dk, dv, slots)
    assert st0 == 0 and st1 == 0
    ok = [r for r in range(n) if r != bad]
    assert torch.equal(y0[ok].view(torch.int16), y1[ok].view(torch.int16))
    keep = [s for i, s in enumerate(slots) if i != bad] + [s for s in range(2 * n) if s not in slots]
    assert torch.equal(p0.S[keep], p1.S[keep])
    assert torch.equal(p0.conv[keep].view(torch.int16), p1.conv[keep].view(torch.int16))
    assert not bool(torch.isfinite(y1[bad, 0].float()).all())  # the poisoned request shows it
    assert torch.equal(y0[bad, 1:].view(torch.int16), y1[bad, 1:].view(torch.int16))  # other heads: untouched


@pytest.mark.parametrize("dk,chunk", [(128, 64), (64, 16)])
def test_nan_in_one_prefill_sequence_stays_in_it(dk, chunk):
    """Three sequences (the tensor-core path at d = 128, the SIMT path at d = 64); a NaN in one token of the
    middle sequence leaves the outputs, final states and checkpoints of the other two bit-for-bit unchanged."""
    kda = _kda()
    H, dv, seed = 3, dk, 41
    lens = [3 * chunk + 7, 2 * chunk + 5, 4 * chunk]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    interval = 2 * chunk
    counts = [l // interval for l in lens]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ck = np.arange(10, 10 + int(offs[-1]), dtype=np.int32)
    tok = ki.token_inputs(seed, T, H, dk, dv)
    wts = ki.layer_weights(seed, H, dk, dv)
    t = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device="cuda")  # noqa: E731

    def run(tk):
        pool = kda.StatePool.empty(10 + len(ck), H, dk, dv)
        prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
        d = {k: to_dev_bf16(v) for k, v in tk.items()}
        y = torch.empty(T, H, dv, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, 3, T, chunk), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.kda_prefill_chunked(pool, prm, t(cu, torch.int32), t([0, 0, 0], torch.int64), t([-1, -1, -1], torch.int32),
                                t([0, 1, 2], torch.int32), chunk, interval, t(offs, torch.int32), t(ck, torch.int32),
                                d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, ws, st)
        torch.cuda.synchronize()
        return y, pool, int(st.item())

    y0, p0, s0 = run(tok)
    t2 = {k: v.copy() for k, v in tok.items()}
    t2["k"][cu[1] + chunk + 3, 1, 5] = BF16_NAN  # sequence 1, its second chunk, head 1
    y1, p1, s1 = run(t2)
    assert s0 == 0 and s1 == 0
    other = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
    assert torch.equal(y0[other].view(torch.int16), y1[other].view(torch.int16))
    good_slots = [0, 2] + [int(x) for x in ck[offs[0]:offs[1]]] + [int(x) for x in ck[offs[2]:offs[3]]]
    assert torch.equal(p0.S[good_slots], p1.S[good_slots])
    assert torch.equal(p0.conv[good_slots].view(torch.int16), p1.conv[good_slots].view(torch.int16))
    # in sequence 1 the tokens before the NaN and the other heads are untouched; head 1 after it is not finite
    assert torch.equal(y0[cu[1]:cu[1] + chunk].view(torch.int16), y1[cu[1]:cu[1] + chunk].view(torch.int16))
    assert torch.equal(y0[cu[1]:cu[2], 0].view(torch.int16), y1[cu[1]:cu[2], 0].view(torch.int16))
    assert not bool(torch.isfinite(y1[cu[2] - 1, 1].float()).all())
