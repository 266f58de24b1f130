"""Fused decode step on the GPU (through the C ABI) against the fp64 oracle, element by element.

Bars: bf16 outputs within 2e-2 (max over (request, head) of max|y - y_ref| / max|y_ref|), fp32 states
within 1e-3 relative Frobenius per (request, head), conv windows and every untouched slot bit-exact.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.kda_testutil import (S_TOL, Y_TOL, bf16_dev_bits, bf16_dev_to_f64, fill_pool, pool_unit_host, s_err,
                                to_dev_bf16, y_err)

pytestmark = pytest.mark.gpu


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


def _setup(H, dk, dv, num_slots, n, seed, src, dst, with_z=True, W=4):
    kda = _kda()
    pool = kda.StatePool.empty(num_slots, H, dk, dv, W)
    S_h, C_h = fill_pool(pool, seed)
    wts = ki.layer_weights(seed, H, dk, dv, W)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    tok = ki.token_inputs(seed, n, H, dk, dv, with_z=with_z)
    dev = {k_: (to_dev_bf16(v_) if v_ is not None else None) for k_, v_ in tok.items()}
    y = torch.empty(n, H, dv, dtype=torch.bfloat16, device="cuda")
    src_t = torch.tensor(src, dtype=torch.int32, device="cuda")
    dst_t = torch.tensor(dst, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    return kda, pool, S_h, C_h, wts, prm, tok, dev, y, src_t, dst_t, status


def _run(kda, pool, prm, dev, y, src_t, dst_t, status):
    kda.kda_decode_step(pool, prm, dev["q"], dev["k"], dev["v"], dev["a"], dev["b"], dev["z"], y, src_t, dst_t,
                        status)
    torch.cuda.synchronize()


def _oracle_for(req_ids, S_h, C_h, src, wts, tok, H, dk, dv, W=4):
    """fp64 oracle for the listed requests (their initial states from the host copy of the pool)."""
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv, W=W)
    S0 = np.zeros((len(req_ids), H, dk, dv))
    C0 = np.zeros((len(req_ids), H, W - 1, 2 * dk + dv))
    for i, r in enumerate(req_ids):
        if src[r] >= 0:
            S0[i], C0[i] = pool_unit_host(S_h, C_h, src[r], H)
    f = {k_: (ki.bf16_bits_to_f64(v_[req_ids]) if v_ is not None else None) for k_, v_ in tok.items()}
    return oracle.forward(cfg, np.arange(len(req_ids) + 1), np.zeros(len(req_ids), dtype=np.int64), f["q"], f["k"],
                          f["v"], f["a"], f["b"], f["z"], wts["conv_w"], wts["norm_w"], S0, C0)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 16), (16, 32), (64, 64), (128, 128)])
@pytest.mark.parametrize("with_z", [True, False])
def test_decode_matches_oracle_small(dk, dv, with_z):
    H, num_slots, n = 3, 24, 7
    src = [5, -1, 11, 2, 20, 7, -1]
    dst = [5, 13, 11, 3, 21, 8, 9]       # in place, fresh, in place, moved, moved, moved, fresh
    kda, pool, S_h, C_h, wts, prm, tok, dev, y, src_t, dst_t, status = _setup(H, dk, dv, num_slots, n, 100 + dk + dv,
                                                                              src, dst, with_z)
    S_before = pool.S.clone()
    C_before = pool.conv.clone()
    _run(kda, pool, prm, dev, y, src_t, dst_t, status)
    assert int(status.item()) == 0
    ref = _oracle_for(list(range(n)), S_h, C_h, src, wts, tok, H, dk, dv)
    assert y_err(bf16_dev_to_f64(y), ref["y"]) <= Y_TOL
    S_after = pool.S.cpu().numpy()
    for r in range(n):
        assert s_err(S_after[dst[r]], ref["S"][r]) <= S_TOL
        np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(pool.conv[dst[r]])), ref["conv"][r])
    untouched = [s for s in range(num_slots) if s not in dst]
    assert torch.equal(pool.S[untouched], S_before[untouched])
    assert torch.equal(pool.conv[untouched].view(torch.int16), C_before[untouched].view(torch.int16))


def test_decode_full_size_sampled():
    """The decode-step workload at full size (batch 64, H=32, dk=dv=128, 4096-slot pool, random distinct
    slots, in place), in the launch configuration the benchmark times; sampled requests against the
    oracle, every other slot bit-exact."""
    H, dk, dv, num_slots, n = 32, 128, 128, 4096, 64
    src = [int(s) for s in ki.random_slots(2, num_slots, n)]
    dst = list(src)
    kda, pool, S_h, C_h, wts, prm, tok, dev, y, src_t, dst_t, status = _setup(H, dk, dv, num_slots, n, 2, src, dst)
    snapS, snapC = pool.S.clone(), pool.conv.clone()
    _run(kda, pool, prm, dev, y, src_t, dst_t, status)
    assert int(status.item()) == 0
    sample = [0, 17, 40, 63]
    ref = _oracle_for(sample, S_h, C_h, src, wts, tok, H, dk, dv)
    assert y_err(bf16_dev_to_f64(y[sample]), ref["y"]) <= Y_TOL
    for i, r in enumerate(sample):
        assert s_err(pool.S[dst[r]].cpu().numpy(), ref["S"][i]) <= S_TOL
        np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(pool.conv[dst[r]])), ref["conv"][i])
    # every slot that is not a destination is bit-for-bit unchanged
    idx = dst_t.long()
    pool.S[idx] = snapS[idx]
    pool.conv[idx] = snapC[idx]
    assert torch.equal(pool.S, snapS)
    assert torch.equal(pool.conv.view(torch.int16), snapC.view(torch.int16))


def test_decode_bad_slots_flag_status_and_skip():
    H, dk, dv, num_slots, n = 2, 16, 16, 8, 4
    src = [1, 99, 2, -2]
    dst = [1, 3, 50, 4]
    kda, pool, S_h, C_h, wts, prm, tok, dev, y, src_t, dst_t, status = _setup(H, dk, dv, num_slots, n, 7, src, dst)
    S_before = pool.S.clone()
    _run(kda, pool, prm, dev, y, src_t, dst_t, status)
    assert int(status.item()) & kda.KDA_DEV_BAD_SLOT
    yf = bf16_dev_to_f64(y)
    assert np.all(yf[1:] == 0.0)
    assert torch.equal(pool.S[[0, 2, 3, 4, 5, 6, 7]], S_before[[0, 2, 3, 4, 5, 6, 7]])
    ref = _oracle_for([0], S_h, C_h, src, wts, tok, H, dk, dv)
    assert y_err(yf[:1], ref["y"]) <= Y_TOL


def test_decode_is_deterministic():
    H, dk, dv, num_slots, n = 8, 128, 128, 64, 16
    src = list(range(0, 32, 2))
    dst = list(range(33, 49))
    outs = []
    for _ in range(2):
        kda, pool, S_h, C_h, wts, prm, tok, dev, y, src_t, dst_t, status = _setup(H, dk, dv, num_slots, n, 9, src,
                                                                                  dst)
        _run(kda, pool, prm, dev, y, src_t, dst_t, status)
        outs.append((y.view(torch.int16).clone(), pool.S.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_multi_step_tracks_oracle():
    """Eight consecutive decode steps in place, state carried in the pool, against the oracle's
    token-by-token recurrence over the same eight tokens."""
    H, dk, dv, num_slots, n, steps = 4, 128, 128, 16, 3, 8
    src = [3, 7, -1]
    kda = _kda()
    pool = kda.StatePool.empty(num_slots, H, dk, dv)
    S_h, C_h = fill_pool(pool, 21)
    wts = ki.layer_weights(21, H, dk, dv)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    tok = ki.token_inputs(21, steps * n, H, dk, dv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dst = [3, 7, 12]
    ys = []
    for s in range(steps):
        sl = slice(s * n, (s + 1) * n)
        dev = {k_: to_dev_bf16(np.ascontiguousarray(v_[sl])) for k_, v_ in tok.items()}
        y = torch.empty(n, H, dv, dtype=torch.bfloat16, device="cuda")
        s_src = src if s == 0 else dst
        kda.kda_decode_step(pool, prm, dev["q"], dev["k"], dev["v"], dev["a"], dev["b"], dev["z"], y,
                            torch.tensor(s_src, dtype=torch.int32, device="cuda"),
                            torch.tensor(dst, dtype=torch.int32, device="cuda"), status)
        ys.append(bf16_dev_to_f64(y))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
    S0 = np.zeros((n, H, dk, dv))
    C0 = np.zeros((n, H, 3, 3 * dk))
    for r in range(n):
        if src[r] >= 0:
            S0[r], C0[r] = pool_unit_host(S_h, C_h, src[r], H)
    f = {k_: ki.bf16_bits_to_f64(v_).reshape(steps, n, *v_.shape[1:]).transpose(1, 0, *range(2, v_.ndim + 1))
         .reshape(n * steps, *v_.shape[1:]) for k_, v_ in tok.items()}
    ref = oracle.forward(cfg, np.arange(0, n * steps + 1, steps), np.zeros(n, dtype=np.int64), f["q"], f["k"],
                         f["v"], f["a"], f["b"], f["z"], wts["conv_w"], wts["norm_w"], S0, C0)
    y_gpu = np.stack(ys, 1).reshape(n * steps, H, dv)
    assert y_err(y_gpu, ref["y"]) <= Y_TOL
    for r in range(n):
        assert s_err(pool.S[dst[r]].cpu().numpy(), ref["S"][r]) <= S_TOL


def test_resume_copies_bit_exact_and_checks_slots():
    kda = _kda()
    H, dk, dv, num_slots = 4, 128, 128, 32
    pool = kda.StatePool.empty(num_slots, H, dk, dv)
    fill_pool(pool, 33, unique=num_slots * H)
    before_S, before_C = pool.S.clone(), pool.conv.clone()
    src = torch.tensor([1, 5, 9], dtype=torch.int32, device="cuda")
    dst = torch.tensor([20, 21, 22], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_resume_from_slot(pool, src, dst, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    exp = oracle.resume_pool(before_S.cpu().numpy(), bf16_dev_bits(before_C), [1, 5, 9], [20, 21, 22])
    np.testing.assert_array_equal(pool.S.cpu().numpy(), exp["pool_S"])
    np.testing.assert_array_equal(bf16_dev_bits(pool.conv), exp["pool_conv"])
    bad_dst = torch.tensor([23, 4096], dtype=torch.int32, device="cuda")
    kda.kda_resume_from_slot(pool, src[:2], bad_dst, status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_BAD_SLOT
    assert torch.equal(pool.S[23], before_S[1])
