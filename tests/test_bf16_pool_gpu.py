"""The bf16 state pool ("moonshotai/Kimi-K3" recipe: --mamba-ssm-cache-dtype bfloat16) on the GPU.

Kernels compute in fp32 and round a state to bf16 (nearest even) where they store it.  The oracle is
given the same storage semantics (it rounds every state it writes to the pool), and the bars are the
usual output bar (2e-2); a stored state is compared with the oracle's unrounded value at 1e-3 + 2^-9
relative Frobenius (the compute bar plus the largest relative rounding error of bf16 storage); windows
and untouched slots are bit-exact.  (Against the fp32-pool recurrence a bf16 pool drifts by about 5e-3
in the state after tens of decode steps; that is the storage format's cost, not a kernel error.)
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.kda_testutil import S_TOL_BF16, Y_TOL, bf16_dev_bits, bf16_dev_to_f64, fill_pool, pool_unit_host, s_err, \
    to_dev_bf16, y_err
from tests.test_prefill_gpu import Problem

pytestmark = pytest.mark.gpu


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 16), (128, 128)])
def test_bf16_pool_decode_multi_step(dk, dv):
    kda = _kda()
    H, slots, n, steps = 3, 16, 5, 6
    pool = kda.StatePool.empty(slots, H, dk, dv, state_dtype=torch.bfloat16)
    S_h, C_h = fill_pool(pool, 70 + dk)
    w = ki.layer_weights(70 + dk, H, dk, dv)
    prm = kda.LayerParams(torch.from_numpy(w["conv_w"]).cuda(), torch.from_numpy(w["norm_w"]).cuda())
    src = [2, -1, 7, 9, 11]
    dst = [2, 3, 8, 9, 12]
    # host model of the pool: the bf16 rounding of the generated contents
    pS = np.stack([oracle.round_to_bf16(pool_unit_host(S_h, C_h, s_, H)[0]) for s_ in range(slots)])
    pC = np.stack([pool_unit_host(S_h, C_h, s_, H)[1] for s_ in range(slots)])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = oracle.Cfg(H=H, dk=dk, dv=dv)
    tok = ki.token_inputs(71, steps * n, H, dk, dv)
    for s in range(steps):
        cur_src = src if s == 0 else dst
        sl = slice(s * n, (s + 1) * n)
        d = {k_: to_dev_bf16(np.ascontiguousarray(v_[sl])) for k_, v_ in tok.items()}
        y = torch.empty(n, H, dv, dtype=torch.bfloat16, device="cuda")
        kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y,
                            torch.tensor(cur_src, dtype=torch.int32, device="cuda"),
                            torch.tensor(dst, dtype=torch.int32, device="cuda"), status)
        f = {k_: ki.bf16_bits_to_f64(v_[sl]) for k_, v_ in tok.items()}
        ref = oracle.decode_pool(cfg, pS, pC, cur_src, dst, f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                                 w["conv_w"], w["norm_w"], state_bf16=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert y_err(bf16_dev_to_f64(y), ref["y"]) <= Y_TOL, s
        got = pool.S.float().cpu().numpy()
        for dd in dst:
            assert s_err(got[dd], ref["pool_S"][dd]) <= S_TOL_BF16, (s, dd)
            np.testing.assert_array_equal(ki.bf16_bits_to_f64(bf16_dev_bits(pool.conv[dd])), ref["pool_conv"][dd])
        # the oracle carries its own (rounded) pool forward; the two sides evolve independently
        pS, pC = ref["pool_S"], ref["pool_conv"]
    untouched = [s_ for s_ in range(slots) if s_ not in dst]
    np.testing.assert_array_equal(pool.S.float().cpu().numpy()[untouched],
                                  np.stack([oracle.round_to_bf16(pool_unit_host(S_h, C_h, s_, H)[0])
                                            for s_ in untouched]))


@pytest.mark.parametrize("dk,dv,chunk", [(16, 16, 16), (128, 128, 64)])
def test_bf16_pool_prefill_with_checkpoints(dk, dv, chunk):
    kda = _kda()
    interval = 2 * chunk
    p = Problem(kda, 3, dk, dv, [3 * chunk + 5, 2 * chunk], [0, interval], [-1, 4], [2, 4], chunk, interval, 24,
                seed=90 + dk, sbf16=True)
    assert p.run() == 0
    p.check(p.reference())


def test_bf16_pool_resume_copies_bits():
    kda = _kda()
    pool = kda.StatePool.empty(16, 4, 128, 128, state_dtype=torch.bfloat16)
    fill_pool(pool, 5, unique=64)
    before = pool.S.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_resume_from_slot(pool, torch.tensor([1, 3], dtype=torch.int32, device="cuda"),
                             torch.tensor([10, 11], dtype=torch.int32, device="cuda"), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pool.S[10].view(torch.int16), before[1].view(torch.int16))
    assert torch.equal(pool.S[11].view(torch.int16), before[3].view(torch.int16))
