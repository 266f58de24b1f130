"""kda_prefill_chunked_noalloc, the prefill entry point for callers that cannot allocate device memory
(for example an engine whose caching allocator owns all free GPU memory, or a plug-in handed only
tensors).  It takes no workspace: the library's fixed scratch array stands in for it.  It runs the same
kernels on the same inputs as kda_prefill_chunked, so its results must be identical bit for bit; a
tolerance would hide a stale-scratch fault.

This file sorts last so that, if it fails, a run stopping at the first failure has already run every
other test.  It must also pass alone in a fresh process.
"""

import numpy as np
import pytest
import torch

from tests.kda_testutil import fill_pool, to_dev_bf16

pytestmark = pytest.mark.gpu

import kda_inputs as ki  # noqa: E402


def _problem(kda, H, lens, starts, src, dst, chunk, interval, slots, seed):
    pool = kda.StatePool.empty(slots, H, 128, 128)
    fill_pool(pool, seed)
    w = ki.layer_weights(seed, H, 128, 128)
    prm = kda.LayerParams(torch.from_numpy(w["conv_w"]).cuda(), torch.from_numpy(w["norm_w"]).cuda())
    T = int(sum(lens))
    tok = {k: to_dev_bf16(v) for k, v in ki.token_inputs(seed, T, H, 128, 128).items()}
    counts = [kda.kda_checkpoint_count(s, l, interval) for s, l in zip(starts, lens)]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    used = set(s for s in src if s >= 0) | set(dst)
    ck = np.array([s for s in range(slots) if s not in used][:int(offs[-1])], dtype=np.int32)
    i32 = lambda a: torch.tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa: E731
    args = (i32(np.concatenate([[0], np.cumsum(lens)])), torch.tensor(starts, dtype=torch.int64, device="cuda"),
            i32(src), i32(dst), chunk, interval, i32(offs), i32(ck))
    return pool, prm, T, tok, args, ck


def test_noalloc_prefill_matches_workspace_entry_point_on_two_calls():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    H, chunk, interval = 8, 64, 128
    lens, starts, src, dst = [300, 77, 129], [0, 64, 5], [-1, 2, 4], [1, 2, 5]
    pool, prm, T, tok, args, ck = _problem(kda, H, lens, starts, src, dst, chunk, interval, 24, seed=77)
    assert kda.kda_prefill_workspace_bytes(pool, len(lens), T, chunk) <= kda.NOALLOC_SCRATCH_BYTES
    start_S, start_C = pool.S.clone(), pool.conv.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # the existing entry point, with a workspace the caller allocated
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, len(lens), T, chunk), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_prefill_chunked(pool, prm, *args, tok["q"], tok["k"], tok["v"], tok["a"], tok["b"], tok["z"], y_ref, ws,
                            status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    S_ref, C_ref = pool.S.clone(), pool.conv.clone()
    written = sorted(set(dst) | set(int(c) for c in ck))

    for call in range(2):  # the second call runs on the scratch the first one left behind
        pool.S.copy_(start_S)
        pool.conv.copy_(start_C)
        y = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
        kda.kda_prefill_chunked_noalloc(pool, prm, *args, tok["q"], tok["k"], tok["v"], tok["a"], tok["b"],
                                        tok["z"], y, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), call
        assert torch.equal(pool.S, S_ref), call  # written slots equal, untouched slots unchanged
        assert torch.equal(pool.conv.view(torch.int16), C_ref.view(torch.int16)), call
        untouched = [s for s in range(24) if s not in written]
        assert torch.equal(pool.S[untouched], start_S[untouched])


def test_noalloc_setup_call_and_argument_checks():
    """A call with nseq = 0 does the per-device set-up and launches nothing; bad arguments are rejected with
    KDA_ERR_INVALID_ARG by the host checks, before any device call."""
    import hybrid_linear_attention_decode_gb300 as kda
    lib = kda.load_library()
    pool = kda.StatePool.empty(4, 2, 128, 128)
    prm = kda.LayerParams(torch.zeros(2, 384, 4, device="cuda"), torch.ones(128, device="cuda"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    # nseq = 0: the set-up call
    kda.kda_prefill_chunked_noalloc(pool, prm, i32([0]), torch.zeros(0, dtype=torch.int64, device="cuda"),
                                    i32([0])[:0], i32([0])[:0], 64, 0, i32([0]), i32([0]), None, None, None, None,
                                    None, None, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # a NULL pool and NULL params: KDA_ERR_INVALID_ARG, whatever the sizes
    rc = lib.kda_prefill_chunked_noalloc(None, None, 1, 64, *([None] * 4), 64, 0, *([None] * 9), None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    assert "pool" in kda.kda_last_error_string() or "params" in kda.kda_last_error_string()
    # an interval that is not a multiple of the chunk
    with pytest.raises(kda.KdaError) as err:
        kda.kda_prefill_chunked_noalloc(pool, prm, i32([0, 64]), torch.zeros(1, dtype=torch.int64, device="cuda"),
                                        i32([-1]), i32([0]), 64, 100, i32([0, 0]), i32([0]), e(64, 2, 128),
                                        e(64, 2, 128), e(64, 2, 128), e(64, 2, 128), e(64, 2), None, e(64, 2, 128),
                                        status)
    assert err.value.rc == kda.KDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_noalloc_prefill_rejects_problems_beyond_the_scratch():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    H = 32
    lens = [1024, 1024]
    pool, prm, T, tok, args, ck = _problem(kda, H, lens, [0, 0], [-1, -1], [0, 1], 64, 128, 64, seed=5)
    assert kda.kda_prefill_workspace_bytes(pool, 2, T, 64) > kda.NOALLOC_SCRATCH_BYTES
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    before = pool.S.clone()
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_chunked_noalloc(pool, prm, *args, tok["q"], tok["k"], tok["v"], tok["a"], tok["b"],
                                        tok["z"], y, status)
    assert e.value.rc == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(pool.S, before)
