"""Segmented prefill launches on the GPU (through the C ABI).

A call whose (sequence, head) chains would leave most SMs idle in the chunk chain (chains x 4 <= SMs, at
least 512 chunks) is launched in segments of about 128 chunks: the intra kernel of one segment runs beside
the state kernel of the segment before, and the state crosses a segment boundary in fp32 through the
workspace.  The arithmetic at a segment boundary is that at a chunk boundary inside one launch, so every
test here is bit-exact against the same work done by calls too small to be segmented:

  * one sequence, resumed from a random state at an unaligned position (a partial first chunk), with a
    checkpoint at every chunk end (so at every segment end, whatever the segment size), against the same
    tokens in two resumed calls;
  * three sequences (one empty) whose chunks are cut by segments at arbitrary points, against one call
    per sequence;
  * a bf16 state pool against the fp32 pool rounded to bf16 (outputs identical, states and checkpoints
    the bf16 rounding of the fp32 ones);
  * a call captured in a CUDA graph and replayed, against the eager call;
  * a resume in place (src == dst) against the same resume into another slot;
and, against the fp64 oracle, one head (so that a segmented workspace fits the no-alloc entry point's
static scratch) with a bf16 pool resumed from a stored state, no output gate and a skipped checkpoint.

The sizes are chosen so that the one-call side is segmented (at least 512 chunks, chains x 4 <= the SM
count, asserted) and every call it is compared with is not (fewer than 512 chunks).  The oracle
comparison of the segmented path at full size is the long-context test in test_prefill_gpu.py (one
131072-token sequence, 32 heads).
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
from tests.kda_testutil import fill_pool, to_dev_bf16

pytestmark = pytest.mark.gpu

D, CH = 128, 64


def _kda():
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    return kda


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tokens(seed, T, H):
    """bf16 token inputs drawn on the device (q, k, v, z ~ N(0,1), decay logits ~ N(3,1), beta logits ~ N(0,1))."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)

    def draw(*shape, shift=0.0):
        return (torch.randn(*shape, generator=g, device="cuda") + shift).to(torch.bfloat16)
    return dict(q=draw(T, H, D), k=draw(T, H, D), v=draw(T, H, D), a=draw(T, H, D, shift=3.0), b=draw(T, H),
                z=draw(T, H, D))


def _ckpt_count(start, length, interval):
    return (start + length) // interval - start // interval


def _call(kda, pool, prm, tok, t0, lens, starts, src, dst, interval, ck_slots):
    """One prefill call over tokens [t0, t0 + sum(lens)) of `tok`; returns y."""
    T = int(sum(lens))
    H = pool.S.shape[1]
    i32 = lambda a: torch.tensor(np.asarray(a, dtype=np.int64), dtype=torch.int32, device="cuda")  # noqa: E731
    cu = np.concatenate([[0], np.cumsum(lens)])
    counts = [_ckpt_count(s, l, interval) for s, l in zip(starts, lens)]
    offs = np.concatenate([[0], np.cumsum(counts)])
    assert len(ck_slots) == offs[-1]
    sl = {k: v[t0:t0 + T].contiguous() for k, v in tok.items()}  # zero rows for an empty call
    y = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(kda.kda_prefill_workspace_bytes(pool, len(lens), T, CH), 16), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xCD)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill_chunked(pool, prm, i32(cu), torch.tensor(starts, dtype=torch.int64, device="cuda"), i32(src),
                            i32(dst), CH, interval, i32(offs), i32(ck_slots if len(ck_slots) else [0]), sl["q"],
                            sl["k"], sl["v"], sl["a"], sl["b"], sl["z"], y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y


def _setup(kda, H, num_slots, seed, sdt=torch.float32):
    pool = kda.StatePool.empty(num_slots, H, D, D, state_dtype=sdt)
    fill_pool(pool, seed)
    wts = ki.layer_weights(seed, H, D, D)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).cuda(), torch.from_numpy(wts["norm_w"]).cuda())
    return pool, prm


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def _same(x, y):
    """Bitwise equality on the device."""
    it = torch.int16 if x.element_size() == 2 else torch.int32
    return torch.equal(x.contiguous().view(it), y.contiguous().view(it))


def test_segmented_call_equals_two_resumed_calls():
    kda = _kda()
    # chunk 0 is [1064, 1088); with an interval of one chunk every chunk end is a checkpoint
    H, interval, T, start = 32, CH, 40000, 1064
    assert H * 4 <= _sms() and T // CH >= 512
    nck = _ckpt_count(start, T, interval)
    assert nck == 625
    pool, prm = _setup(kda, H, 2 * nck + 8, seed=81)
    tok = _tokens(82, T, H)
    cks = list(range(8, 8 + nck))
    src_S = pool.S[1].clone()
    # one call: the segmented path
    yA = _call(kda, pool, prm, tok, 0, [T], [start], [1], [2], interval, cks)
    assert _same(pool.S[1], src_S)  # the source slot is untouched
    # the same tokens in two calls small enough for single launches, resumed through slot 3 at a chunk-aligned
    # position (a call boundary inside an aligned chunk would split that chunk differently)
    T1 = 16024
    assert (start + T1) % CH == 0
    n1 = _ckpt_count(start, T1, interval)
    cks_b = list(range(8 + nck, 8 + 2 * nck))
    y1 = _call(kda, pool, prm, tok, 0, [T1], [start], [1], [3], interval, cks_b[:n1])
    y2 = _call(kda, pool, prm, tok, T1, [T - T1], [start + T1], [3], [4], interval, cks_b[n1:])
    np.testing.assert_array_equal(_bits(yA), _bits(torch.cat([y1, y2])))
    assert _same(pool.S[2], pool.S[4]) and _same(pool.conv[2], pool.conv[4])
    bad = [j for j in range(nck) if not (_same(pool.S[cks[j]], pool.S[cks_b[j]])
                                         and _same(pool.conv[cks[j]], pool.conv[cks_b[j]]))]
    assert not bad, f"checkpoints differ at {bad[:8]}"


def test_segmented_in_place_resume_equals_moved_resume():
    """A segmented call resuming one sequence in place (src == dst, the plan the prefix index makes) gives, bit
    for bit, what the same call gives from a copy of the source into another destination: the history rows
    the first segment reads come from the table kernel's snapshot of the source window, not from the slot the
    last segment overwrites."""
    kda = _kda()
    H, interval, T, start = 8, 4096, 33000, 4096 + 17
    assert H * 4 <= _sms() and T // CH >= 512
    nck = _ckpt_count(start, T, interval)
    pool, prm = _setup(kda, H, 8 + 2 * nck, seed=91)
    tok = _tokens(92, T, H)
    pool.S[2].copy_(pool.S[1])
    pool.conv[2].copy_(pool.conv[1])
    cks_a, cks_b = list(range(8, 8 + nck)), list(range(8 + nck, 8 + 2 * nck))
    yA = _call(kda, pool, prm, tok, 0, [T], [start], [1], [1], interval, cks_a)  # in place
    yB = _call(kda, pool, prm, tok, 0, [T], [start], [2], [3], interval, cks_b)  # moved
    np.testing.assert_array_equal(_bits(yA), _bits(yB))
    assert _same(pool.S[1], pool.S[3]) and _same(pool.conv[1], pool.conv[3])
    for a_, b_ in zip(cks_a, cks_b):
        assert _same(pool.S[a_], pool.S[b_]) and _same(pool.conv[a_], pool.conv[b_])


def test_segmented_call_equals_per_sequence_calls():
    kda = _kda()
    H, interval = 8, 4096
    lens, starts, src, dst = [20000, 0, 15050], [0, 77, 3000], [-1, 5, 6], [1, 2, 3]
    T = sum(lens)
    assert len(lens) * H * 4 <= _sms() and T // CH >= 512
    pool, prm = _setup(kda, H, 40, seed=91)
    tok = _tokens(92, T, H)
    counts = [_ckpt_count(s, l, interval) for s, l in zip(starts, lens)]
    cks = list(range(8, 8 + sum(counts)))
    yA = _call(kda, pool, prm, tok, 0, lens, starts, src, dst, interval, cks)
    outA = [(_bits(pool.S[d]), _bits(pool.conv[d])) for d in dst]
    ckA = [(_bits(pool.S[s]), _bits(pool.conv[s])) for s in cks]
    # one call per sequence, each below the segmentation bound, into fresh slots
    dstB = [21, 22, 23]
    cksB = list(range(24, 24 + sum(counts)))
    ys, t0, o = [], 0, 0
    for n in range(len(lens)):
        ys.append(_call(kda, pool, prm, tok, t0, [lens[n]], [starts[n]], [src[n]], [dstB[n]], interval,
                        cksB[o:o + counts[n]]))
        t0 += lens[n]
        o += counts[n]
    np.testing.assert_array_equal(_bits(yA), _bits(torch.cat(ys)))
    for n, d in enumerate(dstB):
        np.testing.assert_array_equal(outA[n][0], _bits(pool.S[d]), err_msg=f"state {n}")
        np.testing.assert_array_equal(outA[n][1], _bits(pool.conv[d]), err_msg=f"window {n}")
    for j, s in enumerate(cksB):
        np.testing.assert_array_equal(ckA[j][0], _bits(pool.S[s]), err_msg=f"checkpoint {j}")
        np.testing.assert_array_equal(ckA[j][1], _bits(pool.conv[s]), err_msg=f"checkpoint window {j}")


def test_segmented_bf16_pool_is_the_rounded_fp32_pool():
    kda = _kda()
    H, interval, T = 32, 16384, 36000
    assert H * 4 <= _sms() and T // CH >= 512
    tok = _tokens(101, T, H)
    cks = [4, 5]
    res = {}
    for sdt in (torch.float32, torch.bfloat16):
        pool, prm = _setup(kda, H, 8, seed=102, sdt=sdt)
        y = _call(kda, pool, prm, tok, 0, [T], [0], [-1], [1], interval, cks)
        res[sdt] = (y, pool.S[1].clone(), [pool.S[s].clone() for s in cks], pool.conv[1].clone())
    y32, S32, ck32, c32 = res[torch.float32]
    y16, S16, ck16, c16 = res[torch.bfloat16]
    np.testing.assert_array_equal(_bits(y32), _bits(y16))
    np.testing.assert_array_equal(_bits(S32.to(torch.bfloat16)), _bits(S16))
    for a, b in zip(ck32, ck16):
        np.testing.assert_array_equal(_bits(a.to(torch.bfloat16)), _bits(b))
    np.testing.assert_array_equal(_bits(c32), _bits(c16))


def test_segmented_call_under_graph_capture():
    """The side stream forks from the capturing stream and joins it again, so a segmented call captured in a
    CUDA graph replays to the same bits as the eager call."""
    kda = _kda()
    H, interval, T = 32, 8192, 36000
    assert H * 4 <= _sms() and T // CH >= 512
    pool, prm = _setup(kda, H, 16, seed=111)
    tok = _tokens(112, T, H)
    cks_e, cks_g = [2, 3, 4, 5], [7, 8, 9, 10]
    y_e = _call(kda, pool, prm, tok, 0, [T], [0], [-1], [1], interval, cks_e)  # eager; also the warm-up
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    cu, sp, src, dst = i32([0, T]), torch.zeros(1, dtype=torch.int64, device="cuda"), i32([-1]), i32([6])
    offs, cks = i32([0, len(cks_g)]), i32(cks_g)
    y_g = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, 1, T, CH), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.kda_prefill_chunked(pool, prm, cu, sp, src, dst, CH, interval, offs, cks, tok["q"], tok["k"], tok["v"],
                                tok["a"], tok["b"], tok["z"], y_g, ws, st)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert _same(y_g, y_e)
    assert _same(pool.S[6], pool.S[1]) and _same(pool.conv[6], pool.conv[1])
    for a, b in zip(cks_e, cks_g):
        assert _same(pool.S[a], pool.S[b]) and _same(pool.conv[a], pool.conv[b])


def test_segmented_single_head_bf16_resume_noalloc_against_oracle():
    """33 000 tokens of one head: 518 chunks, so the call is segmented, and a workspace of about 55 MB, within
    the no-alloc scratch.  bf16 pool, resumed from a stored state at position 77 (a partial first chunk), no
    output gate, checkpoints every 4096 tokens with one skipped; outputs, final state, every checkpoint and
    every conv window against the fp64 oracle."""
    from tests.test_prefill_gpu import Problem
    kda = _kda()
    H, T = 1, 33000
    assert H * 4 <= _sms() and T // CH >= 512
    p = Problem(kda, H, D, D, [T], [77], [3], [5], CH, 4096, 24, seed=121, with_z=False, ckpt_skip=(2,), sbf16=True)
    assert kda.kda_prefill_workspace_bytes(p.pool, 1, T, CH) <= kda.NOALLOC_SCRATCH_BYTES
    d = {k: (to_dev_bf16(v) if v is not None else None) for k, v in p.tok.items()}
    p.y = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device="cuda")  # noqa: E731
    kda.kda_prefill_chunked_noalloc(p.pool, p.prm, t(p.cu, torch.int32), t(p.starts, torch.int64),
                                    t(p.src, torch.int32), t(p.dst, torch.int32), CH, p.interval,
                                    t(p.offs, torch.int32), t(p.ck, torch.int32), d["q"], d["k"], d["v"], d["a"],
                                    d["b"], d["z"], p.y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert len(p.ck) == 8 and p.ck[2] == -1
    p.check(p.reference())
