"""The C-ABI library builds for sm_103a, loads, and exports every entry point include/kda.h declares;
host-side argument checks work without a GPU (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from hybrid_linear_attention_decode_gb300 import build as kbuild
    import hybrid_linear_attention_decode_gb300 as kda
    kbuild.build()
    return kda.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src)


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("kda_decode_step", "kda_prefill_chunked", "kda_resume_from_slot"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    import hybrid_linear_attention_decode_gb300 as kda
    assert lib.kda_version() >= 1
    assert kda.kda_status_string(0) == "ok"
    for rc in range(1, 5):
        assert kda.kda_status_string(rc) != "unknown status"


def test_checkpoint_count_matches_the_oracle(lib):
    import oracle
    import hybrid_linear_attention_decode_gb300 as kda
    for start in (0, 1, 31, 32, 127, 128, 32768):
        for length in (0, 1, 31, 32, 33, 1024):
            for interval in (0, 16, 32, 128, 32768):
                exp = oracle.ckpt_count(start, length, interval) if interval > 0 else 0
                assert kda.kda_checkpoint_count(start, length, interval) == exp
    assert kda.kda_checkpoint_count(-1, 4, 2) == -1


def test_host_validation_without_gpu(lib):
    import hybrid_linear_attention_decode_gb300 as kda
    # NULL pool / params: rejected before any CUDA call
    assert lib.kda_decode_step(None, None, 1, *([None] * 11)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_resume_from_slot(None, 1, None, None, None, None) == kda.KDA_ERR_INVALID_ARG
    pool = kda._Pool(2, 128, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    # unsupported shape / misaligned pointers are host errors
    bad = kda._Pool(2, 96, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    prm = kda._Params(ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000), 1e-6, 1e-6, 1.0, 1)
    assert lib.kda_decode_step(ctypes.byref(bad), ctypes.byref(prm), 1, *([None] * 11)) == \
        kda.KDA_ERR_UNSUPPORTED_SHAPE
    mis = kda._Pool(2, 128, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1004), ctypes.c_void_p(0x2000))
    assert lib.kda_decode_step(ctypes.byref(mis), ctypes.byref(prm), 1, *([None] * 11)) == kda.KDA_ERR_INVALID_ARG
    # an unknown state dtype is an invalid argument
    odd = kda._Pool(2, 128, 128, 4, 7, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    assert lib.kda_decode_step(ctypes.byref(odd), ctypes.byref(prm), 1, *([None] * 11)) == kda.KDA_ERR_INVALID_ARG
    # n = 0 is a no-op that returns OK without touching the device
    assert lib.kda_decode_step(ctypes.byref(pool), ctypes.byref(prm), 0, *([None] * 11)) == kda.KDA_OK
    assert lib.kda_resume_from_slot(ctypes.byref(pool), 0, None, None, None, None) == kda.KDA_OK


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "hybrid_linear_attention_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower() or f.endswith(".md"), f


def test_binding_argument_counts_match_header(lib):
    """The ctypes signatures declare exactly the parameters include/kda.h gives each entry point."""
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    for name in declared_functions():
        m = re.search(r"KDA_API[^;(]*\b" + name + r"\s*\(([^)]*)\)", src)
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        argtypes = getattr(lib, name).argtypes or []
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))


def test_noalloc_scratch_size_matches_header():
    import hybrid_linear_attention_decode_gb300 as kda
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    m = re.search(r"#define KDA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    assert m and int(m.group(1)) << int(m.group(2)) == kda.NOALLOC_SCRATCH_BYTES


def test_last_error_names_the_rejected_argument(lib):
    import hybrid_linear_attention_decode_gb300 as kda
    prm = kda._Params(ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000), 1e-6, 1e-6, 1.0, 1)
    mis = kda._Pool(2, 128, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1004), ctypes.c_void_p(0x2000))
    assert lib.kda_decode_step(ctypes.byref(mis), ctypes.byref(prm), 1, *([None] * 11)) == kda.KDA_ERR_INVALID_ARG
    assert "16-byte aligned" in kda.kda_last_error_string()
    bad = kda._Pool(2, 96, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    assert lib.kda_decode_step(ctypes.byref(bad), ctypes.byref(prm), 1, *([None] * 11)) == \
        kda.KDA_ERR_UNSUPPORTED_SHAPE
    assert "not compiled in" in kda.kda_last_error_string()
    pool = kda._Pool(2, 128, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    assert lib.kda_resume_from_slot(ctypes.byref(pool), 0, None, None, None, None) == kda.KDA_OK
    assert kda.kda_last_error_string() == ""  # a successful call clears it
    # the interval must be a multiple of the chunk
    rc = lib.kda_prefill_chunked(ctypes.byref(pool), ctypes.byref(prm), 1, 0, *([None] * 4), 64, 96,
                                 *([None] * 9), None, 0, None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG and "multiple of the chunk" in kda.kda_last_error_string()
    with pytest.raises(kda.KdaError) as e:
        kda._check(rc, "kda_prefill_chunked")
    assert "multiple of the chunk" in str(e.value)


def test_check_slots_enforces_the_aliasing_contract(lib):
    import hybrid_linear_attention_decode_gb300 as kda
    ok = kda.kda_check_slots
    ok(8, [0, 1, 2], [0, 1, 2])                 # in place
    ok(8, [-1, -1], [3, 4])                     # fresh requests
    ok(8, [0, 1], [5, 6], [7, -1, 2])           # prefill with checkpoints; -1 skips
    ok(8, [], [])
    cases = [
        ((8, [0, 1], [2, 2]), "written twice"),            # duplicate dst
        ((8, [0, 1], [1, 2]), "written by another"),       # src of item 1 is the dst of item 0
        ((8, [0], [1], [0]), "written by another"),        # src is a checkpoint slot
        ((8, [0], [0], [0]), "written twice"),             # in place, but also a checkpoint
        ((8, [0], [1], [1]), "written twice"),             # checkpoint equals a dst
        ((8, [0], [8]), "outside"),
        ((8, [-2], [1]), "outside"),
        ((8, [0], [1], [9]), "outside"),
    ]
    for args, words in cases:
        with pytest.raises(kda.KdaError) as e:
            ok(*args)
        assert e.value.rc == kda.KDA_ERR_INVALID_ARG and words in str(e.value), (args, str(e.value))


def test_noalloc_checks_arguments_then_size_before_any_device_call(lib):
    """The no-allocation entry point's documented order: argument checks (no CUDA call), then the size check
    against its static scratch (no CUDA call), and only then the device look-up.  On a machine without a GPU
    the first two still answer."""
    import hybrid_linear_attention_decode_gb300 as kda
    prm = kda._Params(ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000), 1e-6, 1e-6, 1.0, 1)
    pool = kda._Pool(2, 128, 128, 4, 0, 0, 8, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))
    p16 = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(16)]  # aligned stand-ins, never dereferenced
    # a NULL pool is an invalid argument
    rc = lib.kda_prefill_chunked_noalloc(None, ctypes.byref(prm), 1, 64, *p16[:4], 64, 0, None, None,
                                         *p16[4:11], None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    # an interval that is not a multiple of the chunk is an invalid argument
    rc = lib.kda_prefill_chunked_noalloc(ctypes.byref(pool), ctypes.byref(prm), 1, 64, *p16[:4], 64, 96,
                                         p16[4], p16[5], *p16[6:13], None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG and "multiple of the chunk" in kda.kda_last_error_string()
    # a problem whose workspace exceeds the static scratch is refused without a launch
    tokens = 1 << 20
    assert lib.kda_prefill_workspace_bytes(ctypes.byref(pool), 1, tokens, 64) > kda.NOALLOC_SCRATCH_BYTES
    rc = lib.kda_prefill_chunked_noalloc(ctypes.byref(pool), ctypes.byref(prm), 1, tokens, *p16[:4], 64, 0, None,
                                         None, *p16[4:11], None, None)
    assert rc == kda.KDA_ERR_WORKSPACE and "static scratch" in kda.kda_last_error_string()
