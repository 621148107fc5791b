"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, rejects bad arguments on the host before any launch, and its
host-side causal tile planner reproduces the pages' tile-count fixtures."""
import ctypes
import os
import re

import pytest
import torch

from exact_tiled_attention_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load_library()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.append(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("attn_fwd", "attn_decode_splitkv", "attn_decode_workspace_bytes"):
        assert required in names
    assert set(binding.EXPORTS) <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libgbattn.so does not export {name}"
    assert lib.gbattn_version().decode().startswith("gbattn")


def test_error_strings(lib):
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10]:
        assert lib.gbattn_error_string(code)
    assert lib.gbattn_error_string(12345) == b"unknown status code"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation rejects first


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=4, Hkv=2, Sq=8, Sk=8, d=64, scale=0.125,
             causal=0, dtype=1, stream=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["Sq"],
                        a["Sk"], a["d"], a["scale"], a["causal"], a["dtype"], a["stream"])


def test_attn_fwd_validation(lib):
    assert _fwd(lib, B=0) == -1
    assert _fwd(lib, Sq=0) == -1
    assert _fwd(lib, Sk=-3) == -1
    assert _fwd(lib, H=4, Hkv=3) == -2
    assert _fwd(lib, d=96) == -3
    assert _fwd(lib, d=256) == -3
    assert _fwd(lib, dtype=7) == -4
    assert _fwd(lib, q=None) == -5
    assert _fwd(lib, o=FAKE + 8) == -5
    assert _fwd(lib, lse=FAKE + 2) == -5


def _fwd_pair(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=4, Hkv=2, Sq=8, Sk=8, d=128, scale=0.125,
             dtype=1, stream=None)
    a.update(kw)
    return lib.attn_fwd_pair(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["Sq"],
                             a["Sk"], a["d"], a["scale"], a["dtype"], a["stream"])


def test_attn_fwd_pair_validation(lib):
    assert _fwd_pair(lib, B=0) == -1
    assert _fwd_pair(lib, Sk=0) == -1
    assert _fwd_pair(lib, H=6, Hkv=4) == -2
    assert _fwd_pair(lib, d=64) == -3  # the CTA-pair path is d = 128 only
    assert _fwd_pair(lib, d=96) == -3
    assert _fwd_pair(lib, dtype=2) == -4
    assert _fwd_pair(lib, v=None) == -5
    assert _fwd_pair(lib, k=FAKE + 4) == -5
    if not torch.cuda.is_available():
        assert _fwd_pair(lib) == -10


def _dec(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, Skm=64, d=128,
             scale=0.1, n=4, ws=FAKE, wsb=1 << 20, dtype=1, stream=None)
    a.update(kw)
    return lib.attn_decode_splitkv(a["q"], a["k"], a["v"], a["sl"], a["o"], a["lse"], a["B"], a["Hq"],
                                   a["Hkv"], a["Skm"], a["d"], a["scale"], a["n"], a["ws"], a["wsb"],
                                   a["dtype"], a["stream"])


def test_decode_validation(lib):
    assert lib.attn_decode_workspace_bytes(64, 32, 16, 128) == 64 * 32 * 16 * 130 * 4
    assert lib.attn_decode_workspace_bytes(0, 32, 16, 128) == 0
    assert _dec(lib, B=0) == -1
    assert _dec(lib, Hq=6, Hkv=4) == -2
    assert _dec(lib, d=80) == -3
    assert _dec(lib, dtype=3) == -4
    assert _dec(lib, sl=None) == -5
    assert _dec(lib, ws=None) == -5
    assert _dec(lib, n=0) == -9
    assert _dec(lib, n=257) == -9
    need = lib.attn_decode_workspace_bytes(2, 8, 4, 128)
    assert _dec(lib, wsb=need - 1) == -6


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_call_without_gpu_is_refused(lib):
    assert _fwd(lib) == -10
    assert lib.gbattn_selftest_bounded_wait(0, None) == -10


def test_causal_tile_planner_matches_page_fixtures(lib, golden):
    for case in golden("causal_tile_counts.json")["cases"]:
        got = binding.gbattn_causal_tile_counts(case["Sq"], case["Sk"], case["Br"], case["Bc"])
        assert (got["full"], got["partial"], got["skipped"]) == (case["full"], case["partial"],
                                                                 case["skipped"])
        if "allowed_cells" in case:
            assert got["allowed_cells"] == case["allowed_cells"]
        if "visited_cells" in case:
            assert got["visited_cells"] == case["visited_cells"]
        if "visited_tiles" in case:
            assert got["full"] + got["partial"] == case["visited_tiles"]


def test_causal_planner_bottom_right_rectangles(lib):
    # Sq > Sk: early rows see nothing; allowed cells follow k <= q + (Sk - Sq).
    got = binding.gbattn_causal_tile_counts(5, 2, 1, 1)
    assert got["allowed_cells"] == 3  # rows 3 and 4 see 1 and 2 keys
    got = binding.gbattn_causal_tile_counts(2, 5, 1, 1)
    assert got["allowed_cells"] == 9
    # the 8192-token causal prefill with 128 x 128 tiles visits 2,080 of 4,096 tiles
    got = binding.gbattn_causal_tile_counts(8192, 8192, 128, 128)
    assert got["full"] + got["partial"] == 2080 and got["partial"] == 64


def _bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=4,
             Hkv=2, Sq=8, Sk=8, d=128, scale=0.1, causal=1, ws=FAKE, wsb=1 << 20, dtype=1, stream=None)
    a.update(kw)
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                        a["B"], a["H"], a["Hkv"], a["Sq"], a["Sk"], a["d"], a["scale"], a["causal"],
                        a["ws"], a["wsb"], a["dtype"], a["stream"])


def test_bwd_workspace_matches_page_ledger(lib, golden):
    """The backward workspace is the fp32 row scalars D alone: at the ledger
    coordinate of M4.4 0x06.1J that is the ledger's 0.5 MiB D entry (the
    ledger's dQaccum and expanded dK/dV have no counterpart here)."""
    g = golden("bwd_scratch_ledger.json")
    c = g["coordinate"]
    mib = 1 << 20
    want = g["objects_mib"]["D"] * mib
    assert lib.attn_bwd_workspace_bytes(c["B"], c["Hq"], c["Sq"], c["d"]) == want
    assert lib.attn_bwd_workspace_bytes(0, 1, 1, 128) == 0


def test_bwd_validation(lib):
    assert _bwd(lib, B=0) == -1
    assert _bwd(lib, Sk=0) == -1
    assert _bwd(lib, H=6, Hkv=4) == -2
    assert _bwd(lib, d=96) == -3
    assert _bwd(lib, dtype=2) == -4
    for name in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv", "ws"):
        assert _bwd(lib, **{name: None}) == -5, name
    assert _bwd(lib, dq=FAKE + 8) == -5
    assert _bwd(lib, lse=FAKE + 2) == -5
    need = lib.attn_bwd_workspace_bytes(1, 4, 8, 128)
    assert _bwd(lib, wsb=need - 1) == -6


def _bwd_atomic(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=4,
             Hkv=2, Sq=8, Sk=8, d=128, scale=0.1, causal=1, ws=FAKE, wsb=1 << 20, dtype=1, stream=None)
    a.update(kw)
    return lib.attn_bwd_atomic(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                               a["B"], a["H"], a["Hkv"], a["Sq"], a["Sk"], a["d"], a["scale"], a["causal"],
                               a["ws"], a["wsb"], a["dtype"], a["stream"])


def test_bwd_atomic_workspace_matches_page_ledger(lib, golden):
    """The atomic backward's workspace is the ledger's D plus its fp32
    dQaccum (M4.4 0x06.1J): 64.5 MiB at the ledger coordinate; no expanded
    dK/dV (the grouped sum happens in the key-tile owner's accumulators)."""
    g = golden("bwd_scratch_ledger.json")
    c = g["coordinate"]
    mib = 1 << 20
    want = (g["objects_mib"]["D"] + g["objects_mib"]["dQaccum"]) * mib
    assert lib.attn_bwd_atomic_workspace_bytes(c["B"], c["Hq"], c["Sq"], c["d"]) == want
    assert lib.attn_bwd_atomic_workspace_bytes(0, 1, 1, 128) == 0


def test_bwd_atomic_validation(lib):
    assert _bwd_atomic(lib, B=0) == -1
    assert _bwd_atomic(lib, Sk=0) == -1
    assert _bwd_atomic(lib, H=6, Hkv=4) == -2
    assert _bwd_atomic(lib, d=96) == -3
    assert _bwd_atomic(lib, d=32) == -3
    assert _bwd_atomic(lib, dtype=2) == -4
    for name in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv", "ws"):
        assert _bwd_atomic(lib, **{name: None}) == -5, name
    assert _bwd_atomic(lib, dq=FAKE + 8) == -5
    assert _bwd_atomic(lib, lse=FAKE + 2) == -5
    need = lib.attn_bwd_atomic_workspace_bytes(1, 4, 8, 128)
    assert need == 256 + 4 * 8 * 128 * 4
    assert _bwd_atomic(lib, wsb=need - 1) == -6


def _dec_noalloc(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, Skm=64, d=128,
             scale=0.1, n=4, dtype=1, stream=None)
    a.update(kw)
    return lib.attn_decode_splitkv_noalloc(a["q"], a["k"], a["v"], a["sl"], a["o"], a["lse"], a["B"],
                                           a["Hq"], a["Hkv"], a["Skm"], a["d"], a["scale"], a["n"],
                                           a["dtype"], a["stream"])


def test_decode_noalloc_validation_precedes_capacity(lib):
    """The no-allocation decode reports each bad argument with the code
    attn_decode_splitkv gives it, even where the (bogus) problem would also
    overflow the fixed scratch array; only a valid problem too large for the
    array gets GBATTN_EWORKSPACE."""
    cap = lib.attn_decode_noalloc_scratch_bytes()
    assert cap == 32 << 20
    assert _dec_noalloc(lib, n=0) == -9
    assert _dec_noalloc(lib, n=300) == -9
    assert _dec_noalloc(lib, n=300, B=4096, Hq=64, Hkv=8) == -9     # would need far more than 32 MiB
    assert _dec_noalloc(lib, d=96) == -3
    assert _dec_noalloc(lib, d=96, B=4096, Hq=64, Hkv=8) == -3
    assert _dec_noalloc(lib, dtype=5) == -4
    assert _dec_noalloc(lib, dtype=5, B=4096, Hq=64, Hkv=8) == -4
    assert _dec_noalloc(lib, sl=None) == -5
    assert _dec_noalloc(lib, sl=FAKE + 2) == -5
    assert _dec_noalloc(lib, o=FAKE + 8) == -5
    assert _dec_noalloc(lib, B=0) == -1
    assert _dec_noalloc(lib, Hq=6, Hkv=4) == -2
    # valid arguments, but the partial states need more than the array holds
    B, Hq, n, d = 4096, 64, 16, 128
    assert lib.attn_decode_workspace_bytes(B, Hq, n, d) > cap
    assert _dec_noalloc(lib, B=B, Hq=Hq, Hkv=8, n=n, d=d) == -6


@pytest.mark.parametrize("wrapper", ["attn_decode_splitkv", "attn_decode_splitkv_noalloc"])
def test_decode_wrappers_reject_mismatched_tensors(wrapper):
    """Both Python decode wrappers check every shape, dtype and length
    agreement before any pointer reaches the library (a smaller v_cache or a
    short seqlens would otherwise make the kernels read out of bounds)."""
    fn = getattr(binding, wrapper)
    B, Hq, Hkv, S, d = 2, 8, 2, 64, 128
    bf = torch.bfloat16
    q = torch.zeros(B, Hq, 1, d, dtype=bf)
    k = torch.zeros(B, Hkv, S, d, dtype=bf)
    sl = torch.full((B,), S, dtype=torch.int32)
    cases = [
        (ValueError, dict(q=torch.zeros(B, Hq, 2, d, dtype=bf))),                 # two queries per sequence
        (ValueError, dict(v=torch.zeros(B, Hkv, S // 2, d, dtype=bf))),           # shorter v_cache
        (ValueError, dict(k=torch.zeros(B + 1, Hkv, S, d, dtype=bf),
                          v=torch.zeros(B + 1, Hkv, S, d, dtype=bf))),            # cache batch differs
        (ValueError, dict(k=torch.zeros(B, Hkv, S, 64, dtype=bf),
                          v=torch.zeros(B, Hkv, S, 64, dtype=bf))),               # head dim differs
        (ValueError, dict(sl=torch.full((B - 1,), S, dtype=torch.int32))),         # short seqlens
        (TypeError, dict(sl=torch.full((B,), S, dtype=torch.int64))),              # int64 lengths
        (TypeError, dict(v=torch.zeros(B, Hkv, S, d, dtype=torch.float16))),       # dtypes differ
        (TypeError, dict(q=torch.zeros(B, Hq, 1, d, dtype=torch.float32),
                         k=torch.zeros(B, Hkv, S, d, dtype=torch.float32),
                         v=torch.zeros(B, Hkv, S, d, dtype=torch.float32))),       # unsupported dtype
        (ValueError, dict(out=torch.zeros(B, Hq, 1, 64, dtype=bf))),               # wrong out shape
        (ValueError, dict(lse=torch.zeros(B, Hq + 1, dtype=torch.float32))),       # wrong lse shape
        (ValueError, dict()),                                                      # consistent, but not CUDA
    ]
    for exc, over in cases:
        a = dict(q=q, k=k, v=k.clone(), sl=sl, out=None, lse=None)
        a.update(over)
        with pytest.raises(exc):
            fn(a["q"], a["k"], a["v"], a["sl"], out=a["out"], lse=a["lse"])


def test_timeline_set_validation(lib):
    """gbattn_timeline_set checks alignment and capacity on the host, and
    NULL turns the timeline off whatever the capacity."""
    try:
        assert lib.gbattn_timeline_set(FAKE + 4, 16) == -5     # not 8-byte aligned
        assert lib.gbattn_timeline_set(FAKE, 0) == -1
        assert lib.gbattn_timeline_set(FAKE, -3) == -1
        assert lib.gbattn_timeline_set(None, -3) == 0
        assert lib.gbattn_timeline_set(FAKE, 8) == 0
    finally:
        assert lib.gbattn_timeline_set(None, 0) == 0


def test_timeline_wrapper_rejects_bad_buffers():
    with pytest.raises(ValueError):
        binding.gbattn_timeline_set(torch.zeros(8, 4, dtype=torch.int64))           # not CUDA
    binding.gbattn_timeline_set(None)
