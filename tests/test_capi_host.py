"""Host-side checks of the C ABI: the library loads, exports every function
the header declares, and rejects bad arguments before touching CUDA.
No case here reaches a kernel launch, so none needs a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rms_norm.h")


@pytest.fixture(scope="module")
def lib():
    import bwd_rms_norm_gb300 as L
    from bwd_rms_norm_gb300 import build
    if not os.path.exists(L.LIB_PATH):
        build.build()
    return L.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:rms_norm|layer_norm|softmax|group_norm)_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("rms_norm_fwd", "rms_norm_bwd", "rms_norm_bwd_workspace_size",
              "rms_norm_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_declares_every_export():
    import bwd_rms_norm_gb300 as L
    assert sorted(L.EXPORTED) == declared_functions()


def test_header_constants_match_binding():
    import bwd_rms_norm_gb300 as L
    text = open(HEADER).read()
    consts = dict(re.findall(r"(RMSN_\w+)\s*=\s*(\d+)", text))
    consts.update(dict(re.findall(r"#define\s+(RMSN_\w+)\s+(\d+)", text)))
    for name in ("RMSN_F32", "RMSN_BF16", "RMSN_F16", "RMSN_ROUND_ONCE", "RMSN_ROUND_TWICE",
                 "RMSN_OK", "RMSN_MAX_HIDDEN", "RMSN_MAX_PARTIALS", "RMSN_DW_CHUNK_BLOCKS"):
        assert int(consts[name]) == getattr(L, name), name


NULL = None
FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: every case fails validation first


def fwd(lib, x=FAKE, g=FAKE, y=FAKE, r=FAKE, rows=4, hidden=64, eps=1e-5, offset=0,
        dtype=1, mode=0):
    return lib.rms_norm_fwd(x, g, y, r, rows, hidden, eps, offset, dtype, mode, None)


def test_fwd_validation(lib):
    assert fwd(lib, dtype=3) == 4
    assert fwd(lib, dtype=-1) == 4
    assert fwd(lib, offset=2) == 8
    assert fwd(lib, mode=2) == 8
    assert fwd(lib, rows=-1) == 2
    assert fwd(lib, hidden=0) == 2
    assert fwd(lib, hidden=65537) == 2
    assert fwd(lib, rows=1 << 31) == 2
    assert fwd(lib, eps=-1e-6) == 3
    assert fwd(lib, eps=float("nan")) == 3
    assert fwd(lib, eps=float("inf")) == 3
    assert fwd(lib, x=NULL) == 1
    assert fwd(lib, g=NULL) == 1
    assert fwd(lib, y=NULL) == 1
    assert fwd(lib, r=NULL) == 1
    # zero rows: nothing to do, no pointer needed, nothing launched
    assert fwd(lib, x=NULL, y=NULL, r=NULL, g=NULL, rows=0) == 0
    assert lib.rms_norm_last_launch_count() == 0


def bwd(lib, dy=FAKE, x=FAKE, g=FAKE, r=FAKE, dx=FAKE, dw=FAKE, rows=4, hidden=64, offset=0,
        dtype=1, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.rms_norm_bwd_workspace_size(rows, hidden, dtype)
    return lib.rms_norm_bwd(dy, x, g, r, dx, dw, rows, hidden, offset, dtype, ws, ws_bytes, None)


def test_bwd_validation(lib):
    assert bwd(lib, dtype=7) == 4
    assert bwd(lib, offset=-1) == 8
    assert bwd(lib, rows=-2) == 2
    assert bwd(lib, hidden=70000) == 2
    assert bwd(lib, dw=NULL) == 1
    for k in ("dy", "x", "g", "r", "dx", "ws"):
        assert bwd(lib, **{k: NULL}) == 1, k
    assert bwd(lib, ws=ctypes.c_void_p(0x1004)) == 5
    assert bwd(lib, ws_bytes=lib.rms_norm_bwd_workspace_size(4, 64, 1) - 4) == 6


def test_workspace_size(lib):
    assert lib.rms_norm_bwd_workspace_size(0, 64, 1) == 0
    assert lib.rms_norm_bwd_workspace_size(10, 64, 1) == 10 * 64 * 4
    assert lib.rms_norm_bwd_workspace_size(5000, 4096, 1) == 1024 * 4096 * 4
    assert lib.rms_norm_bwd_workspace_size(5, 0, 1) == 0
    assert lib.rms_norm_bwd_workspace_size(5, 64, 9) == 0


def test_status_strings(lib):
    for s in range(9):
        assert lib.rms_norm_status_string(s).decode()
    assert lib.rms_norm_status_string(99).decode() == "unknown status"


def test_binding_refuses_cpu_tensors():
    """The Python layer has no CPU path: CPU tensors are an error."""
    import torch
    import bwd_rms_norm_gb300 as L
    x = torch.zeros(2, 8)
    with pytest.raises(RuntimeError, match="CUDA"):
        L.rms_norm_fwd(x, torch.ones(8), 1e-5)


def test_layer_norm_validation(lib):
    f = lambda **k: lib.layer_norm_fwd(k.get("x", FAKE), k.get("g", FAKE), k.get("b", NULL),
                                       k.get("y", FAKE), k.get("m", FAKE), k.get("r", FAKE),
                                       k.get("rows", 4), k.get("hidden", 64), k.get("eps", 1e-5),
                                       k.get("dtype", 1), None)
    assert f(dtype=5) == 4
    assert f(hidden=0) == 2
    assert f(eps=-1.0) == 3
    for k in ("x", "g", "y", "m", "r"):
        assert f(**{k: NULL}) == 1, k
    assert f(rows=0, x=NULL, g=NULL, y=NULL, m=NULL, r=NULL) == 0
    assert lib.layer_norm_bwd_workspace_size(10, 64, 1) == 2 * 10 * 64 * 4

    def b(**k):
        ws_bytes = k.get("ws_bytes", lib.layer_norm_bwd_workspace_size(4, 64, 1))
        return lib.layer_norm_bwd(k.get("dy", FAKE), k.get("x", FAKE), k.get("g", FAKE),
                                  k.get("m", FAKE), k.get("r", FAKE), k.get("dx", FAKE),
                                  k.get("dg", FAKE), k.get("db", NULL), 4, 64, k.get("dtype", 1),
                                  k.get("ws", FAKE), ws_bytes, None)
    assert b(dtype=9) == 4
    assert b(dg=NULL) == 1
    for k in ("dy", "x", "g", "m", "r", "dx", "ws"):
        assert b(**{k: NULL}) == 1, k
    assert b(ws=ctypes.c_void_p(0x1008)) == 5
    assert b(ws_bytes=16) == 6


def test_fp8_forward_validation(lib):
    """Host-side checks of rms_norm_fwd_fp8 (no kernel runs: every case is
    rejected before a launch, or has rows == 0)."""
    def f(**k):
        return lib.rms_norm_fwd_fp8(k.get("x", FAKE), k.get("g", FAKE), k.get("s", FAKE),
                                    k.get("y", FAKE), k.get("r", FAKE), k.get("rows", 4),
                                    k.get("hidden", 64), k.get("eps", 1e-5), k.get("offset", 0),
                                    k.get("dtype", 1), None)
    assert f(dtype=3) == 4
    assert f(offset=2) == 8
    assert f(hidden=0) == 2 and f(hidden=65537) == 2 and f(rows=-1) == 2
    assert f(eps=float("nan")) == 3 and f(eps=float("inf")) == 3
    for k in ("x", "g", "s", "y", "r"):
        assert f(**{k: NULL}) == 1, k
    assert f(rows=0, x=NULL, g=NULL, s=NULL, y=NULL, r=NULL) == 0


def test_softmax_validation(lib):
    """Host-side checks of softmax_fwd / softmax_bwd (every case rejected
    before a launch, or rows == 0)."""
    f = lambda **k: lib.softmax_fwd(k.get("x", FAKE), k.get("y", FAKE), k.get("rows", 4),
                                    k.get("cols", 64), k.get("dtype", 1), None)
    assert f(dtype=7) == 4
    assert f(cols=0) == 2 and f(cols=65537) == 2 and f(rows=-2) == 2
    assert f(x=NULL) == 1 and f(y=NULL) == 1
    assert f(rows=0, x=NULL, y=NULL) == 0
    b = lambda **k: lib.softmax_bwd(k.get("dy", FAKE), k.get("y", FAKE), k.get("dx", FAKE),
                                    k.get("rows", 4), k.get("cols", 64), k.get("dtype", 1), None)
    assert b(dtype=-1) == 4
    assert b(cols=0) == 2
    for k in ("dy", "y", "dx"):
        assert b(**{k: NULL}) == 1, k
    assert b(rows=0, dy=NULL, y=NULL, dx=NULL) == 0


def test_group_norm_validation(lib):
    """Host-side checks of the GroupNorm entry points (every case rejected
    before a launch, or n == 0)."""
    def f(**k):
        return lib.group_norm_fwd(k.get("x", FAKE), k.get("g", FAKE), k.get("b", NULL),
                                  k.get("y", FAKE), k.get("m", FAKE), k.get("r", FAKE),
                                  k.get("n", 2), k.get("c", 8), k.get("s", 64), k.get("G", 4),
                                  k.get("eps", 1e-5), k.get("dtype", 1), None)
    assert f(dtype=3) == 4
    assert f(c=6, G=4) == 2          # channels not a multiple of groups
    assert f(G=0) == 2 and f(s=0) == 2 and f(c=0) == 2 and f(n=-1) == 2
    assert f(c=2, G=2, s=(1 << 30) + 8) == 2
    assert f(eps=-1.0) == 3
    for k in ("x", "g", "y", "m", "r"):
        assert f(**{k: NULL}) == 1, k
    assert f(n=0, x=NULL, g=NULL, y=NULL, m=NULL, r=NULL) == 0
    assert lib.group_norm_bwd_workspace_size(2, 8, 64, 4, 1) == 2 * 16 * 2 * 8 * 4
    assert lib.group_norm_bwd_workspace_size(2, 8, 64, 3, 1) == 0

    def b(**k):
        ws_bytes = k.get("ws_bytes", lib.group_norm_bwd_workspace_size(2, 8, 64, 4, 1))
        return lib.group_norm_bwd(k.get("dy", FAKE), k.get("x", FAKE), k.get("g", FAKE),
                                  k.get("m", FAKE), k.get("r", FAKE), k.get("dx", FAKE),
                                  k.get("dg", FAKE), k.get("db", NULL), 2, 8, 64, 4,
                                  k.get("dtype", 1), k.get("ws", FAKE), ws_bytes, None)
    assert b(dtype=9) == 4
    assert b(dg=NULL) == 1
    for k in ("dy", "x", "g", "m", "r", "dx", "ws"):
        assert b(**{k: NULL}) == 1, k
    assert b(ws=ctypes.c_void_p(0x1004)) == 5
    assert b(ws_bytes=64) == 6


def test_last_kernels_without_launches(lib):
    """Before any launch on this thread, or after a call rejected on the
    host, no kernel is reported (no GPU involved)."""
    names = (ctypes.c_char_p * 4)()
    assert fwd(lib, dtype=3) == 4
    assert lib.rms_norm_last_kernels(names, 4) == 0
    assert lib.rms_norm_last_kernels(None, 4) < 0


def test_selftest_rejects_null_pointers(lib):
    n, t = ctypes.c_uint(0), ctypes.c_double(0.0)
    assert lib.rms_norm_selftest_wait_limit(None, ctypes.byref(t)) == 1   # RMSN_ERR_NULL
    assert lib.rms_norm_selftest_wait_limit(ctypes.byref(n), None) == 1


def test_rms_norm_module_host_side():
    """The autograd layer builds its weight on the host, checks its
    arguments, and refuses CPU inputs like every other call."""
    import torch
    import bwd_rms_norm_gb300 as L
    m = L.RMSNorm(16, eps=1e-5)
    assert torch.equal(m.weight.detach(), torch.ones(16))
    g = L.RMSNorm(16, offset=1, dtype=torch.bfloat16)
    assert g.weight.dtype == torch.bfloat16 and torch.count_nonzero(g.weight).item() == 0
    with pytest.raises(ValueError):
        L.RMSNorm(16, offset=2)
    with pytest.raises(ValueError):
        L.RMSNorm(16, cast_mode="round_thrice")
    with pytest.raises(RuntimeError, match="CUDA"):
        m(torch.zeros(3, 16, requires_grad=True))


def test_blocked_backward_validation(lib):
    """The fixed-block backward and the chunk total refuse bad arguments
    before any CUDA call."""
    ws = lib.rms_norm_bwd_blocked_workspace_size(100, 64, 8)
    assert ws == 13 * 64 * 4                       # ceil(100 / 8) partial rows
    assert lib.rms_norm_bwd_blocked_workspace_size(100, 64, 0) == 0
    assert lib.rms_norm_dw_chunk_count(100, 8) == 1
    assert lib.rms_norm_dw_chunk_count(32 * 8 + 1, 8) == 2
    assert lib.rms_norm_dw_chunk_count(0, 8) == 0
    assert lib.rms_norm_dw_chunk_count(10, 0) == -2

    def call(rows=100, hidden=64, brows=8, chunks=FAKE, ws_bytes=ws, dtype=1, offset=0):
        return lib.rms_norm_bwd_blocked(FAKE, FAKE, FAKE, FAKE, FAKE, chunks, rows, hidden, brows,
                                        offset, dtype, FAKE, ws_bytes, None)

    assert call(brows=0) == 8                      # RMSN_ERR_ARG
    assert call(rows=-1) == 2                      # RMSN_ERR_SHAPE
    assert call(hidden=0) == 2
    assert call(dtype=7) == 4
    assert call(offset=2) == 8
    assert call(chunks=None) == 1                  # RMSN_ERR_NULL
    assert call(ws_bytes=ws - 4) == 6              # RMSN_ERR_WORKSPACE
    assert call(rows=0) == 0                       # nothing to do
    assert lib.rms_norm_dw_sum(FAKE, -1, 64, FAKE, None) == 2
    assert lib.rms_norm_dw_sum(FAKE, 3, 0, FAKE, None) == 2
    assert lib.rms_norm_dw_sum(FAKE, 3, 64, None, None) == 1
    assert lib.rms_norm_dw_sum(None, 3, 64, FAKE, None) == 1


@pytest.mark.parametrize("rows,brows", [(0, 4), (1, 4), (1000, 4), (16384, 16), (4097, 1),
                                        (12345, 7)])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_rank_rows_are_whole_chunks(lib, rows, brows, world):
    """rms_norm_rank_rows tiles the rows with contiguous slabs whose
    boundaries are whole chunks (32 blocks), as evenly as the chunks allow."""
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    spans = []
    for r in range(world):
        assert lib.rms_norm_rank_rows(rows, brows, world, r, ctypes.byref(lo),
                                      ctypes.byref(hi)) == 0
        spans.append((lo.value, hi.value))
    assert spans[0][0] == 0 and spans[-1][1] == rows
    chunk = 32 * brows
    for (a, b), (c, _) in zip(spans, spans[1:]):
        assert b == c
        assert b % chunk == 0 or b == rows
    counts = [-(-(b - a) // chunk) for a, b in spans]
    assert max(counts) - min(counts) <= 1
    assert lib.rms_norm_rank_rows(rows, brows, world, world, ctypes.byref(lo),
                                  ctypes.byref(hi)) == 8
    assert lib.rms_norm_rank_rows(rows, 0, world, 0, ctypes.byref(lo), ctypes.byref(hi)) == 8


def test_sm_budget_setting(lib):
    assert lib.rms_norm_sm_budget() == 0
    assert lib.rms_norm_set_sm_budget(-1) == 8
    assert lib.rms_norm_set_sm_budget(100) == 0
    assert lib.rms_norm_sm_budget() == 100
    assert lib.rms_norm_set_sm_budget(0) == 0
    assert lib.rms_norm_sm_budget() == 0
