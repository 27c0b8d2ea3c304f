"""The C ABI library: it loads, exports every symbol include/gdn.h declares, and
rejects bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import math
import os
import re

import pytest

from chunked_gated_delta_gdn_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(gdn_\w+)\s*\(", text, flags=re.M)))


def test_library_loads_and_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and "gdn_decode" in names
    for name in names:
        assert hasattr(lib, name), "libgdn.so does not export %s" % name
    assert set(_lib.EXPORTS) <= set(names)
    assert lib.gdn_version() >= 100


def test_status_strings():
    for code, name in enumerate(["GDN_OK", "GDN_ERR_NULL", "GDN_ERR_SHAPE", "GDN_ERR_DTYPE",
                                 "GDN_ERR_LAYOUT", "GDN_ERR_UNSUPPORTED", "GDN_ERR_CUDA",
                                 "GDN_ERR_WORKSPACE"]):
        assert _lib.status_string(code) == name
    assert _lib.status_string(99) == "GDN_ERR_UNKNOWN"


def test_path_selection_and_workspace_sizes():
    lib = _lib.load()
    assert lib.gdn_chunk_fwd_path(128, 128, _lib.GDN_F32, _lib.GDN_F32) == 0
    assert lib.gdn_chunk_fwd_path(64, 64, _lib.GDN_BF16, _lib.GDN_BF16) == 0
    assert lib.gdn_chunk_fwd_path(256, 128, _lib.GDN_BF16, _lib.GDN_BF16) == -1
    assert lib.gdn_chunk_fwd_path(128, 128, 7, 0) == -1
    tc = lib.gdn_chunk_fwd_path(128, 128, _lib.GDN_BF16, _lib.GDN_BF16)
    assert tc in (0, 1)
    ws = lib.gdn_chunk_fwd_workspace_size(1, 256, 2, 2, 64, 64, 1, _lib.GDN_F32, _lib.GDN_F32)
    nc = 256 // 64 + 1
    assert ws >= 4 * nc * 2 * (64 * 64 + 64 * 64 + 64 + 64 * 64)
    assert lib.gdn_chunk_fwd_workspace_size(1, 256, 2, 3, 64, 64, 1, 0, 0) == (1 << 64) - 1
    if tc == 1:
        # the tensor-core path's launch plan: unit tables of 40-byte entries, 256-byte aligned
        # parts; with 128 chains (more than a third of any GB300's SMs) nothing splits, so there
        # are no segment matrices
        ws = lib.gdn_chunk_fwd_workspace_size(4, 32768, 16, 32, 128, 128, 4, 1, 1)
        assert 128 * 40 <= ws < 128 * 40 + 4 * 256


FAKE = 1 << 20   # never dereferenced: every call below fails validation first


def chunk_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, B=1, T=64, Hqk=1, Hv=1, K=64, V=64,
                io=_lib.GDN_F32, bdt=_lib.GDN_F32, scale=float("nan"), chunk=64, init=None,
                ofs=0, fin=None, l2=1, cu=None, N=1, si=None, slots=0, o=FAKE, ws=None,
                wsb=0, status=None, stream=None)
    args.update(kw)
    return _lib.load().gdn_chunk_fwd(*args.values())


def test_chunk_fwd_rejects_bad_arguments():
    assert chunk_call(chunk=32) == _lib.GDN_ERR_UNSUPPORTED
    assert chunk_call(q=None) == _lib.GDN_ERR_NULL
    assert chunk_call(o=None) == _lib.GDN_ERR_NULL
    assert chunk_call(ofs=1, fin=None) == _lib.GDN_ERR_NULL
    assert chunk_call(Hv=3, Hqk=2) == _lib.GDN_ERR_SHAPE
    assert chunk_call(K=0) == _lib.GDN_ERR_SHAPE
    assert chunk_call(K=130) == _lib.GDN_ERR_SHAPE
    assert chunk_call(K=6) == _lib.GDN_ERR_SHAPE          # 24 bytes: not a multiple of 16
    assert chunk_call(io=5) == _lib.GDN_ERR_DTYPE
    assert chunk_call(io=_lib.GDN_F32, bdt=_lib.GDN_BF16) == _lib.GDN_ERR_DTYPE
    assert chunk_call(cu=FAKE, B=2) == _lib.GDN_ERR_SHAPE
    assert chunk_call(si=FAKE, slots=0) == _lib.GDN_ERR_SHAPE
    assert chunk_call(q=FAKE + 4) == _lib.GDN_ERR_LAYOUT
    assert chunk_call(g=FAKE + 2) == _lib.GDN_ERR_LAYOUT
    assert chunk_call(ws=None, wsb=0) == _lib.GDN_ERR_WORKSPACE   # fp32 path needs scratch
    assert chunk_call(ws=FAKE, wsb=16) == _lib.GDN_ERR_WORKSPACE
    assert chunk_call(B=0) == _lib.GDN_OK                          # nothing to do
    assert chunk_call(cu=FAKE, N=0) == _lib.GDN_OK


def decode_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, slots=8, idx=None, n=4,
                Hqk=1, Hv=1, K=128, V=128, io=_lib.GDN_BF16, bdt=_lib.GDN_BF16,
                scale=float("nan"), l2=1, o=FAKE, status=None, stream=None)
    args.update(kw)
    return _lib.load().gdn_decode(*args.values())


def test_decode_rejects_bad_arguments():
    assert decode_call(state=None) == _lib.GDN_ERR_NULL
    assert decode_call(n=9, idx=None) == _lib.GDN_ERR_SHAPE      # identity needs n <= slots
    assert decode_call(n=-1) == _lib.GDN_ERR_SHAPE
    assert decode_call(Hv=3, Hqk=2) == _lib.GDN_ERR_SHAPE
    assert decode_call(io=3) == _lib.GDN_ERR_DTYPE
    assert decode_call(state=FAKE + 8) == _lib.GDN_ERR_LAYOUT
    assert decode_call(beta=FAKE + 1) == _lib.GDN_ERR_LAYOUT
    assert decode_call(n=0) == _lib.GDN_OK


def test_python_binding_validates_on_cpu_tensors():
    torch = pytest.importorskip("torch")
    from chunked_gated_delta_gdn_gb300 import chunk_gated_delta_rule, gated_delta_decode
    x = torch.zeros(1, 4, 1, 8)
    with pytest.raises(ValueError, match="CUDA"):
        chunk_gated_delta_rule(x, x, x, torch.zeros(1, 4, 1), torch.zeros(1, 4, 1))
    with pytest.raises(ValueError, match="CUDA"):
        gated_delta_decode(x[0], x[0], x[0], torch.zeros(4, 1), torch.zeros(4, 1),
                           torch.zeros(2, 1, 8, 8))


def product_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, B=1, T=64, n_h=2, Hqk=1, Hv=1, K=64,
                V=64, io=_lib.GDN_F32, bdt=_lib.GDN_F32, scale=float("nan"), chunk=64, init=None,
                ofs=0, fin=None, l2=1, cu=None, N=1, si=None, slots=0, o=FAKE, ws=None, wsb=0,
                status=None, stream=None)
    args.update(kw)
    return _lib.load().gdn_product_chunk_fwd(*args.values())


def test_product_entry_points_reject_bad_arguments():
    lib = _lib.load()
    assert product_call(n_h=0) == _lib.GDN_ERR_SHAPE
    assert product_call(chunk=32) == _lib.GDN_ERR_UNSUPPORTED
    assert product_call(q=None) == _lib.GDN_ERR_NULL
    assert product_call(Hv=3, Hqk=2) == _lib.GDN_ERR_SHAPE
    assert product_call(q=FAKE + 4) == _lib.GDN_ERR_LAYOUT
    assert product_call(ws=None, wsb=0) == _lib.GDN_ERR_WORKSPACE
    need = lib.gdn_product_chunk_fwd_workspace_size(1, 64, 2, 1, 1, 64, 64, 1, 0, 0)
    assert need != (1 << 64) - 1
    assert product_call(ws=FAKE, wsb=need - 1) == _lib.GDN_ERR_WORKSPACE
    assert product_call(ws=FAKE + 16, wsb=need) == _lib.GDN_ERR_LAYOUT   # needs 256-byte alignment
    # the workspace holds q', g', o' of the 128 writes plus the chunk kernels' own scratch
    assert need >= 128 * 64 * 4 + 128 * 4 + 128 * 64 * 4 + \
        lib.gdn_chunk_fwd_workspace_size(1, 128, 1, 1, 64, 64, 1, 0, 0)
    assert lib.gdn_product_chunk_fwd_workspace_size(1, 64, 0, 1, 1, 64, 64, 1, 0, 0) == (1 << 64) - 1
    # one write per token is the gated delta rule: same scratch
    assert lib.gdn_product_chunk_fwd_workspace_size(1, 64, 1, 1, 1, 64, 64, 1, 0, 0) == \
        lib.gdn_chunk_fwd_workspace_size(1, 64, 1, 1, 64, 64, 1, 0, 0)
    dec = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, None, 4, 2, 1, 1, 128, 128, _lib.GDN_BF16,
           _lib.GDN_BF16, float("nan"), 1, FAKE, None, None, None]
    bad = list(dec); bad[9] = 0
    assert lib.gdn_product_decode(*bad) == _lib.GDN_ERR_SHAPE
    bad = list(dec); bad[5] = None
    assert lib.gdn_product_decode(*bad) == _lib.GDN_ERR_NULL


def bwd_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, B=1, T=64, Hqk=1, Hv=1, K=64, V=64,
                io=_lib.GDN_F32, bdt=_lib.GDN_F32, scale=float("nan"), chunk=64, init=None, l2=1,
                cu=None, N=1, do=FAKE, dfin=None, dq=FAKE, dk=FAKE, dv=FAKE, dg=FAKE, db=FAKE,
                dinit=None, ws=None, wsb=0, status=None, stream=None)
    args.update(kw)
    return _lib.load().gdn_chunk_bwd(*args.values())


def test_backward_entry_point_rejects_bad_arguments():
    lib = _lib.load()
    need = lib.gdn_chunk_bwd_workspace_size(1, 64, 1, 1, 64, 64, 1, 0, 0)
    # per chunk and value head: W, U, dUp, dX (C x 64), S, dS, Z (64 x 64), T (C x C), G (C);
    # per token: dQ, dK of every value head; each piece rounded up to 256 bytes
    per_chunk = 4 * (4 * 64 * 64 + 3 * 64 * 64 + 64 * 64 + 64)
    assert per_chunk * 2 + 64 * 2 * 64 * 4 <= need <= per_chunk * 2 + 64 * 2 * 64 * 4 + 13 * 256
    assert lib.gdn_chunk_bwd_workspace_size(1, 64, 2, 3, 64, 64, 1, 0, 0) == (1 << 64) - 1
    assert bwd_call(chunk=32) == _lib.GDN_ERR_UNSUPPORTED
    assert bwd_call(do=None) == _lib.GDN_ERR_NULL
    assert bwd_call(db=None) == _lib.GDN_ERR_NULL
    assert bwd_call(Hv=3, Hqk=2) == _lib.GDN_ERR_SHAPE
    assert bwd_call(K=256) == _lib.GDN_ERR_SHAPE
    assert bwd_call(io=5) == _lib.GDN_ERR_DTYPE
    assert bwd_call(dq=FAKE + 4) == _lib.GDN_ERR_LAYOUT
    assert bwd_call(dg=FAKE + 2) == _lib.GDN_ERR_LAYOUT
    assert bwd_call(dinit=FAKE + 8) == _lib.GDN_ERR_LAYOUT
    assert bwd_call(B=2, cu=FAKE) == _lib.GDN_ERR_SHAPE
    assert bwd_call() == _lib.GDN_ERR_WORKSPACE
    assert bwd_call(ws=FAKE, wsb=need - 1) == _lib.GDN_ERR_WORKSPACE
    assert bwd_call(ws=FAKE + 8, wsb=need) == _lib.GDN_ERR_LAYOUT
    assert bwd_call(T=0, N=0, B=1, cu=FAKE) == _lib.GDN_OK


def test_wait_selftest_validates_on_the_host():
    """Argument errors of the bounded-wait self-test return before any launch (no GPU needed)."""
    lib = _lib.load()
    assert lib.gdn_selftest_wait_timeout(None, 1000, 0, None, None) == _lib.GDN_ERR_NULL


def test_backward_workspace_is_sized_per_path():
    """The tensor-core backward (bf16, K = V = 128) keeps bf16 operand tiles and none of the
    fp32 path's W / dUp / Z slots: its scratch is well under half of the fp32 layout's."""
    lib = _lib.load()
    args = (4, 32768, 16, 32, 128, 128, 4)
    tc = lib.gdn_chunk_bwd_workspace_size(*args, _lib.GDN_BF16, _lib.GDN_BF16)
    fp = lib.gdn_chunk_bwd_workspace_size(*args, _lib.GDN_F32, _lib.GDN_F32)
    print("backward scratch at 4 x 32768 tokens: %.2f GB (tensor cores), %.2f GB (fp32)"
          % (tc / 1e9, fp / 1e9))
    assert tc < 0.45 * fp
    # per (chunk, head): bf16 S, dS (32 KB each), U', dX (16 KB each), T and P (16 KB), the row
    # dots and the per-token vectors of the reverse pass (the grad pass sums the value heads of a
    # query/key head on chip: no per-value-head dq, dk scratch)
    NC, Hv = 32768 * 4 // 64 + 4, 32
    floor = NC * Hv * (32768 * 2 + 16384 * 3)
    assert floor <= tc <= floor * 1.03
