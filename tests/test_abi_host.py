"""The C-ABI library loads without a GPU, exports every symbol include/fa.h
declares, and rejects bad arguments on the host before anything is launched."""
import os
import re

import pytest

import io_aware_exact_09_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fa.build()
    return fa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fa.EXPORTED)


def test_status_strings_and_sizes(L):
    assert fa.fa_status_string(0) == "ok"
    assert "timed out" in fa.fa_status_string(5)
    # every code the header declares has its own string; anything else is unknown
    strs = [fa.fa_status_string(c) for c in range(7)]
    assert len(set(strs)) == 7 and all(x and x != "unknown status" for x in strs), strs
    assert fa.fa_status_string(7) == fa.fa_status_string(-1) == "unknown status"
    assert fa.fa_tile_size() == 128
    assert fa.fa_fwd_workspace_size(1, 2, 128, 64) == 256
    # status + D [B,H,N] fp32 + dQacc [B,H,N,d] fp32, 256-byte rounded
    assert fa.fa_bwd_workspace_size(1, 2, 128, 64) == 256 + 1024 + 65536
    assert fa.fa_bwd_workspace_size(1, 1, 3, 64) == 256 + 256 + 768
    # d = 128: + 128 KiB per CTA of a split key tile, for N > 128 only:
    # min(256, B * H * T * min(4, T)) of them, T = ceil(N / 128)
    slot = 128 * 256 * 4
    assert fa.fa_bwd_workspace_size(1, 2, 128, 128) == 256 + 1024 + 131072
    assert fa.fa_bwd_workspace_size(1, 1, 256, 128) == 256 + 1024 + 131072 + 4 * slot
    assert fa.fa_bwd_workspace_size(1, 2, 512, 128) == 256 + 4096 + 524288 + 32 * slot
    rows = 16 * 16384
    assert fa.fa_bwd_workspace_size(1, 16, 16384, 128) == 256 + rows * 4 + rows * 128 * 4 + 256 * slot
    # the forward's split area (FP8 forward): d = 128 and at least 32 key tiles,
    # min(512, B * H * ceil(T / 2) * min(4, T / 16)) slots of 2 x 128 x 130 fp32
    fslot = 2 * 128 * 130 * 4
    assert fa.fa_fwd_workspace_size(1, 2, 4095, 128) == 256
    assert fa.fa_fwd_workspace_size(1, 2, 4096, 128) == 256 + 64 * fslot
    assert fa.fa_fwd_workspace_size(1, 1, 8192, 128) == 256 + 128 * fslot
    assert fa.fa_fwd_workspace_size(1, 16, 16384, 128) == 256 + 512 * fslot
    assert fa.fa_fwd_workspace_size(4, 16, 16384, 64) == 256
    # the ragged backward does not split
    assert fa.fa_bwd_varlen_workspace_size(16, 16384, 128) == 256 + rows * 4 + rows * 128 * 4
    assert fa.fa_host_workspace_size(1, 2, 128, 64, 1) > fa.fa_host_workspace_size(1, 2, 128, 64, 0)


def _fwd(B=1, H=1, N=128, d=64, scale=0.125, ptr=256, ws=256, wsz=256):
    return fa.lib().fa_fwd(ptr, ptr, ptr, ptr, ptr, B, H, N, d, scale, 0, None, None, ws, wsz, None)


def test_forward_argument_errors(L):
    assert _fwd(d=96) == 2                 # FA_ERR_UNSUPPORTED
    assert _fwd(d=256) == 2
    assert _fwd(B=-1) == 1                 # FA_ERR_INVALID_ARGUMENT
    assert _fwd(scale=float("nan")) == 1
    assert _fwd(scale=0.0) == 1
    assert _fwd(scale=-1.0) == 1
    assert _fwd(ptr=None) == 1
    assert _fwd(ptr=258) == 1              # misaligned
    assert _fwd(ws=None) == 3              # FA_ERR_WORKSPACE
    assert _fwd(wsz=8) == 3
    assert _fwd(B=0) == 0                  # empty: nothing to do
    assert _fwd(N=0) == 0


def test_size_limits(L):
    """The grids number (b*h) and (tile, b*h) items in 32-bit integers: past
    INT_MAX the calls return FA_ERR_UNSUPPORTED before touching the GPU; one
    tile short of it they go on to the next check (a missing workspace).  A
    block mask is listed per row of at most 2048 key tiles."""
    assert _fwd(B=1 << 16, H=1 << 16) == 2                       # B*H = 2^32
    assert _fwd(B=1 << 13, H=1 << 13, N=128 * 32) == 2           # tiles * B*H = 2^31
    assert _fwd(B=1 << 13, H=1 << 13, N=128 * 31, ws=None) == 3  # 31 * 2^26 < 2^31
    f = fa.lib().fa_fwd
    assert f(256, 256, 256, 256, 256, 1, 1, 128 * 2049, 64, 0.125, 0, None, 256, 256, 256, None) == 2
    b = fa.lib().fa_bwd
    ok_ws = fa.fa_bwd_workspace_size(1, 1, 128, 64)
    assert b(256, 256, 256, 256, 256, 256, 256, 256, 256, 1 << 16, 1 << 16, 128, 64, 0.1, 0, None, None, 256,
             ok_ws, None) == 2
    assert b(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 1, 128 * 2049, 64, 0.1, 0, None, 256, 256,
             1 << 40, None) == 2
    # the host-buffer path and the no-alloc backward reject it before any CUDA
    # call (here, without a GPU, any CUDA call would fail with FA_ERR_CUDA)
    h = fa.lib().fa_attention_host
    need = fa.fa_host_workspace_size(1, 1, 128 * 2049, 64, 0)
    assert h(256, 256, 256, None, 256, 256, None, None, None, 1, 1, 128 * 2049, 64, 0.1, 0, None, 256, 256, need,
             None) == 2
    n = fa.lib().fa_bwd_noalloc
    assert n(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 1, 128 * 2049, 64, 0.1, 0, None, 256, None) == 2


def test_backward_and_plan_argument_errors(L):
    b = fa.lib().fa_bwd
    ok_ws = fa.fa_bwd_workspace_size(1, 1, 128, 64)
    assert b(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 1, 128, 96, 0.1, 0, None, None, 256, ok_ws,
             None) == 2
    assert b(256, 256, 256, 256, 256, 256, None, 256, 256, 1, 1, 128, 64, 0.1, 0, None, None, 256, ok_ws,
             None) == 1
    assert b(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 1, 128, 64, 0.1, 0, None, None, 256, ok_ws - 1,
             None) == 3
    assert b(256, 256, 256, 256, 256, 256, 256, 256, 256, 0, 1, 128, 64, 0.1, 0, None, None, None, 0,
             None) == 0
    p = fa.lib().fa_tile_plan
    assert p(-1, 128, 0, None, None, 256, 256, 256, None) == 1
    assert p(1, 128, 0, None, None, None, 256, 256, None) == 1
    assert p(1, 128, 0, None, None, 256, None, 256, None) == 3
    assert p(0, 128, 0, None, None, None, None, 0, None) == 0


def test_host_path_argument_errors(L):
    h = fa.lib().fa_attention_host
    assert h(256, 256, 256, None, 256, 256, None, None, None, 1, 1, 128, 80, 0.1, 0, None, None, 256, 1 << 30,
             None) == 2
    assert h(256, 256, 256, 256, 256, 256, None, 256, 256, 1, 1, 128, 64, 0.1, 0, None, None, 256, 1 << 30,
             None) == 1  # backward requested without dQ
    assert h(256, 256, 256, None, 256, 256, None, None, None, 1, 1, 128, 64, 0.1, 0, None, None, 256, 16,
             None) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.import_module("io_aware_exact_09_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mod.lib()


def test_decode_argument_errors(L):
    dec = fa.lib().fa_decode
    ws = fa.fa_decode_workspace_size(1, 1, 1, 1000, 128, 0)
    assert ws > 256
    assert dec(256, 256, 256, 256, 256, 1, 1, 1, 1000, 96, 0.1, 0, None, 0, 256, ws, None) == 2
    assert dec(256, 256, 256, 256, 256, 1, 1, -1, 1000, 128, 0.1, 0, None, 0, 256, ws, None) == 1
    assert dec(None, 256, 256, 256, 256, 1, 1, 1, 1000, 128, 0.1, 0, None, 0, 256, ws, None) == 1
    assert dec(256, 256, 256, 256, 256, 1, 1, 1, 1000, 128, 0.1, 0, None, 0, 256, ws - 16, None) == 3
    assert dec(256, 256, 256, 256, 256, 1, 1, 0, 1000, 128, 0.1, 0, None, 0, None, 0, None) == 0
    # more splits requested than key tiles: the workspace query caps it the same way
    assert fa.fa_decode_workspace_size(1, 1, 1, 1000, 128, 1000) == fa.fa_decode_workspace_size(1, 1, 1, 1000, 128, 8)


def test_selftest_argument_errors(L):
    # rejected before any launch: no workspace, or too small for its result words
    st = fa.lib().fa_selftest_wait_timeout
    assert st(None, 256, None) == 3
    assert st(256, 16, None) == 3
    assert st(258, 256, None) == 3
