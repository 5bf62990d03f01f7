"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function that ``include/*.h`` declares,
and reject malformed or unsupported arguments on the host before touching the
GPU.  Only argument combinations that are rejected (or are documented no-ops)
are called here, so no CUDA work is issued.
"""
import ctypes
import glob
import os
import re

import pytest

import serving_kda_chunked_gb300 as kda
from serving_kda_chunked_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(kda_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = _declared_functions()
    for n in ("kda_prefill_chunked", "kda_decode_step", "kda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), "libkda.so does not export %s" % name


def test_status_strings(lib):
    assert kda.status_string(kda.KDA_OK) == "KDA_OK"
    assert "INVALID" in kda.status_string(kda.KDA_ERR_INVALID_ARG)
    assert "UNSUPPORTED" in kda.status_string(kda.KDA_ERR_UNSUPPORTED)
    assert "UNKNOWN" in kda.status_string(99)
    assert kda.abi_version() >> 16 == 2


P = 0x10000  # a 16-byte aligned stand-in address; never dereferenced here


def _prefill(lib, fn="kda_prefill_chunked", **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, S0=None, cu=P, N=1, T=64, H=2, dk=128,
             dv=128, dtype=0, chunk=64, o=P, S_T=P, ws=None, ws_bytes=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return getattr(lib, fn)(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]),
        vp(a["S0"]), vp(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"],
        a["dtype"], a["chunk"], vp(a["o"]), vp(a["S_T"]), vp(a["ws"]), a["ws_bytes"], None)


def _decode(lib, fn="kda_decode_step", **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, S=P, B=4, H=2, dk=128, dv=128, dtype=0, o=P)
    a.update(kw)
    vp = ctypes.c_void_p
    return getattr(lib, fn)(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), vp(a["S"]),
        a["B"], a["H"], a["dk"], a["dv"], a["dtype"], vp(a["o"]), None)


@pytest.mark.parametrize("kw,expect", [
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(N=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-5), kda.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(chunk=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(chunk=0), kda.KDA_ERR_INVALID_ARG),
    (dict(q=None), kda.KDA_ERR_INVALID_ARG),
    (dict(g=None), kda.KDA_ERR_INVALID_ARG),
    (dict(o=None), kda.KDA_ERR_INVALID_ARG),
    (dict(cu=None), kda.KDA_ERR_INVALID_ARG),
    (dict(S_T=None), kda.KDA_ERR_INVALID_ARG),
    (dict(q=P + 2), kda.KDA_ERR_INVALID_ARG),
    (dict(v=P + 8), kda.KDA_ERR_INVALID_ARG),
    (dict(S0=P + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(beta=P + 1), kda.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=10), kda.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=0), kda.KDA_OK),                      # empty batch: no-op
    (dict(ws=None), kda.KDA_ERR_INVALID_ARG),          # bf16, d=128 needs a workspace
    (dict(ws=P, ws_bytes=1024), kda.KDA_ERR_INVALID_ARG),
    (dict(ws=P + 8, ws_bytes=1 << 40), kda.KDA_ERR_INVALID_ARG),
])
def test_prefill_host_validation(lib, kw, expect):
    assert _prefill(lib, **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(B=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(dtype=2), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=32, dv=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(S=None), kda.KDA_ERR_INVALID_ARG),
    (dict(beta=None), kda.KDA_ERR_INVALID_ARG),
    (dict(S=P + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(o=P + 2), kda.KDA_ERR_INVALID_ARG),
    (dict(B=0), kda.KDA_OK),                           # empty batch: no-op
])
def test_decode_host_validation(lib, kw, expect):
    assert _decode(lib, **kw) == expect


def _decode_pooled(lib, fn="kda_decode_step_pooled", **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, S=P, slots=P, Pn=8, B=4, H=2, dk=128, dv=128,
             dtype=0, o=P)
    a.update(kw)
    vp = ctypes.c_void_p
    return getattr(lib, fn)(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), vp(a["S"]),
        vp(a["slots"]), a["Pn"], a["B"], a["H"], a["dk"], a["dv"], a["dtype"], vp(a["o"]), None)


@pytest.mark.parametrize("kw,expect", [
    (dict(Pn=0), kda.KDA_ERR_INVALID_ARG),
    (dict(slots=None), kda.KDA_ERR_INVALID_ARG),
    (dict(slots=P + 2), kda.KDA_ERR_INVALID_ARG),
    (dict(S=None), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=64, dv=128), kda.KDA_ERR_UNSUPPORTED),
    (dict(B=0), kda.KDA_OK),
])
def test_decode_pooled_host_validation(lib, kw, expect):
    assert _decode_pooled(lib, **kw) == expect
    if "dk" not in kw:   # the per-head-gate form validates the same way (g: 4-byte alignment)
        assert _decode_pooled(lib, fn="kda_gdn_decode_step_pooled", **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(g=None), kda.KDA_ERR_INVALID_ARG),
    (dict(g=P + 2), kda.KDA_ERR_INVALID_ARG),     # one gate per head: 4-byte alignment
    (dict(q=P + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(ws=None), kda.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=0), kda.KDA_OK),
])
def test_gdn_prefill_host_validation(lib, kw, expect):
    assert _prefill(lib, fn="kda_gdn_prefill_chunked", **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(g=None), kda.KDA_ERR_INVALID_ARG),
    (dict(g=P + 1), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=32, dv=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(B=0), kda.KDA_OK),
])
def test_gdn_decode_host_validation(lib, kw, expect):
    assert _decode(lib, fn="kda_gdn_decode_step", **kw) == expect


def test_workspace_size_query(lib):
    n = kda.kda_prefill_workspace_size(1, 8192, 32, 128, 128, kda.KDA_BF16)
    # header + chunk table, then one 74,240-byte operand block per (chunk, head)
    assert n == 1024 + (8192 // 64 + 1) * 32 * 74240
    # long inputs are processed in windows of 2048 chunks
    big = kda.kda_prefill_workspace_size(1, 1 << 20, 32, 128, 128, kda.KDA_BF16)
    assert big == 1024 + 2048 * 32 * 74240
    # one sequence with few heads adds the chunk-affine scan's segment maps:
    # H=2, 129 chunks -> 8 segments, 3 fp32 128x128 matrices each per head
    small = kda.kda_prefill_workspace_size(1, 8192, 2, 128, 128, kda.KDA_BF16)
    images = 1024 + (8192 // 64 + 1) * 2 * 74240
    assert small == ((images + 255) // 256) * 256 + 2 * 8 * 3 * 65536
    assert kda.kda_prefill_workspace_size(1, 8192, 32, 128, 128, kda.KDA_FP32) == 0
    assert kda.kda_prefill_workspace_size(1, 8192, 32, 64, 64, kda.KDA_BF16) == 0
    assert kda.kda_prefill_workspace_size(1, 8192, 32, 96, 96, kda.KDA_BF16) == 0


def test_noalloc_scratch_size(lib):
    assert kda.kda_noalloc_scratch_bytes() == 64 << 20


def test_binding_rejects_host_tensors(lib):
    import torch
    q = torch.zeros(4, 2, 64)
    with pytest.raises(ValueError, match="CUDA"):
        kda.kda_decode_step(q, q, q, q, torch.zeros(4, 2), torch.zeros(4, 2, 64, 64))
    with pytest.raises(ValueError, match="CUDA"):
        kda.kda_prefill_chunked_noalloc(q, q, q, q, torch.zeros(4, 2),
                                        torch.zeros(2, dtype=torch.int32))


def _host_prefill(lib, cu_vals, **kw):
    """kda_prefill_chunked_host with a real host offsets array."""
    cu = (ctypes.c_int32 * len(cu_vals))(*cu_vals)
    a = dict(q=P, k=P, v=P, g=P, beta=P, S0=None, N=len(cu_vals) - 1, T=cu_vals[-1], H=2,
             dk=128, dv=128, dtype=0, chunk=64, o=P, S_T=P, ws=P, ws_bytes=1 << 40)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.kda_prefill_chunked_host(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), vp(a["S0"]),
        ctypes.cast(cu, vp), a["N"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"], a["chunk"],
        vp(a["o"]), vp(a["S_T"]), vp(a["ws"]), a["ws_bytes"], None)


@pytest.mark.parametrize("cu_vals,kw,expect", [
    ([0, 64], dict(H=0), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    ([0, 64], dict(chunk=128), kda.KDA_ERR_UNSUPPORTED),
    ([0, 64], dict(dtype=5), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(q=None), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(S_T=None), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(ws=None), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(ws_bytes=4096), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(ws=P + 8), kda.KDA_ERR_INVALID_ARG),
    ([0, 64], dict(T=1 << 31), kda.KDA_ERR_INVALID_ARG),
    ([1, 64], {}, kda.KDA_ERR_INVALID_ARG),             # cu[0] != 0
    ([0, 64], dict(T=65), kda.KDA_ERR_INVALID_ARG),     # cu[N] != T
    ([0, 40, 30, 64], {}, kda.KDA_ERR_INVALID_ARG),     # decreasing offsets
    ([0], dict(N=0, T=0), kda.KDA_OK),                  # empty batch: no-op
    ([0], dict(N=0, T=5), kda.KDA_ERR_INVALID_ARG),
])
def test_host_prefill_validation(lib, cu_vals, kw, expect):
    assert _host_prefill(lib, cu_vals, **kw) == expect


def test_host_workspace_size(lib):
    f = kda.kda_prefill_host_workspace_size
    import torch
    small = f(1, 8192, 32, 128, 128, torch.bfloat16)
    # two staging slots of at least 512 tokens (q, k, v bf16, g, beta fp32; o bf16)
    # plus the prefill scratch of one piece and the state
    assert small >= 2 * 512 * 32 * (3 * 256 + 512 + 4 + 256) + 32 * 128 * 128 * 4
    assert f(1, 1 << 20, 32, 128, 128, torch.bfloat16) > small    # 16,384-token pieces
    assert f(4, 8192, 32, 128, 128, torch.bfloat16) > small       # more states
    assert f(1, 256, 2, 64, 64, torch.float32) > 0                # CUDA-core path
    assert f(0, 0, 32, 128, 128, torch.bfloat16) == 0
    assert f(1, 64, 32, 96, 96, torch.bfloat16) == 0
    assert f(1, 1 << 31, 32, 128, 128, torch.bfloat16) == 0


def test_device_pointer_check_runs_after_host_validation(lib):
    """A call that passes every host check reaches the device-pointer check
    (cudaPointerGetAttributes on each pointer) before any launch: without a
    device it reports KDA_ERR_CUDA; with one, the fake addresses used here are
    not device memory and are rejected as invalid.  Nothing is launched."""
    import torch
    ws = 0x100000
    st = _prefill(lib, ws=ws, ws_bytes=1 << 40)
    dst = _decode(lib)
    if torch.cuda.is_available():
        assert st == kda.KDA_ERR_INVALID_ARG and dst == kda.KDA_ERR_INVALID_ARG
    else:
        assert st == kda.KDA_ERR_CUDA and dst == kda.KDA_ERR_CUDA


def test_noalloc_check_without_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("covered by the GPU tests")
    assert lib.kda_prefill_noalloc_check(None) == kda.KDA_ERR_CUDA


def test_binding_requires_one_device(lib):
    """All tensors of a call must be on q's device (meta tensors stand in for a
    second device: the check looks at devices only)."""
    import torch
    from serving_kda_chunked_gb300 import _binding
    dev = torch.device("cuda", 0)
    _binding._same_device(torch.device("meta"), k=torch.empty(1, device="meta"), S0=None)
    with pytest.raises(ValueError, match="one device"):
        _binding._same_device(dev, k=torch.empty(1, device="meta"))
    with pytest.raises(ValueError, match="one device"):
        _binding._same_device(dev, workspace=torch.empty(1))
