"""The bounded-wait timeout path and the device-pointer checks, on the GPU.

Every device-side wait of the tensor-core prefill is bounded: a wait that
gives up records KDA_ERR_TIMEOUT in the call's status word, the kernel
unwinds, and the state-chain kernels of the call then write nothing.  To make
that path run without hanging or faulting anything, the test uses
``libkda_faultinj.so`` -- the same sources built with KDA_FAULT_INJECTION --
whose ``kda_test_force_timeout`` makes the per-chunk kernel wait on an
mbarrier that nothing arrives at, *before* it allocates tensor memory or
issues any copy or MMA.  The wait gives up after 64 polls with nothing in
flight, so the context stays usable, which the test then shows by running the
same library normally and checking the result against the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
import serving_kda_chunked_gb300 as kda
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def libs():
    from serving_kda_chunked_gb300 import build
    build.build()
    main = kda.load()
    fi = ctypes.CDLL(build.FAULTINJ_LIB)
    for lib in (fi,):
        lib.kda_prefill_chunked.argtypes = main.kda_prefill_chunked.argtypes
        lib.kda_prefill_chunked.restype = ctypes.c_int
        lib.kda_prefill_chunked_noalloc.argtypes = main.kda_prefill_chunked_noalloc.argtypes
        lib.kda_prefill_chunked_noalloc.restype = ctypes.c_int
        lib.kda_prefill_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.kda_prefill_check.restype = ctypes.c_int
        lib.kda_prefill_noalloc_check.argtypes = [ctypes.c_void_p]
        lib.kda_prefill_noalloc_check.restype = ctypes.c_int
        lib.kda_prefill_workspace_size.argtypes = main.kda_prefill_workspace_size.argtypes
        lib.kda_prefill_workspace_size.restype = ctypes.c_uint64
        lib.kda_test_force_timeout.argtypes = [ctypes.c_int32]
        lib.kda_test_force_timeout.restype = None
    assert not hasattr(main, "kda_test_force_timeout"), "the library must not carry the hook"
    return main, fi


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _inputs(seed=7):
    cfg = ki.PrefillConfig("timeout", H=4, d=128, dtype="bf16", n_seqs=3, s0_std=0.05)
    return ki.prefill_inputs(cfg, device=DEV, seed=seed, lengths=[300, 0, 170])


def _call(lib, inp, o, S_T, ws):
    q, k, v, g, beta, S0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "S0", "cu_seqlens"))
    T, H, d = q.shape
    N = cu.shape[0] - 1
    if ws is None:
        return lib.kda_prefill_chunked_noalloc(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0),
                                               _p(cu), N, T, H, d, d, kda.KDA_BF16, 64, _p(o),
                                               _p(S_T), _stream())
    return lib.kda_prefill_chunked(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(cu), N, T,
                                   H, d, d, kda.KDA_BF16, 64, _p(o), _p(S_T), _p(ws),
                                   ws.numel(), _stream())


def _check_against_oracle(inp, o, S_T):
    o_ref, S_ref, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["S0"], inp["cu_seqlens"])
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


@pytest.mark.parametrize("api", ["workspace", "noalloc"])
def test_forced_timeout_reports_and_leaves_outputs_untouched(libs, api):
    _, fi = libs
    inp = _inputs()
    T, H, d = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    ws = None
    if api == "workspace":
        need = fi.kda_prefill_workspace_size(N, T, H, d, d, kda.KDA_BF16, 64)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)

    def status():
        if ws is None:
            return fi.kda_prefill_noalloc_check(_stream())
        return fi.kda_prefill_check(_p(ws), _stream())

    sentinel = 12345.0
    o = torch.full((T, H, d), sentinel, dtype=torch.bfloat16, device=DEV)
    S_T = torch.full((N, H, d, d), sentinel, dtype=torch.float32, device=DEV)
    fi.kda_test_force_timeout(1)
    try:
        st = _call(fi, inp, o, S_T, ws)
    finally:
        fi.kda_test_force_timeout(0)
    assert st == kda.KDA_OK       # the launch itself succeeds
    assert status() == kda.KDA_ERR_TIMEOUT
    # the per-chunk kernel gave up before writing anything; the chain kernels
    # saw the status and wrote nothing either
    assert bool((o == sentinel).all()), "o was written after a timeout"
    assert bool((S_T == sentinel).all()), "S_T was written after a timeout"

    # the context is still usable: the next call on the same device is normal
    st = _call(fi, inp, o, S_T, ws)
    assert st == kda.KDA_OK
    assert status() == kda.KDA_OK
    _check_against_oracle(inp, o, S_T)


def test_timeout_hook_off_matches_library(libs):
    """With the hook off, the test build computes what the library computes."""
    main, fi = libs
    inp = _inputs(seed=8)
    T, H, d = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    need = main.kda_prefill_workspace_size(N, T, H, d, d, kda.KDA_BF16, 64)
    outs = []
    for lib in (main, fi):
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        o = torch.empty((T, H, d), dtype=torch.bfloat16, device=DEV)
        S_T = torch.empty((N, H, d, d), dtype=torch.float32, device=DEV)
        assert _call(lib, inp, o, S_T, ws) == kda.KDA_OK
        assert lib.kda_prefill_check(_p(ws), _stream()) == kda.KDA_OK
        outs.append((o, S_T))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_device_entry_points_reject_host_memory(libs):
    """Every device pointer is checked: page-locked or pageable host memory in
    place of a device tensor is rejected before any launch."""
    main, _ = libs
    inp = _inputs(seed=9)
    T, H, d = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    need = main.kda_prefill_workspace_size(N, T, H, d, d, kda.KDA_BF16, 64)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o = torch.empty((T, H, d), dtype=torch.bfloat16, device=DEV)
    S_T = torch.empty((N, H, d, d), dtype=torch.float32, device=DEV)
    pinned_q = inp["q"].cpu().pin_memory()
    pageable_o = np.zeros((T, H, d), dtype=np.uint16)
    # host q (page-locked: reachable by the device, still rejected)
    bad = dict(inp)
    bad["q"] = pinned_q
    assert _call(main, bad, o, S_T, ws) == kda.KDA_ERR_INVALID_ARG
    # pageable host memory as the output
    q, k, v, g, beta, S0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "S0", "cu_seqlens"))
    st = main.kda_prefill_chunked(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(cu), N, T, H,
                                  d, d, kda.KDA_BF16, 64,
                                  ctypes.c_void_p(pageable_o.ctypes.data), _p(S_T), _p(ws),
                                  ws.numel(), _stream())
    assert st == kda.KDA_ERR_INVALID_ARG
    # host workspace
    ws_host = torch.empty(need, dtype=torch.uint8).pin_memory()
    assert _call(main, inp, o, S_T, ws_host) == kda.KDA_ERR_INVALID_ARG
    # decode: a host state
    dinp = ki.decode_inputs("decode", device=DEV, steps=1, B=2, H=2)
    S_host = dinp["S0"].cpu().pin_memory()
    od = torch.empty((2, 2, 128), dtype=torch.bfloat16, device=DEV)
    st = main.kda_decode_step(_p(dinp["q"][0]), _p(dinp["k"][0]), _p(dinp["v"][0]),
                              _p(dinp["g"][0]), _p(dinp["beta"][0]), _p(S_host), 2, 2, 128,
                              128, kda.KDA_BF16, _p(od), _stream())
    assert st == kda.KDA_ERR_INVALID_ARG
    # and the same call with device memory goes through
    assert _call(main, inp, o, S_T, ws) == kda.KDA_OK
    assert main.kda_prefill_check(_p(ws), _stream()) == kda.KDA_OK
    _check_against_oracle(inp, o, S_T)
