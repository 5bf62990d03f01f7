"""The no-allocation prefill entry point against the regular one.

Callers that cannot allocate device memory (their allocator is owned by a
framework, or they only hold the tensors they were handed) use
``kda_prefill_chunked_noalloc``: it keeps its scratch in a fixed device array
inside the library instead of a caller-provided workspace.  This file is
collected last on purpose, so that a run stopping at the first failure has
run every other test before it.

Both entry points are called through the C ABI on the same inputs; the
outputs must agree within the parity tolerance (they use the same kernels, so
in practice they agree exactly).  Two calls in a row with different inputs
check that what the shared array keeps from the previous call does not leak
into the next one.
"""
import ctypes

import pytest
import torch

import kda_inputs as ki
import serving_kda_chunked_gb300 as kda
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from serving_kda_chunked_gb300 import build
    build.build()
    return kda.load()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _both(lib, inp):
    q, k, v, g, beta, S0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "S0", "cu_seqlens"))
    T, H, d = q.shape
    N = cu.shape[0] - 1
    o_ref = torch.empty_like(v)
    S_ref = torch.empty((N, H, d, d), dtype=torch.float32, device=DEV)
    ws_bytes = lib.kda_prefill_workspace_size(N, T, H, d, d, kda.KDA_BF16, 64)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    st = lib.kda_prefill_chunked(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(cu), N, T, H,
                                 d, d, kda.KDA_BF16, 64, _p(o_ref), _p(S_ref), _p(ws),
                                 ws_bytes, _stream())
    assert st == kda.KDA_OK, kda.status_string(st)
    # its device status too
    st = kda.kda_prefill_check(ws)
    assert st == kda.KDA_OK, kda.status_string(st)
    o = torch.full_like(v, float("nan"))
    S = torch.full((N, H, d, d), float("nan"), dtype=torch.float32, device=DEV)
    st = lib.kda_prefill_chunked_noalloc(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(cu),
                                         N, T, H, d, d, kda.KDA_BF16, 64, _p(o), _p(S),
                                         _stream())
    assert st == kda.KDA_OK, kda.status_string(st)
    # its device status: no bounded wait gave up
    st = lib.kda_prefill_noalloc_check(_stream())
    assert st == kda.KDA_OK, kda.status_string(st)
    torch.cuda.synchronize()
    return o, S, o_ref, S_ref


def test_noalloc_matches_regular_entry_point_on_two_calls(lib):
    # 32 heads need several windows of the 64 MiB array for ~4k tokens
    assert lib.kda_noalloc_scratch_bytes() == 64 << 20
    for seed, lengths in ((0, [2500, 1500]), (1, [3000, 0, 700])):
        cfg = ki.PrefillConfig("noalloc", H=32, d=128, dtype="bf16", n_seqs=len(lengths),
                               s0_std=0.02)
        inp = ki.prefill_inputs(cfg, device=DEV, seed=seed, lengths=lengths)
        o, S, o_ref, S_ref = _both(lib, inp)
        assert_close("o (seed %d)" % seed, o, o_ref.double().cpu().numpy(), 2e-3)
        assert_close("S_T (seed %d)" % seed, S, S_ref.double().cpu().numpy(), 2e-3)


def test_noalloc_rejects_what_does_not_fit(lib):
    x = torch.zeros(16, dtype=torch.float32, device=DEV)
    cu = torch.zeros(2, dtype=torch.int32, device=DEV)
    # one chunk of 1000 heads needs 74 MB > 64 MiB
    st = lib.kda_prefill_chunked_noalloc(_p(x), _p(x), _p(x), _p(x), _p(x), None, _p(cu), 1, 64,
                                         1000, 128, 128, kda.KDA_BF16, 64, _p(x), _p(x),
                                         _stream())
    assert st == kda.KDA_ERR_TOO_LARGE
    assert "no-allocation" in kda.status_string(st)


def test_noalloc_through_the_python_binding():
    """The binding's wrapper of the no-allocation entry point gives the same
    outputs as the regular call, into caller buffers."""
    cfg = ki.PrefillConfig("na_py", H=4, d=128, dtype="bf16", T=1000, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=61)
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], inp["S0"])
    o_ref, S_ref = kda.kda_prefill_chunked(*args)
    o = torch.empty_like(o_ref)
    S_T = torch.empty_like(S_ref)
    kda.kda_prefill_chunked_noalloc(*args, o=o, S_T=S_T)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
