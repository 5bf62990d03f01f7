"""GPU checks of the host-buffer prefill (``kda_prefill_chunked_host``).

The call cuts the token range into pieces on chunk boundaries of the
sequences it cuts and carries each sequence's fp32 state between pieces, so
every chunk is computed exactly as in one ``kda_prefill_chunked`` call over
the whole batch (same chain form): outputs and final states must agree bit
for bit with that call, and within the usual tolerance with the oracle.
"""
import pytest
import torch

import kda_inputs as ki
import oracle
import serving_kda_chunked_gb300 as kda
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from serving_kda_chunked_gb300 import build
    build.build()
    kda.load()


def _device_call(inp):
    T, H, dk = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    need = kda.kda_prefill_workspace_size(N, T, H, dk, inp["v"].shape[-1], inp["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV) if need else None
    o, S_T = kda.kda_prefill_chunked(*(inp[n] for n in NAMES), inp["cu_seqlens"], inp["S0"],
                                     workspace=ws)
    if ws is not None:
        st = kda.kda_prefill_check(ws)
        assert st == kda.KDA_OK, kda.status_string(st)
    torch.cuda.synchronize()
    return o, S_T


def _host_call(inp, pinned=True):
    host = {n: inp[n].cpu() for n in NAMES}
    S0 = None if inp["S0"] is None else inp["S0"].cpu()
    if pinned:
        host = {n: t.pin_memory() for n, t in host.items()}
        S0 = None if S0 is None else S0.pin_memory()
    cu = inp["cu_seqlens"].cpu()
    T, H, dk = host["q"].shape
    N = cu.shape[0] - 1
    need = kda.kda_prefill_host_workspace_size(N, T, H, dk, host["v"].shape[-1],
                                               host["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o, S_T = kda.kda_prefill_chunked_host(*(host[n] for n in NAMES), cu, S0, workspace=ws)
    st = kda.kda_prefill_check(ws)
    assert st == kda.KDA_OK, kda.status_string(st)
    return o, S_T


def _ragged(dtype, d, H, seed):
    # lengths off the chunk grid, an empty sequence, and sequences longer than
    # one piece (512 tokens), so that cuts fall inside sequences
    lengths = [700, 0, 37, 1290, 64, 513, 5, 900]
    cfg = ki.PrefillConfig("ragged", H=H, d=d, dtype=dtype, n_seqs=len(lengths), s0_std=0.3)
    return ki.prefill_inputs(cfg, device=DEV, seed=seed, lengths=lengths)


def test_host_equals_device_single_sequence_workload():
    """T = 8192, H = 32, d = 128, bf16: pieces of 1,408 tokens halving to 320
    at the end (cuts on chunk boundaries)."""
    inp = ki.prefill_inputs("single", device=DEV)
    o_d, S_d = _device_call(inp)
    o_h, S_h = _host_call(inp)
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(S_h, S_d.cpu())


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp32", 64), ("bf16", 64)])
def test_host_equals_device_ragged(dtype, d):
    inp = _ragged(dtype, d, H=4, seed=11)
    o_d, S_d = _device_call(inp)
    o_h, S_h = _host_call(inp)
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(S_h, S_d.cpu())
    # the empty sequence passes its initial state through
    assert torch.equal(S_h[1], inp["S0"][1].cpu())


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp32", 64)])
def test_host_path_against_oracle(dtype, d):
    inp = _ragged(dtype, d, H=3, seed=12)
    o_h, S_h = _host_call(inp)
    o_ref, S_ref, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["S0"], inp["cu_seqlens"])
    tol = TOL[torch.bfloat16 if dtype == "bf16" else torch.float32]
    assert_close("o", o_h, o_ref, tol)
    assert_close("S_T", S_h, S_ref, tol)


def test_host_path_pageable_buffers():
    inp = _ragged("bf16", 128, H=2, seed=13)
    o_p, S_p = _host_call(inp, pinned=True)
    o_u, S_u = _host_call(inp, pinned=False)
    assert torch.equal(o_p, o_u)
    assert torch.equal(S_p, S_u)


def test_host_path_zero_tokens_and_no_initial_state():
    """Every sequence empty: S_T = S0; with S0 omitted: zeros."""
    H, d = 2, 128
    q = torch.empty((0, H, d), dtype=torch.bfloat16)
    g = torch.empty((0, H, d), dtype=torch.float32)
    beta = torch.empty((0, H), dtype=torch.float32)
    cu = torch.zeros(3, dtype=torch.int32)
    S0 = torch.randn((2, H, d, d), dtype=torch.float32)
    _, S_T = kda.kda_prefill_chunked_host(q, q, q, g, beta, cu, S0)
    torch.cuda.synchronize()
    assert torch.equal(S_T, S0)
    _, S_T = kda.kda_prefill_chunked_host(q, q, q, g, beta, cu, None)
    torch.cuda.synchronize()
    assert torch.equal(S_T, torch.zeros_like(S0))


def test_host_path_many_short_sequences():
    """Dozens of sequences per piece; the pieces may take the other chain form
    than the whole batch would (it depends on the sequence count), so the
    check is against the oracle."""
    lengths = [3, 1, 0, 2, 64, 7] * 120
    cfg = ki.PrefillConfig("short", H=2, d=128, dtype="bf16", n_seqs=len(lengths), s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=14, lengths=lengths)
    o_h, S_h = _host_call(inp)
    o_ref, S_ref, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["S0"], inp["cu_seqlens"])
    assert_close("o", o_h, o_ref, 2e-3)
    assert_close("S_T", S_h, S_ref, 2e-3)
