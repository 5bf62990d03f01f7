"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Inputs come from ``kda_inputs`` (seeded, drawn on the GPU), the oracle
consumes exactly the stored values, and every output is compared with the
metric in ``parity.py``: err <= 2e-3 for bf16 inputs with fp32 state, <= 1e-5
for fp32 inputs.  Sizes span several chunks and ragged tails; the full-size
workloads are checked in full where the oracle finishes in seconds, else on
the sampled subsets named in each test.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
import serving_kda_chunked_gb300 as kda
from parity import TOL, assert_close, err, oracle_prefill_windowed

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from serving_kda_chunked_gb300 import build
    build.build()
    kda.load()


def _checked(fn):
    """A prefill entry point with an explicit workspace whose device status
    (a bounded wait that gave up) is checked after the call."""
    def call(q, k, v, g, beta, cu_seqlens, S0=None, **kw):
        T, H, dk = q.shape
        need = kda.kda_prefill_workspace_size(cu_seqlens.shape[0] - 1, T, H, dk, v.shape[-1],
                                              q.dtype)
        ws = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
        out = fn(q, k, v, g, beta, cu_seqlens, S0, workspace=ws, **kw)
        st = kda.kda_prefill_check(ws)
        assert st == kda.KDA_OK, kda.status_string(st)
        return out
    return call


prefill = _checked(kda.kda_prefill_chunked)
gdn_prefill = _checked(kda.kda_gdn_prefill_chunked)


def _run_prefill(inp, chunk=64, S0=None):
    S0 = inp["S0"] if S0 is None else S0
    o, S_T = prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                     inp["cu_seqlens"], S0, chunk=chunk)
    torch.cuda.synchronize()
    return o, S_T


def _oracle_prefill(inp, S0="default"):
    S0 = inp["S0"] if isinstance(S0, str) else S0
    o, S_T, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               S0, inp["cu_seqlens"])
    return o, S_T


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_small_multi_step(d, dtype):
    cfg = ki.DecodeConfig("t", B=5, H=3, d=d, steps=12, dtype=dtype)
    inp = ki.decode_inputs(cfg, device=DEV, seed=1)
    S = inp["S0"].clone()
    S_ref = inp["S0"].double().cpu().numpy()
    for s in range(cfg.steps):
        o = kda.kda_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                                inp["beta"][s], S)
        o_ref, S_ref = oracle.decode_step(inp["q"][s], inp["k"][s], inp["v"][s],
                                          inp["g"][s], inp["beta"][s], S_ref)
        torch.cuda.synchronize()
        assert_close("o step %d" % s, o, o_ref, TOL[DT[dtype]])
        assert_close("S step %d" % s, S, S_ref, TOL[DT[dtype]])


def test_decode_workload_first_steps_full():
    """B=256, H=32, d=128 decode: every sequence and head, first 8 steps."""
    inp = ki.decode_inputs("decode", device=DEV, steps=8)
    S = inp["S0"].clone()
    S_ref = inp["S0"].double().cpu().numpy()
    for s in range(8):
        o = kda.kda_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                                inp["beta"][s], S)
        o_ref, S_ref = oracle.decode_step(inp["q"][s], inp["k"][s], inp["v"][s],
                                          inp["g"][s], inp["beta"][s], S_ref)
        torch.cuda.synchronize()
        assert_close("o", o, o_ref, 2e-3)
    assert_close("S", S, S_ref, 2e-3)


def test_decode_workload_1024_steps_sampled_sequences():
    """All 1024 in-place steps on the full B=256 batch; sequences 0..7 (every
    head) are checked at every step.  A sequence's decode tokens form one
    sequence for the oracle's prefill, which is the same recurrence."""
    inp = ki.decode_inputs("decode", device=DEV)
    steps, nb = inp["q"].shape[0], 8
    S = inp["S0"].clone()
    o_hist = torch.empty((steps, nb, 32, 128), dtype=torch.bfloat16, device=DEV)
    for s in range(steps):
        o = kda.kda_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                                inp["beta"][s], S)
        o_hist[s] = o[:nb]
    torch.cuda.synchronize()
    seq = lambda x: x[:, :nb].transpose(0, 1).reshape((nb * steps,) + tuple(x.shape[2:]))
    o_ref, S_ref, _ = oracle.prefill(seq(inp["q"]), seq(inp["k"]), seq(inp["v"]),
                                     seq(inp["g"]), seq(inp["beta"]), inp["S0"][:nb],
                                     np.arange(nb + 1) * steps)
    o_ref = o_ref.reshape(nb, steps, 32, 128).transpose(1, 0, 2, 3)
    assert_close("o[1024 steps, seq 0..7]", o_hist, o_ref, 2e-3)
    assert_close("S[seq 0..7]", S[:nb], S_ref, 2e-3)


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
def test_prefill_tiny_fp32():
    """B=1, H=2, T=256, d=64, fp32 inputs: tolerance 1e-5."""
    inp = ki.prefill_inputs("tiny", device=DEV)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 1e-5)
    assert_close("S_T", S_T, S_ref, 1e-5)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_prefill_ragged_packed_batch(d, dtype):
    """Packed sequences of lengths that hit every chunk edge: empty, 1, one
    short of a chunk, exactly one chunk, one past, several chunks + tail."""
    lengths = [1, 63, 0, 64, 65, 200, 130, 7]
    cfg = ki.PrefillConfig("ragged", H=3, d=d, dtype=dtype, n_seqs=len(lengths),
                           s0_std=0.3)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=3, lengths=lengths)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, TOL[DT[dtype]])
    assert_close("S_T", S_T, S_ref, TOL[DT[dtype]])
    # the empty sequence passes its initial state through unchanged
    assert torch.equal(S_T[2], inp["S0"][2])


def test_prefill_single_sequence_workload():
    """B=1, H=32, T=8192, d=128, bf16: checked in full."""
    inp = ki.prefill_inputs("single", device=DEV)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


@pytest.mark.parametrize("variant,reps", [("kda", 60), ("gdn", 60), ("varlen", 12), ("scan", 30)])
def test_prefill_repeated_calls_are_bit_identical(variant, reps):
    """The same call, repeated, gives the same bits: the kernels have no
    reduction whose order depends on timing, so any difference is a race
    (a buffer reused before its last reader finished).  Other work of
    varying length is queued between calls to shift the timing.  The
    variants cover the slice chain (KDA, GDN), the wide chain form (varlen)
    and the chunk-affine scan (one sequence, H = 2)."""
    fn = prefill
    if variant == "varlen":
        inp = ki.prefill_inputs("varlen", device=DEV)
    elif variant == "scan":
        inp = ki.prefill_inputs(ki.prefill_config("single", H=2, T=131072), device=DEV)
    else:
        inp = ki.prefill_inputs("single", device=DEV, seed=0 if variant == "kda" else 14)
    if variant == "gdn":
        inp = dict(inp)
        inp["g"] = inp["g"][..., 0].contiguous()
        fn = gdn_prefill
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], inp["S0"])
    o0, S0 = fn(*args)
    torch.cuda.synchronize()
    o0, S0 = o0.clone(), S0.clone()
    bad = []
    for r in range(reps):
        if r % 3 == 1:
            torch.cuda._sleep(20000 * (r % 7))
        o, S_T = fn(*args)
        if not (torch.equal(o, o0) and torch.equal(S_T, S0)):
            bad.append(r)
    assert not bad, "calls %s differ from the first" % bad


def test_prefill_varlen_workload():
    """16 packed sequences, lengths in [512, 16384], S0 ~ N(0, 0.02^2): in full."""
    inp = ki.prefill_inputs("varlen", device=DEV)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


def test_prefill_long_context_workload():
    """T = 1,048,576, H=32, d=128, slow gates.  (i) A 65,536-token prefix call
    against the oracle in full.  (ii) The oracle continues from the GPU's
    prefix state over the remaining tokens on state columns 0..7 of every head
    (columns never mix, so this is exact for those columns) and is compared
    with the full call's final state.  (iii) The full call's first 65,536
    outputs equal the prefix call's bit for bit (same chunks, same order)."""
    inp = ki.prefill_inputs("long", device=DEV)
    T, P = inp["q"].shape[0], 65536
    o_full, S_full = _run_prefill(inp)
    pre = {key: inp[key][:P] for key in ("q", "k", "v", "g", "beta")}
    pre["cu_seqlens"] = torch.tensor([0, P], dtype=torch.int32, device=DEV)
    o_pre, S_pre = prefill(pre["q"], pre["k"], pre["v"], pre["g"],
                                           pre["beta"], pre["cu_seqlens"], None)
    torch.cuda.synchronize()
    # (iii)
    assert torch.equal(o_full[:P], o_pre)
    # (i)
    o_ref, S_ref = oracle_prefill_windowed(inp, 0, P, None)
    assert_close("o prefix", o_pre, o_ref, 2e-3)
    assert_close("S prefix", S_pre[0], S_ref, 2e-3)
    # (ii)
    cols = slice(0, 8)
    S_start = S_pre[0][..., cols].double().cpu().numpy()
    _, S_end = oracle_prefill_windowed(inp, P, T, S_start, cols=cols)
    assert_close("S_T (cols 0..7, from GPU prefix state)", S_full[0][..., cols], S_end, 2e-3)


# ---------------------------------------------------------------------------
# segmentation, aliasing, determinism, guards
# ---------------------------------------------------------------------------
def test_resume_from_state_is_exact_on_chunk_boundaries():
    cfg = ki.PrefillConfig("seg", H=4, d=128, dtype="bf16", T=640, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=5)
    o, S_T = _run_prefill(inp)
    T1 = 256
    cu1 = torch.tensor([0, T1], dtype=torch.int32, device=DEV)
    cu2 = torch.tensor([0, 640 - T1], dtype=torch.int32, device=DEV)
    sl = lambda x, a, b: x[a:b].contiguous()
    o1, S1 = prefill(*(sl(inp[n], 0, T1) for n in ("q", "k", "v", "g", "beta")),
                                     cu1, inp["S0"])
    o2, S2 = prefill(*(sl(inp[n], T1, 640) for n in ("q", "k", "v", "g", "beta")),
                                     cu2, S1)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o1, o2]), o)
    assert torch.equal(S2, S_T)


def test_prefill_then_decode_matches_longer_prefill():
    cfg = ki.PrefillConfig("pd", H=4, d=128, dtype="bf16", T=200, s0_std=0.05)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=6)
    n_dec, T0 = 8, 192
    cu0 = torch.tensor([0, T0], dtype=torch.int32, device=DEV)
    _, S = prefill(*(inp[n][:T0].contiguous() for n in ("q", "k", "v", "g", "beta")),
                                   cu0, inp["S0"])
    outs = []
    for t in range(T0, T0 + n_dec):
        outs.append(kda.kda_decode_step(*(inp[n][t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")),
                                        S))
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o decode tail", torch.cat(outs), o_ref[T0:T0 + n_dec], 2e-3)
    assert_close("S after decode", S, S_ref, 2e-3)


def test_state_in_place_alias_and_determinism():
    lengths = [300, 77]
    cfg = ki.PrefillConfig("alias", H=2, d=128, dtype="bf16", n_seqs=2, s0_std=0.2)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=7, lengths=lengths)
    o_a, S_a = _run_prefill(inp)
    o_b, S_b = _run_prefill(inp)
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b)
    S_io = inp["S0"].clone()
    o_c, S_c = prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                       inp["cu_seqlens"], S_io, S_T=S_io)
    torch.cuda.synchronize()
    assert S_c.data_ptr() == S_io.data_ptr()
    assert torch.equal(o_c, o_a) and torch.equal(S_c, S_a)


def test_outputs_stay_inside_their_buffers():
    """Guard rows around o and S_T keep their sentinel values."""
    lengths = [70, 129]
    cfg = ki.PrefillConfig("guard", H=2, d=128, dtype="bf16", n_seqs=2, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=8, lengths=lengths)
    T, G = sum(lengths), 16
    o_buf = torch.full((T + 2 * G, 2, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    s_buf = torch.full((2 + 2, 2, 128, 128), -3.0, dtype=torch.float32, device=DEV)
    o, S_T = prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["cu_seqlens"], inp["S0"], o=o_buf[G:G + T],
                                     S_T=s_buf[1:3])
    torch.cuda.synchronize()
    assert torch.all(o_buf[:G] == 7.0) and torch.all(o_buf[G + T:] == 7.0)
    assert torch.all(s_buf[0] == -3.0) and torch.all(s_buf[3] == -3.0)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


def test_corrupt_offsets_stay_in_bounds():
    """Offsets beyond T_total or decreasing are clamped into [0, T_total] on
    the device: [0, 60, 1000, 5] with T_total = 100 acts as [0, 60, 100, 100]
    (the last sequence is empty), and nothing is written outside o / S_T."""
    cfg = ki.PrefillConfig("bad", H=2, d=64, dtype="bf16", T=100)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=9)
    cu = torch.tensor([0, 60, 1000, 5], dtype=torch.int32, device=DEV)
    S0 = torch.zeros((3, 2, 64, 64), device=DEV)
    o, S_T = prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     cu, S0)
    torch.cuda.synchronize()
    o_ref, S_ref, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     None, [0, 60, 100, 100])
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)
    assert torch.all(S_T[2] == 0)


# ---------------------------------------------------------------------------
# decode over a state-slot pool
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_pooled_slots(dtype):
    """Sequences name their state slot in a pool; untouched slots stay
    bit-identical, a slot outside the pool skips its sequence (o row = 0)."""
    P, B, H, d, steps = 12, 7, 3, 128, 4
    cfg = ki.DecodeConfig("pool", B=B, H=H, d=d, steps=steps, dtype=dtype)
    inp = ki.decode_inputs(cfg, device=DEV, seed=11)
    gen = torch.Generator(device="cpu").manual_seed(5)
    pool = (torch.randn((P, H, d, d), generator=gen) * 0.05).to(DEV)
    ref = pool.double().cpu().numpy()
    tol = TOL[DT[dtype]]
    for s in range(steps):
        perm = torch.randperm(P, generator=gen)[:B].to(torch.int32)
        perm[3] = -1 if s % 2 == 0 else P + 2          # a skipped sequence
        slots = perm.to(DEV)
        before = pool.clone()
        o = kda.kda_decode_step_pooled(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                                       inp["beta"][s], pool, slots)
        torch.cuda.synchronize()
        live = [b for b in range(B) if 0 <= int(perm[b]) < P]
        idx = [int(perm[b]) for b in live]
        o_ref, S_new = oracle.decode_step(inp["q"][s][live], inp["k"][s][live], inp["v"][s][live],
                                          inp["g"][s][live], inp["beta"][s][live], ref[idx])
        ref[idx] = S_new
        assert_close("o", o[live], o_ref, tol)
        assert_close("pool slots", pool[idx], S_new, tol)
        assert torch.all(o[3] == 0)
        untouched = [p for p in range(P) if p not in idx]
        assert torch.equal(pool[untouched], before[untouched])


# ---------------------------------------------------------------------------
# strong gates: the pairwise intra-chunk path of the tensor-core kernel
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_prefill_strong_gates(dtype):
    """gate scale 8: a chunk's cumulative log-gate reaches hundreds, beyond
    the range where exp(gamma) and exp(-gamma) factor safely, so the
    intra-chunk products are formed pair by pair."""
    lengths = [64, 1, 190, 77]
    cfg = ki.PrefillConfig("strong", H=2, d=128, dtype=dtype, n_seqs=len(lengths),
                           s0_std=0.3, gate_scale=8.0)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=17, lengths=lengths)
    assert float(inp["g"].sum(0).min()) < -500.0
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, TOL[DT[dtype]])
    assert_close("S_T", S_T, S_ref, TOL[DT[dtype]])


def _strong_every_third_chunk(inp, scale=8.0):
    """Multiply the log-gate of every third 64-token chunk of each sequence
    (chunk index 1, 4, 7, ...) by ``scale``: those chunks leave the range of
    the single-reference factors, their neighbours do not."""
    g = inp["g"]
    for n, (a, b) in enumerate(zip(inp["cu_seqlens"][:-1].tolist(), inp["cu_seqlens"][1:].tolist())):
        for c0 in range(a + 64, b, 3 * 64):
            g[c0:min(c0 + 64, b)] *= scale
    return inp


@pytest.mark.parametrize("variant", ["kda", "gdn"])
def test_prefill_mixed_strong_chunks(variant):
    """Out-of-range chunks between ordinary ones, with several (chunk, head)
    tasks per CTA: a chunk on the pairwise path keeps its staging tiles until
    that path has read them, and the next task's loads start after it; the
    ordinary chunks around it take the tensor-core path in the same CTA."""
    lengths = [9000, 7000, 130, 64]
    cfg = ki.PrefillConfig("mixed", H=2, d=128, dtype="bf16", n_seqs=len(lengths), s0_std=0.3)
    inp = _strong_every_third_chunk(ki.prefill_inputs(cfg, device=DEV, seed=23, lengths=lengths))
    tasks = sum((L + 63) // 64 for L in lengths) * 2
    assert tasks > 3 * torch.cuda.get_device_properties(0).multi_processor_count
    if variant == "kda":
        o, S_T = _run_prefill(inp)
        o_ref, S_ref = _oracle_prefill(inp)
    else:
        gh = inp["g"][..., 0].contiguous()
        o, S_T = gdn_prefill(inp["q"], inp["k"], inp["v"], gh, inp["beta"], inp["cu_seqlens"],
                             inp["S0"])
        torch.cuda.synchronize()
        o_ref, S_ref, _ = oracle.gdn_prefill(inp["q"], inp["k"], inp["v"], gh, inp["beta"],
                                             inp["S0"], inp["cu_seqlens"])
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


# ---------------------------------------------------------------------------
# Gated DeltaNet: one gate per head and token
# ---------------------------------------------------------------------------
def _head_gate(g):
    """One log-gate per (token, head): the first channel of the per-channel draw."""
    return g[..., 0].contiguous()


def _gdn_case(inp):
    gh = _head_gate(inp["g"])
    o, S_T = gdn_prefill(inp["q"], inp["k"], inp["v"], gh, inp["beta"],
                                         inp["cu_seqlens"], inp["S0"])
    torch.cuda.synchronize()
    o_ref, S_ref, _ = oracle.gdn_prefill(inp["q"], inp["k"], inp["v"], gh, inp["beta"],
                                         inp["S0"], inp["cu_seqlens"])
    return o, S_T, o_ref, S_ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_gdn_prefill_ragged(d, dtype):
    lengths = [1, 63, 0, 64, 65, 200, 130, 7]
    cfg = ki.PrefillConfig("ragged", H=3, d=d, dtype=dtype, n_seqs=len(lengths), s0_std=0.3)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=13, lengths=lengths)
    o, S_T, o_ref, S_ref = _gdn_case(inp)
    assert_close("o", o, o_ref, TOL[DT[dtype]])
    assert_close("S_T", S_T, S_ref, TOL[DT[dtype]])
    assert torch.equal(S_T[2], inp["S0"][2])


def test_gdn_prefill_single_sequence_workload():
    """B=1, H=32, T=8192, d=128, bf16 with one gate per head: checked in full."""
    inp = ki.prefill_inputs("single", device=DEV, seed=14)
    o, S_T, o_ref, S_ref = _gdn_case(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


def test_gdn_prefill_strong_gates():
    lengths = [64, 190, 77]
    cfg = ki.PrefillConfig("strong", H=2, d=128, dtype="bf16", n_seqs=len(lengths),
                           s0_std=0.3, gate_scale=8.0)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=18, lengths=lengths)
    o, S_T, o_ref, S_ref = _gdn_case(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_gdn_decode_multi_step(d, dtype):
    cfg = ki.DecodeConfig("t", B=5, H=3, d=d, steps=10, dtype=dtype)
    inp = ki.decode_inputs(cfg, device=DEV, seed=19)
    S = inp["S0"].clone()
    S_ref = inp["S0"].double().cpu().numpy()
    for s in range(cfg.steps):
        gh = _head_gate(inp["g"][s])
        o = kda.kda_gdn_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], gh,
                                    inp["beta"][s], S)
        o_ref, S_ref = oracle.gdn_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], gh,
                                              inp["beta"][s], S_ref)
        torch.cuda.synchronize()
        assert_close("o step %d" % s, o, o_ref, TOL[DT[dtype]])
        assert_close("S step %d" % s, S, S_ref, TOL[DT[dtype]])


# ---------------------------------------------------------------------------
# many sequences (the one-CTA-per-head chain form) and degenerate gates
# ---------------------------------------------------------------------------
def test_prefill_many_short_sequences():
    """120 packed sequences of 0-200 tokens, H=4: 1,920 state slices, more than
    two waves, so the chain runs one CTA per (sequence, head)."""
    gen = torch.Generator(device="cpu").manual_seed(31)
    lengths = torch.randint(0, 201, (120,), generator=gen).tolist()
    lengths[5] = 0
    lengths[6] = 64
    lengths[7] = 1
    cfg = ki.PrefillConfig("many", H=4, d=128, dtype="bf16", n_seqs=len(lengths), s0_std=0.2)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=32, lengths=lengths)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)
    assert torch.equal(S_T[5], inp["S0"][5])


def test_prefill_thousands_of_sequences():
    """3,150 packed sequences (0-65 tokens, every chunk edge), H = 2: more
    sequences than the 1,024 threads of the chunk-table and window-plan
    kernels, and more chunks (3,150) than one window, so both kernels loop
    and the second window plans only the sequences left.  The host-buffer
    call (pieces of ~8,800 tokens over hundreds of sequences each) is checked
    against the oracle too."""
    lengths = [0, 1, 5, 17, 64, 65, 3] * 450
    cfg = ki.PrefillConfig("thousands", H=2, d=128, dtype="bf16", n_seqs=len(lengths),
                           s0_std=0.2)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=33, lengths=lengths)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)
    empty = [n for n, L in enumerate(lengths) if L == 0]
    assert torch.equal(S_T[empty], inp["S0"][empty])
    host = [inp[n].cpu() for n in ("q", "k", "v", "g", "beta")]
    o_h, S_h = kda.kda_prefill_chunked_host(*host, inp["cu_seqlens"].cpu(), inp["S0"].cpu())
    torch.cuda.synchronize()
    assert_close("o (host buffers)", o_h, o_ref, 2e-3)
    assert_close("S_T (host buffers)", S_h, S_ref, 2e-3)


@pytest.mark.parametrize("case", ["beta0", "gate0"])
def test_prefill_degenerate_gates(case):
    """beta = 0: nothing is written, the state only decays (o_t = S_t^T q_t with
    S_t = Diag(e^gamma_t) S0).  g = 0: no decay, the plain delta rule."""
    lengths = [150, 64, 9]
    cfg = ki.PrefillConfig("degen", H=2, d=128, dtype="bf16", n_seqs=len(lengths), s0_std=0.3)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=33, lengths=lengths)
    if case == "beta0":
        inp["beta"].zero_()
    else:
        inp["g"].zero_()
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


# ---------------------------------------------------------------------------
# chunk-affine scan: one long sequence with few heads, chunks cut into
# segments whose maps are chained (phase 0 / combine / phase 1)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,T", [(2, 8192 + 37), (1, 20000)])
def test_prefill_segment_scan(H, T):
    cfg = ki.PrefillConfig("scan", H=H, d=128, dtype="bf16", T=T, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=41)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


def test_prefill_segment_scan_two_windows():
    """H=1, 140,000 tokens: 2,188 chunks, two windows of segments, the state
    carried from the first window's last segment into the second."""
    cfg = ki.PrefillConfig("scan2", H=1, d=128, dtype="bf16", T=140000, s0_std=0.1,
                           gate_scale=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=42)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


def test_gdn_prefill_segment_scan():
    """One sequence, two heads, one gate per head: the chunk-affine scan path."""
    cfg = ki.PrefillConfig("gdnscan", H=2, d=128, dtype="bf16", T=5000, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=43)
    o, S_T, o_ref, S_ref = _gdn_case(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)


# ---------------------------------------------------------------------------
# CUDA graphs: both calls enqueue only kernels on the caller's stream, so a
# captured graph replays them exactly
# ---------------------------------------------------------------------------
def test_prefill_and_decode_replay_in_a_cuda_graph():
    cfg = ki.PrefillConfig("graph", H=4, d=128, dtype="bf16", T=700, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=51)
    dcfg = ki.DecodeConfig("graphd", B=3, H=4, d=128, steps=2, dtype="bf16")
    dec = ki.decode_inputs(dcfg, device=DEV, seed=52)
    T, H, d = inp["q"].shape
    ws = torch.empty(kda.kda_prefill_workspace_size(1, T, H, d, d, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    o = torch.empty_like(inp["v"])
    S_T = torch.empty_like(inp["S0"])
    S_dec = dec["S0"].clone()
    o_dec = torch.empty_like(dec["v"][0])

    def work():
        kda.kda_prefill_chunked(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                inp["cu_seqlens"], inp["S0"], o=o, S_T=S_T, workspace=ws)
        kda.kda_decode_step(dec["q"][0], dec["k"][0], dec["v"][0], dec["g"][0], dec["beta"][0],
                            S_dec, o=o_dec)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        work()                                  # eager, on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    o_ref, S_ref, od_ref, Sd_ref = o.clone(), S_T.clone(), o_dec.clone(), S_dec.clone()

    S_dec.copy_(dec["S0"])
    o.zero_(); S_T.zero_(); o_dec.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        work()
    graph.replay()
    torch.cuda.synchronize()
    assert kda.kda_prefill_check(ws) == kda.KDA_OK
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    assert torch.equal(o_dec, od_ref) and torch.equal(S_dec, Sd_ref)


def test_gdn_decode_pooled_slots():
    """Per-head gates over a state-slot pool."""
    P, B, H, d = 9, 5, 2, 128
    cfg = ki.DecodeConfig("gpool", B=B, H=H, d=d, steps=2, dtype="bf16")
    inp = ki.decode_inputs(cfg, device=DEV, seed=53)
    gen = torch.Generator(device="cpu").manual_seed(54)
    pool = (torch.randn((P, H, d, d), generator=gen) * 0.05).to(DEV)
    ref = pool.double().cpu().numpy()
    for s in range(2):
        perm = torch.randperm(P, generator=gen)[:B].to(torch.int32)
        perm[1] = -3
        slots = perm.to(DEV)
        before = pool.clone()
        gh = _head_gate(inp["g"][s])
        o = kda.kda_gdn_decode_step_pooled(inp["q"][s], inp["k"][s], inp["v"][s], gh,
                                           inp["beta"][s], pool, slots)
        torch.cuda.synchronize()
        live = [b for b in range(B) if 0 <= int(perm[b]) < P]
        idx = [int(perm[b]) for b in live]
        o_ref, S_new = oracle.gdn_decode_step(inp["q"][s][live], inp["k"][s][live],
                                              inp["v"][s][live], gh[live], inp["beta"][s][live],
                                              ref[idx])
        ref[idx] = S_new
        assert_close("o", o[live], o_ref, 2e-3)
        assert_close("pool slots", pool[idx], S_new, 2e-3)
        assert torch.all(o[1] == 0)
        untouched = [p for p in range(P) if p not in idx]
        assert torch.equal(pool[untouched], before[untouched])


def test_prefill_more_heads_than_one_wave():
    """H=48, one sequence: 192 chain slices, more than the SMs, so the slice
    chains run in two waves; 48 heads per chunk in the per-chunk kernel."""
    cfg = ki.PrefillConfig("h48", H=48, d=128, dtype="bf16", T=1000, s0_std=0.1)
    inp = ki.prefill_inputs(cfg, device=DEV, seed=71)
    o, S_T = _run_prefill(inp)
    o_ref, S_ref = _oracle_prefill(inp)
    assert_close("o", o, o_ref, 2e-3)
    assert_close("S_T", S_T, S_ref, 2e-3)
