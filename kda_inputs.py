"""Seeded synthetic inputs for the KDA prefill and decode workloads.

This module draws random tensors and nothing else: it holds no step of the
KDA recurrence.  Both the CUDA path (tests, bench) and the fp64 oracle consume
what it returns, so parity is always checked on identical stored values.

Workloads (the five shapes the library is measured and checked on):

* ``tiny``    -- B=1, H=2, T=256, dk=dv=64, fp32 q/k/v; S0 = 0; chunk 64.
* ``single``  -- B=1, H=32, T=8192, dk=dv=128, bf16 q/k/v; S0 = 0.
* ``varlen``  -- 16 packed sequences, lengths uniform in [512, 16384]
  (inclusive), H=32, d=128, bf16; S0 ~ N(0, 0.02^2) per sequence.
* ``long``    -- B=1, T=1,048,576, H=32, d=128, bf16; gates scaled by 0.1.
* ``decode``  -- 256 sequences x 1024 steps, H=32, d=128, bf16 per-step
  q/k/v; S0 ~ N(0, 0.02^2), fp32, updated in place.

Value recipe (every workload): q, k ~ N(0, 1) then L2-normalised over dk in
fp32 and stored in the workload's dtype; v ~ N(0, 1); beta = sigmoid(N(0, 1));
log-gate g = -softplus(N(0, 1)) * gate_scale, fp32, one value per channel.

Draw order from one generator seeded with ``seed`` on the target device:
q, k, v, x_g, x_beta, S0 (decode: S0 first, then q, k, v, x_g, x_beta over all
steps).  Large tensors are drawn window by window along the token (or step)
axis so that temporaries stay bounded.  Sequence lengths come from a separate
CPU generator so that shapes agree on every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

__all__ = ["PrefillConfig", "DecodeConfig", "PREFILL", "DECODE",
           "prefill_config", "prefill_inputs", "decode_inputs", "seq_lengths"]


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    H: int
    d: int
    dtype: str                       # "bf16" or "fp32" (q, k, v and o)
    T: int | None = None             # dense single sequence of length T
    n_seqs: int = 1
    len_range: tuple | None = None   # (lo, hi) inclusive, for packed batches
    gate_scale: float = 1.0
    s0_std: float = 0.0
    chunk: int = 64


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H: int
    d: int
    steps: int
    dtype: str = "bf16"
    gate_scale: float = 1.0
    s0_std: float = 0.02


PREFILL = {
    "tiny": PrefillConfig("tiny", H=2, d=64, dtype="fp32", T=256),
    "single": PrefillConfig("single", H=32, d=128, dtype="bf16", T=8192),
    "varlen": PrefillConfig("varlen", H=32, d=128, dtype="bf16", n_seqs=16,
                            len_range=(512, 16384), s0_std=0.02),
    "long": PrefillConfig("long", H=32, d=128, dtype="bf16", T=1 << 20,
                          gate_scale=0.1),
}
DECODE = {
    "decode": DecodeConfig("decode", B=256, H=32, d=128, steps=1024),
}

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}
_WINDOW_ELEMS = 1 << 28   # elements per drawn window (1 GiB of fp32)


def prefill_config(name: str, **overrides) -> PrefillConfig:
    return replace(PREFILL[name], **overrides)


def seq_lengths(cfg: PrefillConfig, seed: int = 0) -> list[int]:
    """Sequence lengths of a workload (CPU generator, machine independent)."""
    if cfg.len_range is None:
        return [int(cfg.T)] * cfg.n_seqs
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    lo, hi = cfg.len_range
    return [int(x) for x in torch.randint(lo, hi + 1, (cfg.n_seqs,), generator=gen)]


def _draw(shape, gen, device, window_axis0=True):
    """N(0,1) fp32 tensor, drawn in windows along axis 0."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    per_row = 1
    for s in shape[1:]:
        per_row *= int(s)
    rows = max(1, _WINDOW_ELEMS // max(per_row, 1))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen,
                                 device=device, dtype=torch.float32)
    return out


def _unit_rows(x: torch.Tensor, dtype) -> torch.Tensor:
    """L2-normalise the last axis in fp32, then store in ``dtype`` (windowed)."""
    out = torch.empty(x.shape, dtype=dtype, device=x.device)
    flat_in = x.view(-1, x.shape[-1])
    flat_out = out.view(-1, x.shape[-1])
    rows = max(1, _WINDOW_ELEMS // x.shape[-1])
    for r0 in range(0, flat_in.shape[0], rows):
        r1 = min(flat_in.shape[0], r0 + rows)
        flat_out[r0:r1] = torch.nn.functional.normalize(
            flat_in[r0:r1], dim=-1).to(dtype)
    return out


def _gate(x: torch.Tensor, scale: float) -> torch.Tensor:
    """g = -softplus(x) * scale, in place on the fp32 draw (windowed)."""
    flat = x.view(-1)
    for r0 in range(0, flat.numel(), _WINDOW_ELEMS):
        r1 = min(flat.numel(), r0 + _WINDOW_ELEMS)
        flat[r0:r1] = -torch.nn.functional.softplus(flat[r0:r1]) * scale
    return x


def prefill_inputs(cfg: PrefillConfig | str, device="cpu", seed: int = 0,
                   lengths: list[int] | None = None) -> dict:
    """Draw one prefill batch.

    Returns a dict with q, k [T, H, d] (cfg dtype), v [T, H, d] (cfg dtype),
    g [T, H, d] fp32, beta [T, H] fp32, S0 [N, H, d, d] fp32 or None,
    cu_seqlens [N+1] int32 (on ``device``), lengths (list) and cfg.
    """
    if isinstance(cfg, str):
        cfg = PREFILL[cfg]
    if lengths is None:
        lengths = seq_lengths(cfg, seed)
    T = int(sum(lengths))
    H, d = cfg.H, cfg.d
    dt = _TORCH_DTYPE[cfg.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _unit_rows(_draw((T, H, d), gen, device), dt)
    k = _unit_rows(_draw((T, H, d), gen, device), dt)
    v = _draw((T, H, d), gen, device)
    if dt != torch.float32:
        v = v.to(dt)
    g = _gate(_draw((T, H, d), gen, device), cfg.gate_scale)
    beta = torch.sigmoid(_draw((T, H), gen, device))
    S0 = None
    if cfg.s0_std > 0:
        S0 = _draw((len(lengths), H, d, d), gen, device) * cfg.s0_std
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    cu_seqlens = torch.tensor(cu, dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, cu_seqlens=cu_seqlens,
                lengths=list(lengths), cfg=cfg)


def decode_inputs(cfg: DecodeConfig | str, device="cpu", seed: int = 0,
                  steps: int | None = None, B: int | None = None,
                  H: int | None = None) -> dict:
    """Draw a decode workload: S0 [B, H, d, d] fp32, then per-step
    q, k, v [steps, B, H, d] (cfg dtype), g [steps, B, H, d] fp32 and
    beta [steps, B, H] fp32."""
    if isinstance(cfg, str):
        cfg = DECODE[cfg]
    cfg = replace(cfg, steps=steps if steps is not None else cfg.steps,
                  B=B if B is not None else cfg.B,
                  H=H if H is not None else cfg.H)
    n, Bn, Hn, d = cfg.steps, cfg.B, cfg.H, cfg.d
    dt = _TORCH_DTYPE[cfg.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    S0 = _draw((Bn, Hn, d, d), gen, device) * cfg.s0_std
    q = _unit_rows(_draw((n, Bn, Hn, d), gen, device), dt)
    k = _unit_rows(_draw((n, Bn, Hn, d), gen, device), dt)
    v = _draw((n, Bn, Hn, d), gen, device)
    if dt != torch.float32:
        v = v.to(dt)
    g = _gate(_draw((n, Bn, Hn, d), gen, device), cfg.gate_scale)
    beta = torch.sigmoid(_draw((n, Bn, Hn), gen, device))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, cfg=cfg)
