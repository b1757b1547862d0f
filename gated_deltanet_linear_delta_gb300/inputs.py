"""Seeded synthetic inputs for the gated delta rule layer.

This module draws random numbers and nothing else: it holds no arithmetic of
the method (no normalisation, no gates, no recurrence). Both the CUDA path and
the fp64 oracle are fed from it, so that they see identical values.

Recipe (one ``torch.Generator`` on the CPU, seeded, tensors drawn in the fixed
order q, k, v, g, b, state; every draw is fp32, then cast to the I/O dtype):

* q, k ~ N(0, 1), raw (the layer L2-normalises them per head itself);
* v ~ N(0, 1);
* g = -softplus(N(0, 1)): a log-decay, so alpha = exp(g) lies in (0, 1);
* b ~ N(0, 1): beta logits, so the effective beta = sigmoid(b) has the
  distribution "sigmoid(N(0,1))";
* initial states ~ N(0, 0.02) i.i.d. fp32 when a nonzero state is asked for;
* packed variable-length batches draw integer lengths uniformly from an
  inclusive range, from the same generator, before the tensors.

The "slow gate" variant (g = -softplus(N(0,1)) * 1e-3, b ~ N(-2, 1)) keeps the
state alive over thousands of tokens so that the state carried across chunks
and calls has a visible effect on the outputs. ``gate_scale`` multiplies the
drawn g (after the slow-gate factor, if any): values above 1 give fast decays,
whose in-block cumulative log-decay spans a wider range (about 51 * gate_scale
over 64 tokens on average).

Shapes (tokens packed): q, k [Ttot, Hk, dk]; v [Ttot, Hv, dv];
g, b [Ttot, Hv]; state [B, Hv, dv, dk] (fp32); cu_seqlens int32 [B+1].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.nn.functional as F

_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclass
class GDNBatch:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    b: torch.Tensor
    state: torch.Tensor | None  # fp32 [B, Hv, dv, dk] or None (= zeros)
    cu_seqlens: torch.Tensor | None  # int32 [B+1] or None (= B equal sequences)
    B: int
    T: int  # tokens per sequence when cu_seqlens is None, else total tokens
    Hk: int
    Hv: int
    dk: int
    dv: int
    chunk: int = 64
    meta: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return int(self.q.shape[0])

    def to(self, device) -> "GDNBatch":
        def mv(x):
            return None if x is None else x.to(device)
        return GDNBatch(mv(self.q), mv(self.k), mv(self.v), mv(self.g), mv(self.b), mv(self.state),
                        mv(self.cu_seqlens), self.B, self.T, self.Hk, self.Hv, self.dk, self.dv,
                        self.chunk, dict(self.meta))


def _draws(gen, Ttot, Hk, Hv, dk, dv, slow_gate: bool):
    q = torch.randn(Ttot, Hk, dk, generator=gen)
    k = torch.randn(Ttot, Hk, dk, generator=gen)
    v = torch.randn(Ttot, Hv, dv, generator=gen)
    g = -F.softplus(torch.randn(Ttot, Hv, generator=gen))
    b = torch.randn(Ttot, Hv, generator=gen)
    if slow_gate:
        g = g * 1e-3
        b = b - 2.0
    return q, k, v, g, b


def make_batch(B=1, T=64, Hk=2, Hv=2, dk=32, dv=32, dtype="f32", chunk=16, seed=0,
               init_state=False, state_std=0.02, lengths=None, slow_gate=False,
               gate_scale=1.0) -> GDNBatch:
    """Draw one batch. ``lengths`` (a list of ints) packs variable-length sequences."""
    gen = torch.Generator().manual_seed(seed)
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        B = len(lengths)
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        Ttot = int(cu[-1])
    else:
        cu = None
        Ttot = B * T
    q, k, v, g, b = _draws(gen, Ttot, Hk, Hv, dk, dv, slow_gate)
    if gate_scale != 1.0:
        g = g * gate_scale
    state = None
    if init_state:
        state = torch.randn(B, Hv, dv, dk, generator=gen) * state_std
    dt = _DTYPES[dtype]
    return GDNBatch(q.to(dt), k.to(dt), v.to(dt), g.to(dt), b.to(dt), state, cu, B,
                    Ttot if cu is not None else T, Hk, Hv, dk, dv, chunk,
                    {"seed": seed, "dtype": dtype, "slow_gate": slow_gate, "gate_scale": gate_scale})


def varlen_lengths(n=16, lo=256, hi=16384, seed=0) -> list[int]:
    """Integer lengths drawn uniformly from [lo, hi] (inclusive)."""
    gen = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def make_decode_inputs(N, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", seed=0, steps=1,
                       state_std=0.02, with_state=True):
    """Inputs for `steps` decode steps of N sequences: tensors with a leading step axis.

    Returns (q [steps,N,Hk,dk], k, v [steps,N,Hv,dv], g [steps,N,Hv], b, state [N,Hv,dv,dk] fp32).
    """
    gen = torch.Generator().manual_seed(seed)
    q, k, v, g, b = _draws(gen, steps * N, Hk, Hv, dk, dv, slow_gate=False)
    dt = _DTYPES[dtype]
    state = torch.randn(N, Hv, dv, dk, generator=gen) * state_std if with_state else None
    shp = lambda x: x.reshape(steps, N, *x.shape[1:]).to(dt)  # noqa: E731
    return shp(q), shp(k), shp(v), shp(g), shp(b), state


# The five workloads of the layer (sizes fixed here, by name).
def tiny_fp32(seed=0) -> GDNBatch:
    """B=1, T=64, Hk=Hv=2, dk=dv=32, fp32, chunk 16, zero initial state."""
    return make_batch(B=1, T=64, Hk=2, Hv=2, dk=32, dv=32, dtype="f32", chunk=16, seed=seed)


def prefill_4k(seed=0) -> GDNBatch:
    """One sequence of 4096 tokens, Hk=16, Hv=32, dk=dv=128, bf16, chunk 64, zero state."""
    return make_batch(B=1, T=4096, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=seed)


def prefill_long(T=32768, seed=0) -> GDNBatch:
    """One sequence of T (32768 or 131072) tokens with a seeded N(0,0.02) initial state."""
    return make_batch(B=1, T=T, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=seed,
                      init_state=True)


def prefill_varlen(n=16, lo=256, hi=16384, seed=0) -> GDNBatch:
    """n packed sequences, lengths uniform in [lo, hi], each with its own initial state."""
    lengths = varlen_lengths(n, lo, hi, seed)
    return make_batch(Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=seed,
                      init_state=True, lengths=lengths)
