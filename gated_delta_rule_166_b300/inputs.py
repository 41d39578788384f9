"""Seeded synthetic inputs for the Gated Delta Rule-2 path.

This module draws inputs only; it holds none of the recurrence's arithmetic.
Tests, the bench and the smoke check all take their inputs from here, so the
CUDA library and the CPU oracle always see the same values (the oracle gets the
cast values upcast exactly to fp64).

Distributions (the workloads of the Gated DeltaNet-2 page's 1.3B model: 16
heads, d_k = d_v = 128, sequence 4K):

* q, k ~ N(0, 1), each (batch, token, head) row L2-normalised (the page's
  symbol table calls k a normalised key; q gets the same treatment).
* v ~ N(0, 1).
* b, w = sigmoid(N(0, 1)) per channel (b over key channels, w over value
  channels), or -- for the KDA-style "tied" mode -- one draw per (token, head)
  shared by b and w and broadcast over channels.
* log_decay = -softplus(N(0, 1) + shift) per key channel, or one draw per
  (token, head) broadcast over the key channels (Gated DeltaNet-style scalar
  decay).  Extra regimes exercise the inter-chunk carry: "slow"
  (-softplus(N - 4), about -0.018 per step), "zero" (D = I) and "mixed" (half
  the key channels fast, half slow).
* S0 ~ N(0, s0_std^2) in fp32, or None (zero initial state).

Draw order is fixed (q, k, v, b, w, log_decay, S0) on a CPU
``torch.Generator`` seeded with ``seed``; values are drawn in fp32, the rows
normalised, and then everything except S0 is cast to ``dtype``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.nn.functional as F


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    b: torch.Tensor
    w: torch.Tensor
    log_decay: torch.Tensor
    S0: torch.Tensor | None

    def tensors(self):
        return (self.q, self.k, self.v, self.b, self.w, self.log_decay)

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device, non_blocking=True)
        return PrefillInputs(*(mv(t) for t in self.tensors()), mv(self.S0))


def _normalise_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _decay(gen, shape, regime: str, shift: float) -> torch.Tensor:
    z = torch.randn(shape, generator=gen, device=gen.device)
    if regime == "fast":
        return -F.softplus(z + shift)
    if regime == "slow":
        return -F.softplus(z - 4.0)
    if regime == "zero":
        return torch.zeros(shape, device=gen.device)
    if regime == "mixed":
        fast = -F.softplus(z + shift)
        slow = -F.softplus(z - 4.0)
        half = shape[-1] // 2
        return torch.cat([fast[..., :half], slow[..., half:]], dim=-1)
    raise ValueError(f"unknown decay regime {regime!r}")


def make_prefill_inputs(B: int, T: int, H: int, dk: int, dv: int, *,
                        dtype=torch.bfloat16, seed: int = 0,
                        gates: str = "channel", decay: str = "channel",
                        decay_regime: str = "fast", decay_shift: float = 2.0,
                        s0_std: float | None = None,
                        b_scale: float = 1.0, device: str = "cpu") -> PrefillInputs:
    """Draw one prefill problem.

    gates: "channel" (b, w per channel) or "tied" (KDA: b = w = one scalar per
    token and head).  decay: "channel" or "scalar" (one value per token and
    head, broadcast over d_k).  b_scale multiplies b after the sigmoid (the
    page's ablation widens the erase range to [0, 2]).  device: where the
    seeded generator draws (the same distributions; a CUDA generator gives other
    values than the CPU one for the same seed, and is for inputs too large to
    draw on the host in time, such as the decode bench's 1024 token sets).
    """
    gen = torch.Generator(device=device).manual_seed(int(seed))
    rn = lambda *shape: torch.randn(*shape, generator=gen, device=device)  # noqa: E731
    q = _normalise_rows(rn(B, T, H, dk))
    k = _normalise_rows(rn(B, T, H, dk))
    v = rn(B, T, H, dv)
    if gates == "channel":
        b = torch.sigmoid(rn(B, T, H, dk))
        w = torch.sigmoid(rn(B, T, H, dv))
    elif gates == "tied":
        s = torch.sigmoid(rn(B, T, H, 1))
        b = s.expand(B, T, H, dk).contiguous()
        w = s.expand(B, T, H, dv).contiguous()
    else:
        raise ValueError(f"unknown gates mode {gates!r}")
    b = b * b_scale
    if decay == "channel":
        g = _decay(gen, (B, T, H, dk), decay_regime, decay_shift)
    elif decay == "scalar":
        g = _decay(gen, (B, T, H, 1), decay_regime, decay_shift).expand(B, T, H, dk).contiguous()
    else:
        raise ValueError(f"unknown decay mode {decay!r}")
    S0 = None
    if s0_std is not None:
        S0 = rn(B, H, dk, dv) * s0_std
    cast = lambda t: t.to(dtype).contiguous()
    return PrefillInputs(cast(q), cast(k), cast(v), cast(b), cast(w), cast(g), S0)


@dataclass
class SparseInputs:
    """One sparse-write problem: per (batch, token, head) the K selected slot
    indices and the key-side values at those slots; value-side tensors as in the
    dense case; the slot memory S0 [B, H, M, dv] (fp32)."""
    idx: torch.Tensor   # [B, T, H, K] int32
    q: torch.Tensor     # [B, T, H, K]
    k: torch.Tensor     # [B, T, H, K]
    v: torch.Tensor     # [B, T, H, dv]
    b: torch.Tensor     # [B, T, H, K]
    w: torch.Tensor     # [B, T, H, dv]
    log_decay: torch.Tensor   # [B, T, H, K]
    S0: torch.Tensor    # [B, H, M, dv] fp32

    @property
    def M(self) -> int:
        return int(self.S0.shape[2])

    def tensors(self):
        return (self.idx, self.q, self.k, self.v, self.b, self.w, self.log_decay)

    def to(self, device):
        return SparseInputs(*(t.to(device, non_blocking=True) for t in self.tensors()),
                            self.S0.to(device, non_blocking=True))


def make_sparse_inputs(B: int, T: int, H: int, M: int, K: int, dv: int, *,
                       dtype=torch.bfloat16, seed: int = 0, s0_std: float = 0.02,
                       decay_regime: str = "fast", decay_shift: float = 2.0) -> SparseInputs:
    """Draw one sparse gated-delta-write problem over a memory of M slots.

    Slot selection (a stand-in for a product-key router's top-K, which needs
    trained keys): per (batch, token, head) a uniform start r0 in [0, M) and K - 1
    gaps uniform in [1, G] with G = max(1, (M - 1) // K); the slots are r0 plus
    the running sums of the gaps, mod M.  The K slots of one token are therefore
    distinct, and consecutive tokens share slots about K^2 / M times.

    Values at the selected slots follow the dense distributions: q and k
    L2-normalised over the K entries, b = sigmoid(N), log_decay = -softplus(N +
    shift) (or the other regimes), and w, v as in the dense case.  The slot
    memory S0 ~ N(0, s0_std^2) stands for a learned initial memory.  Draw order:
    slot starts, gaps, q, k, v, b, w, log_decay, S0."""
    if K > M:
        raise ValueError("K must not exceed M")
    gen = torch.Generator().manual_seed(int(seed))
    r0 = torch.randint(0, max(M, 1), (B, T, H, 1), generator=gen)
    G = max(1, (M - 1) // max(K, 1))
    gaps = torch.randint(1, G + 1, (B, T, H, max(K - 1, 0)), generator=gen)
    offs = torch.cat([torch.zeros(B, T, H, 1, dtype=torch.long), torch.cumsum(gaps, dim=-1)], dim=-1)[..., :K]
    idx = ((r0 + offs) % max(M, 1)).to(torch.int32).contiguous()
    q = _normalise_rows(torch.randn(B, T, H, K, generator=gen))
    k = _normalise_rows(torch.randn(B, T, H, K, generator=gen))
    v = torch.randn(B, T, H, dv, generator=gen)
    b = torch.sigmoid(torch.randn(B, T, H, K, generator=gen))
    w = torch.sigmoid(torch.randn(B, T, H, dv, generator=gen))
    g = _decay(gen, (B, T, H, K), decay_regime, decay_shift)
    S0 = torch.randn(B, H, M, dv, generator=gen) * s0_std
    cast = lambda t: t.to(dtype).contiguous()
    return SparseInputs(idx, cast(q), cast(k), cast(v), cast(b), cast(w), cast(g), S0.contiguous())


def make_decode_state(B: int, H: int, dk: int, dv: int, *, seed: int,
                      std: float = 0.02) -> torch.Tensor:
    """fp32 decode state S ~ N(0, std^2), [B, H, dk, dv]."""
    gen = torch.Generator().manual_seed(int(seed))
    return torch.randn(B, H, dk, dv, generator=gen) * std


def make_decode_token(B: int, H: int, dk: int, dv: int, *, seed: int, step: int,
                      dtype=torch.bfloat16) -> PrefillInputs:
    """One decode token per (batch, head) for step ``step``: the prefill
    distributions with T = 1, drawn from a generator seeded by (seed, step).
    Token tensors are returned as [B, H, d] (no T axis); S0 is None."""
    x = make_prefill_inputs(B, 1, H, dk, dv, dtype=dtype,
                            seed=int(seed) * 1_000_003 + 7919 * int(step) + 1)
    sq = lambda t: t[:, 0].contiguous()
    return PrefillInputs(*(sq(t) for t in x.tensors()), None)


# The workloads, by name.  Seeds: tiny case 0; the others 1..5.
WORKLOADS = {
    # fp32 tiny case the oracle finishes instantly
    "tiny_f32": dict(B=1, T=256, H=2, dk=32, dv=32, dtype=torch.float32, seed=0),
    # one GDN-2 1.3B layer: 16 heads, d=128, 4K tokens, batch 4
    "gdn2_layer_T4096": dict(B=4, T=4096, H=16, dk=128, dv=128, dtype=torch.bfloat16, seed=1),
    # long-context prefill with a learned-style initial state
    "long_T65536": dict(B=1, T=65536, H=16, dk=128, dv=128, dtype=torch.bfloat16, seed=2,
                        decay_shift=4.0, s0_std=0.02),
    # KDA: b = w = one scalar per token and head, channel-wise decay
    "kda_T2048": dict(B=8, T=2048, H=16, dk=128, dv=128, dtype=torch.bfloat16, seed=3,
                      gates="tied"),
    # Gated DeltaNet: tied scalar gates and a scalar decay per token and head
    "gdn_T2048": dict(B=8, T=2048, H=16, dk=128, dv=128, dtype=torch.bfloat16, seed=4,
                      gates="tied", decay="scalar"),
}

# Autoregressive decode: 256 sequences, 16 heads, d = 128, fp32 state
DECODE_WORKLOAD = dict(B=256, H=16, dk=128, dv=128, seed=5, steps=1024, state_std=0.02)


def make_workload(name: str, **overrides) -> PrefillInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return make_prefill_inputs(**cfg)


# Sparse gated delta write over a slot memory: 2048 slots per head, 32 selected
# per token, d_v = 128, 16 heads, 4K tokens, batch 4 (memory 16x the dense
# d_k = 128 state; per-token work 1/4 of the dense update's)
SPARSE_WORKLOAD = dict(B=4, T=4096, H=16, M=2048, K=32, dv=128, dtype=torch.bfloat16, seed=6, s0_std=0.02)


def make_sparse_workload(**overrides) -> SparseInputs:
    cfg = dict(SPARSE_WORKLOAD)
    cfg.update(overrides)
    return make_sparse_inputs(**cfg)
