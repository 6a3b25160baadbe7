"""Seeded input generators for the decode and prefill workloads.

Shapes follow the static-KV-cache decode of "MiniCPM4 `forward_step` Attention
Performance Fix" (section 2.2: cache ``(batch, 8, 8192, 128)``; section 4.1:
one new row per KV head written at ``position_id``) and the prefill of
"step14_3 -- batched attention" (``Q [seq_len, H, d_head]``, ``K_full``/``V_full``
``[total_len, H, d_head]``).

Everything here draws numbers; nothing here computes attention.  Values are
drawn N(0,1) in fp32 from a seeded ``torch.Generator`` and rounded to bf16
(round-to-nearest-even, done by ``Tensor.to``).  The same seed on the same
device gives the same tensors, so a test can regenerate inputs for the oracle
instead of copying them from a kernel's output.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# Named workloads.  Sizes are the ones the decode/prefill pages use: Hkv=8,
# D=128, max_len=8192 for decode; 32 heads of d_head=64 for prefill.
WORKLOADS = {
    # one decode step: rows 0..99 filled, the new row lands at position 100
    "single_step": dict(kind="decode", B=1, Hq=16, Hkv=8, D=128, L=8192,
                        positions="fixed:100", fill="prefix"),
    # 8192 consecutive append+decode steps from position 0
    "streaming": dict(kind="stream", B=1, Hq=16, Hkv=8, D=128, L=8192,
                      steps=8192),
    # B=64 sequences at positions uniform in [0, 8191]
    "ragged": dict(kind="decode", B=64, Hq=32, Hkv=8, D=128, L=8192,
                   positions="uniform", fill="all"),
    # causal prefill of 512 new tokens over a 2048-token cached prefix
    "prefill_prefix": dict(kind="prefill", S=512, start_pos=2048, Hq=32,
                           Hkv=32, d=64),
    # causal prefill from scratch, 2048 tokens
    "prefill": dict(kind="prefill", S=2048, start_pos=0, Hq=32, Hkv=32, d=64),
    # prompt chunks at the decode shapes (GQA, D=128): 512 tokens over a
    # 2048-token cache, and 2048 tokens from scratch
    "prefill_d128_chunk": dict(kind="prefill", S=512, start_pos=2048, Hq=32,
                               Hkv=8, d=128),
    "prefill_d128": dict(kind="prefill", S=2048, start_pos=0, Hq=32, Hkv=8, d=128),
    # B=256, g=8, every sequence at the last position, 1% of key rows x8
    "stress": dict(kind="decode", B=256, Hq=64, Hkv=8, D=128, L=8192,
                   positions="fixed:8191", fill="all", peaky=0.01),
}


def bf16_from_f32(x: torch.Tensor) -> torch.Tensor:
    """Round an fp32 tensor to bf16 (round-to-nearest-even)."""
    return x.to(torch.bfloat16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g, device, chunk_rows: int = 1 << 22) -> torch.Tensor:
    """N(0,1) fp32 -> bf16, drawn in slices along dim 0 to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    per = max(1, chunk_rows // max(1, flat.shape[1]))
    for i in range(0, flat.shape[0], per):
        j = min(flat.shape[0], i + per)
        flat[i:j] = torch.randn((j - i, flat.shape[1]), generator=g,
                                device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


@dataclasses.dataclass
class DecodeCase:
    """One decode step's inputs.

    ``k_cache``/``v_cache`` hold the cache *before* this step's append; the new
    rows ``k_new``/``v_new`` belong at ``positions[b]``.  ``key_scale_mask``
    (if any) marks the (b, kvh, row) key rows that were multiplied by 8,
    including row ``positions[b]`` whose value is carried by ``k_new``.
    """

    q: torch.Tensor          # [B, Hq, D] bf16
    k_new: torch.Tensor      # [B, Hkv, D] bf16
    v_new: torch.Tensor      # [B, Hkv, D] bf16
    k_cache: torch.Tensor    # [B, Hkv, L, D] bf16
    v_cache: torch.Tensor    # [B, Hkv, L, D] bf16
    positions: torch.Tensor  # [B] int32
    scale: float
    name: str = ""

    @property
    def shape(self):
        B, Hq, D = self.q.shape
        return dict(B=B, Hq=Hq, Hkv=self.k_cache.shape[1],
                    L=self.k_cache.shape[2], D=D)


@dataclasses.dataclass
class PrefillCase:
    q: torch.Tensor   # [S, Hq, d] bf16
    k: torch.Tensor   # [start_pos + S, Hkv, d] bf16
    v: torch.Tensor   # [start_pos + S, Hkv, d] bf16
    start_pos: int
    scale: float
    name: str = ""


def _positions(spec, B, L, g, device):
    if isinstance(spec, (list, tuple)):
        return torch.tensor(list(spec), dtype=torch.int32, device=device)
    if isinstance(spec, torch.Tensor):
        return spec.to(device=device, dtype=torch.int32)
    if spec.startswith("fixed:"):
        return torch.full((B,), int(spec.split(":")[1]), dtype=torch.int32,
                          device=device)
    if spec == "uniform":
        return torch.randint(0, L, (B,), generator=g, device=device,
                             dtype=torch.int64).to(torch.int32)
    raise ValueError(f"unknown positions spec {spec!r}")


def decode_case(B=1, Hq=16, Hkv=8, D=128, L=8192, positions="fixed:100",
                fill="prefix", peaky: float = 0.0, poison: bool = False,
                seed: int = 0, device="cpu", name: str = "",
                scale: Optional[float] = None) -> DecodeCase:
    """Draw one decode step.

    fill="prefix": cache rows < positions[b] are N(0,1), the rest zero (the
    zero-initialised static cache of the decode page).  fill="all": every row
    of the cache is N(0,1).  poison=True overwrites rows > positions[b] with
    NaN, so any read past the attended range shows up in the output.
    peaky>0: each (b, kvh, row) key row is multiplied by 8 with that
    probability (exact in bf16).
    """
    g = _gen(seed, device)
    pos = _positions(positions, B, L, g, device)
    q = _randn_bf16((B, Hq, D), g, device)
    k_new = _randn_bf16((B, Hkv, D), g, device)
    v_new = _randn_bf16((B, Hkv, D), g, device)
    k_cache = _randn_bf16((B, Hkv, L, D), g, device)
    v_cache = _randn_bf16((B, Hkv, L, D), g, device)
    rows = torch.arange(L, device=device, dtype=torch.int32).view(1, 1, L)
    p = pos.view(B, 1, 1)
    if peaky > 0:
        sel = torch.rand((B, Hkv, L), generator=g, device=device) < peaky
        k_cache.mul_(torch.where(sel, 8.0, 1.0).to(torch.bfloat16).unsqueeze(-1))
        at_pos = sel.gather(2, pos.long().clamp(0, L - 1).view(B, 1, 1).expand(B, Hkv, 1)).squeeze(-1)
        k_new.mul_(torch.where(at_pos, 8.0, 1.0).to(torch.bfloat16).unsqueeze(-1))
    if fill == "prefix":
        keep = (rows < p).unsqueeze(-1)
        k_cache.mul_(keep)
        v_cache.mul_(keep)
    elif fill != "all":
        raise ValueError(fill)
    if poison:
        bad = (rows > p).unsqueeze(-1).expand_as(k_cache)
        k_cache.masked_fill_(bad, float("nan"))
        v_cache.masked_fill_(bad, float("nan"))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return DecodeCase(q, k_new, v_new, k_cache, v_cache, pos, float(scale), name)


def prefill_case(S=512, start_pos=2048, Hq=32, Hkv=32, d=64, seed: int = 0,
                 device="cpu", name: str = "",
                 scale: Optional[float] = None) -> PrefillCase:
    g = _gen(seed, device)
    T = start_pos + S
    q = _randn_bf16((S, Hq, d), g, device) if S > 0 else torch.empty((0, Hq, d), dtype=torch.bfloat16, device=device)
    k = _randn_bf16((T, Hkv, d), g, device) if T > 0 else torch.empty((0, Hkv, d), dtype=torch.bfloat16, device=device)
    v = _randn_bf16((T, Hkv, d), g, device) if T > 0 else torch.empty((0, Hkv, d), dtype=torch.bfloat16, device=device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return PrefillCase(q, k, v, int(start_pos), float(scale), name)


def streaming_inputs(steps=8192, B=1, Hq=16, Hkv=8, D=128, seed: int = 0,
                     device="cpu"):
    """Per-step new rows for the streaming loop: q [steps,B,Hq,D], k/v
    [steps,B,Hkv,D] and positions [steps,B] (step s writes/attends position s)."""
    g = _gen(seed, device)
    q = _randn_bf16((steps, B, Hq, D), g, device)
    k = _randn_bf16((steps, B, Hkv, D), g, device)
    v = _randn_bf16((steps, B, Hkv, D), g, device)
    pos = torch.arange(steps, dtype=torch.int32, device=device).view(steps, 1).expand(steps, B).contiguous()
    return q, k, v, pos


def rope_tables(positions, D: int = 128, base: float = 10000.0, device="cpu"):
    """cos/sin tables [B, D] float32 for the rotary embedding at each
    sequence's position: the usual frequencies base**(-2i/D), i < D/2, each
    repeated for both halves of the row.  Angles and their cos/sin are taken in
    float64 and rounded once to float32; they are inputs to the rotation (the
    model's table), not part of it."""
    pos = torch.as_tensor(positions).to(device="cpu", dtype=torch.float64).view(-1, 1)
    inv = base ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    ang = pos * inv.view(1, -1)
    ang = torch.cat([ang, ang], dim=1)
    return (torch.cos(ang).to(torch.float32).to(device).contiguous(),
            torch.sin(ang).to(torch.float32).to(device).contiguous())


def workload_case(name: str, seed: int = 0, device="cpu", poison=False):
    """The named workload's inputs (decode or prefill)."""
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    if kind == "decode":
        return decode_case(seed=seed, device=device, poison=poison, name=name, **w)
    if kind == "prefill":
        return prefill_case(seed=seed, device=device, name=name, **w)
    raise ValueError(f"{name} is a {kind} workload")
