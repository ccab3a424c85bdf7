"""Seeded synthetic inputs for the chunked KDA forward.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the method's arithmetic: it only draws random tensors with the
shapes, dtypes and value distributions of the workloads below and casts them.
Both the GPU path and the fp64 oracle receive the *same* cast values.

Recipe (one ``torch.Generator`` on the CPU, ``manual_seed(seed)``; fp32
``randn`` drawn in this fixed order):

1. q  [B,T,H,K] ~ N(0,1), then L2-normalised per (token, head) in fp32
   (exact x / ||x||), then cast to the q/k/v dtype;
2. k  [B,T,H,K] likewise;
3. v  [B,T,H,V] ~ N(0,1), cast;
4. beta-logits [B,T,H] ~ N(0,1);  beta = sigmoid(.) in fp32;
5. g-raw [B,T,H,K] ~ N(0,1);  g = max(logsigmoid(.), -5) in fp32 (log-decay);
6. initial_state [B,H,K,V] ~ N(0, std) fp32, only when the workload has one;
7. conv weights [3, H*K, 4] ~ N(0, 0.5) fp32, only when the workload runs the
   short-conv prologue.  Then steps 1-3 draw the *pre-conv* inputs x_q, x_k,
   x_v ~ N(0,1) instead (no L2 normalisation; the prologue normalises q, k).

The shapes are those of the pages' representative KDA specs: B=1, H=8,
T=1024 with four non-64-aligned segments (page "Add packed KDA forward
megakernel", section "TPU performance versus openxla/tokamax"), and B=1, H=32,
T=8192, K=V=128 fixed and packed with 25 balanced segments (same page,
section "2026-09-29 representative-shape forward A/B").  No dataset is used.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch
import torch.nn.functional as F

__all__ = ["Workload", "WORKLOADS", "make_inputs", "segment_ids_from_lengths",
           "custom_workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str = "bf16"                 # dtype of q, k, v and o ("bf16"/"f32")
    init_state_std: Optional[float] = None   # None: zero initial state
    segments: Optional[tuple] = None    # run lengths per row (ids 1..n)
    prologue: bool = False              # draw pre-conv x and conv weights
    output_final_state: bool = True

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H


WORKLOADS = {
    "tiny_fp32_h2_t128_d32": Workload(
        "tiny_fp32_h2_t128_d32", B=1, T=128, H=2, K=32, V=32, dtype="f32"),
    "fixed_bf16_h8_t1024": Workload(
        "fixed_bf16_h8_t1024", B=1, T=1024, H=8, K=128, V=128),
    "packed_bf16_h8_t1024_4seg": Workload(
        "packed_bf16_h8_t1024_4seg", B=1, T=1024, H=8, K=128, V=128,
        segments=(197, 301, 259, 267)),
    "fixed_bf16_h32_t8192": Workload(
        "fixed_bf16_h32_t8192", B=1, T=8192, H=32, K=128, V=128,
        init_state_std=0.1),
    "packed_bf16_h32_t8192_25seg": Workload(
        "packed_bf16_h32_t8192_25seg", B=1, T=8192, H=32, K=128, V=128,
        segments=tuple([328] * 17 + [327] * 8)),
    "packed_bf16_h32_t8192_25seg_conv": Workload(
        "packed_bf16_h32_t8192_25seg_conv", B=1, T=8192, H=32, K=128, V=128,
        segments=tuple([328] * 17 + [327] * 8), prologue=True),
    # not one of the pages' workloads: a long context with few heads (the
    # same token-heads as B1 H32 T8192), where one state chain per
    # (row, head, value tile) leaves most SMs idle; timed for the
    # chunk-parallel state scan
    "fixed_bf16_h8_t32768": Workload(
        "fixed_bf16_h8_t32768", B=1, T=32768, H=8, K=128, V=128,
        init_state_std=0.1),
    # not one of the pages' workloads: the B1 H32 T8192 shape at a quarter of
    # the tokens, the size the detailed (many-pass) profiles are taken on
    "fixed_bf16_h32_t2048": Workload(
        "fixed_bf16_h32_t2048", B=1, T=2048, H=32, K=128, V=128,
        init_state_std=0.1),
}


def _freeze(x):
    if isinstance(x, (list, tuple)):
        return tuple(_freeze(y) for y in x)
    return x


def custom_workload(B, T, H, K, V, dtype="bf16", init_state_std=None,
                    segments=None, prologue=False, name="custom"):
    return Workload(name, B, T, H, K, V, dtype, init_state_std,
                    _freeze(segments) if segments is not None else None,
                    prologue)


def _is_item(x) -> bool:
    return isinstance(x, int) or (isinstance(x, tuple) and len(x) == 2
                                  and x[0] == "pad")


def segment_ids_from_lengths(B: int, T: int, segments) -> torch.Tensor:
    """1-based ids [B,T] int32 from run lengths.

    ``segments`` is either one sequence of items (used for every row) or one
    sequence per row.  An item is a run length n (the next id, n tokens) or
    ``("pad", n)`` (n padding tokens, id 0).  Tokens after the listed items
    are padding.
    """
    segments = _freeze(segments)
    rows = [segments] * B if all(_is_item(x) for x in segments) else \
        list(segments)
    assert len(rows) == B
    seg = torch.zeros(B, T, dtype=torch.int32)
    for b, items in enumerate(rows):
        t = 0
        sid = 0
        for item in items:
            if isinstance(item, tuple):
                t += int(item[1])
                continue
            sid += 1
            assert t + item <= T, "segments longer than T"
            seg[b, t:t + item] = sid
            t += item
    return seg


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def _l2(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw the workload's inputs on the CPU (see the module docstring)."""
    gen = torch.Generator().manual_seed(seed)
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = randn(B, T, H, K)
    k = randn(B, T, H, K)
    v = randn(B, T, H, V)
    if not w.prologue:
        q, k = _l2(q), _l2(k)
    beta = torch.sigmoid(randn(B, T, H))
    g = torch.clamp(F.logsigmoid(randn(B, T, H, K)), min=-5.0)
    S0 = None
    if w.init_state_std is not None:
        S0 = randn(B, H, K, V) * float(w.init_state_std)
    conv_w = None
    if w.prologue:
        assert K == V, "the prologue's weight layout assumes K == V"
        conv_w = randn(3, H * K, 4) * 0.5
    seg = None
    if w.segments is not None:
        seg = segment_ids_from_lengths(B, T, w.segments)
    out = dict(q=_cast(q, w.dtype).contiguous(), k=_cast(k, w.dtype).contiguous(),
               v=_cast(v, w.dtype).contiguous(), g=g.contiguous(),
               beta=beta.contiguous(), initial_state=S0, segment_ids=seg,
               conv_w=conv_w, scale=K ** -0.5)
    return out


def make_upstream_grads(w: Workload, seed: int = 0) -> dict:
    """Upstream gradients for the backward: d_o [B,T,H,V] ~ N(0,1) in the
    workload's q/k/v dtype and d_final [B,H,K,V] ~ N(0,1) fp32, drawn on the
    CPU from their own seeded generator."""
    gen = torch.Generator().manual_seed(10_000 + seed)
    d_o = torch.randn(w.B, w.T, w.H, w.V, generator=gen, dtype=torch.float32)
    d_final = torch.randn(w.B, w.H, w.K, w.V, generator=gen, dtype=torch.float32)
    return dict(d_o=_cast(d_o, w.dtype).contiguous(), d_final=d_final.contiguous())
