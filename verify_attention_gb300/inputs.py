"""Seeded synthetic inputs for the FP8 paged-KV path.

This module only draws random tensors and lays out pages; it holds none of the
method's arithmetic (no encoding, no attention).  Both the CUDA path and the CPU
oracle take their inputs from here.

Shapes follow the pages' model: 8 KV heads of dimension 128 ("Laguna S 2.1
KV-cache precision decision", section "BF16 versus FP8 in concrete terms"),
72 query heads (GQA group 9), 36 sliding-window-512 layers and 12 global
layers, page sizes 32 and 64 ("Laguna FP8 KV -- replicated embedding win,
page-32 build, and host boundary", section "Page-32 attention experiment").
Values are N(0,1) drawn in fp32 and rounded to bf16; the static per-tensor
scales are minmax/448, the "minmax", "tensor", "symmetric" kv_cache_scheme of
the KV-cache precision page, computed once from the generated tensors the way
an offline calibration would.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

HQ, HKV, HEAD_DIM = 72, 8, 128
E4M3_MAX = 448.0


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, gen, device="cpu", scale=None, outlier_frac=0.0, outlier_mult=8.0):
    """N(0,1) in fp32, optionally multiplied (per element) and with a fraction of
    outlier entries multiplied by ``outlier_mult``, then rounded to bf16."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if scale is not None:
        x = x * scale
    if outlier_frac > 0:
        hit = torch.rand(shape, generator=gen, dtype=torch.float32, device=device) < outlier_frac
        x = torch.where(hit, x * outlier_mult, x)
    return x.to(torch.bfloat16)


def minmax_scale(*tensors) -> float:
    """Static symmetric per-tensor scale: fp32(max |x|) / 448 in fp32."""
    amax = max(float(t.abs().max().float().item()) for t in tensors)
    return float(np.float32(amax) / np.float32(E4M3_MAX))


def minmax_scales_per_head(*tensors) -> torch.Tensor:
    """Static symmetric per-head scales of [T][Hkv][D] tensors: fp32(max |x| over
    head h) / 448 in fp32, one per KV head (float32 [Hkv], CPU)."""
    amax = torch.stack([t.abs().float().amax(dim=(0, 2)) for t in tensors]).amax(dim=0).cpu()
    return (amax.to(torch.float32) / torch.tensor(E4M3_MAX, dtype=torch.float32)).to(torch.float32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass
class PagedLayout:
    page_size: int
    num_pages: int
    block_table: torch.Tensor        # int32 [B][max_pages_per_seq], -1 = unused
    seq_lens: torch.Tensor           # int32 [B]

    @property
    def max_pages_per_seq(self) -> int:
        return self.block_table.shape[1]

    def slots(self, b: int, positions) -> torch.Tensor:
        """Cache slots (page * page_size + offset) of logical positions of seq b."""
        pos = torch.as_tensor(positions, dtype=torch.int64)
        pages = self.block_table[b].to(torch.int64)[pos // self.page_size]
        return pages * self.page_size + pos % self.page_size


def paged_layout(seq_lens: List[int], page_size: int, gen, extra_pages: int = 0,
                 max_pages_per_seq: Optional[int] = None) -> PagedLayout:
    """One shared pool of sum(ceil(L/ps)) (+extra) physical pages handed out in a
    seeded random order; unused block-table entries are -1."""
    need = [math.ceil(L / page_size) for L in seq_lens]
    total = sum(need) + extra_pages
    perm = torch.randperm(total, generator=gen).to(torch.int32)
    width = max_pages_per_seq or max(need)
    bt = torch.full((len(seq_lens), width), -1, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    return PagedLayout(page_size, total, bt, torch.tensor(seq_lens, dtype=torch.int32))


@dataclasses.dataclass
class LayerCase:
    """Everything one layer of insert + attention needs (CPU tensors)."""
    layout: PagedLayout
    M: int
    q: torch.Tensor                  # bf16 [B][M][Hq][D]
    k_prior: torch.Tensor            # bf16 [T_prior][Hkv][D]  context already cached
    v_prior: torch.Tensor
    slots_prior: torch.Tensor        # int64 [T_prior]
    k_new: torch.Tensor              # bf16 [B*M][Hkv][D]  the M new tokens per sequence
    v_new: torch.Tensor
    slots_new: torch.Tensor          # int64 [B*M]
    k_scale: float
    v_scale: float
    window_left: int                 # -1 = global
    sm_scale: float = 1.0 / math.sqrt(HEAD_DIM)
    k_scale_h: Optional[torch.Tensor] = None   # fp32 [Hkv] per-head minmax/448 scales of the whole K
    v_scale_h: Optional[torch.Tensor] = None

    @property
    def B(self):
        return self.q.shape[0]


def layer_case(seed: int, seq_lens: List[int], M: int, page_size: int, window: Optional[int] = None,
               Hq: int = HQ, Hkv: int = HKV, D: int = HEAD_DIM, k_head_scale=None,
               outlier_frac: float = 0.0, extra_pages: int = 0, device="cpu") -> LayerCase:
    """Synthetic layer: Q/K/V ~ N(0,1) bf16, new rows appended at the end of each
    sequence, a shuffled page pool, minmax/448 scales over the whole K (V) tensor.

    ``window`` is the window length W in keys including the query itself; the
    kernel argument is window_left = W - 1 (-1 for a global layer).
    ``k_head_scale``: (lo, hi) draws one U(lo, hi) multiplier per KV head for K.
    """
    g = generator(seed)
    layout = paged_layout(seq_lens, page_size, g, extra_pages=extra_pages)
    B = len(seq_lens)
    total = int(sum(seq_lens))
    hs = None
    if k_head_scale is not None:
        lo, hi = k_head_scale
        hs = (lo + (hi - lo) * torch.rand((Hkv,), generator=g)).view(1, Hkv, 1)
    gd = generator(seed * 7919 + 17, device) if device != "cpu" else g
    k_all = bf16_normal((total, Hkv, D), gd, device, scale=hs.to(device) if hs is not None else None,
                        outlier_frac=outlier_frac)
    v_all = bf16_normal((total, Hkv, D), gd, device, outlier_frac=outlier_frac)
    q = bf16_normal((B, M, Hq, D), gd, device)
    k_scale = minmax_scale(k_all)
    v_scale = minmax_scale(v_all)
    prior_idx, new_idx, slots_prior, slots_new = [], [], [], []
    start = 0
    for b, L in enumerate(seq_lens):
        prior_idx.append(torch.arange(start, start + L - M))
        new_idx.append(torch.arange(start + L - M, start + L))
        slots_prior.append(layout.slots(b, torch.arange(0, L - M)))
        slots_new.append(layout.slots(b, torch.arange(L - M, L)))
        start += L
    pi = torch.cat(prior_idx).to(k_all.device)
    ni = torch.cat(new_idx).to(k_all.device)
    return LayerCase(layout=layout, M=M, q=q, k_prior=k_all[pi], v_prior=v_all[pi],
                     slots_prior=torch.cat(slots_prior), k_new=k_all[ni], v_new=v_all[ni],
                     slots_new=torch.cat(slots_new), k_scale=k_scale, v_scale=v_scale,
                     window_left=(window - 1) if window else -1,
                     k_scale_h=minmax_scales_per_head(k_all), v_scale_h=minmax_scales_per_head(v_all))


# ------------------------------------------------------- fused-norm inputs

def rope_cos_sin(theta: float, max_pos: int, D: int = HEAD_DIM) -> torch.Tensor:
    """Rotary model constant handed to both sides as an input, like the norm
    weights: fp32 [max_pos][D] = cos of the D/2 frequencies theta^(-2k/D) at each
    position, then their sines, evaluated in float64 and rounded once."""
    k = np.arange(D // 2, dtype=np.float64)
    inv_freq = np.power(np.float64(theta), -2.0 * k / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return torch.from_numpy(table)


@dataclasses.dataclass
class FusedCase:
    q: torch.Tensor                  # bf16 [T][Hq][D]  (pre-norm)
    k: torch.Tensor                  # bf16 [T][Hkv][D] (pre-norm)
    v: torch.Tensor                  # bf16 [T][Hkv][D]
    positions: torch.Tensor          # int64 [T]
    q_norm_w: torch.Tensor           # bf16 [D]
    k_norm_w: torch.Tensor           # bf16 [D]
    cos_sin: torch.Tensor            # fp32 [max_pos][D]
    slots: torch.Tensor              # int64 [T]
    eps: float = 1e-6


def fused_case(seed: int, layout: PagedLayout, M: int, theta: float = 1e6, Hq: int = HQ,
               Hkv: int = HKV, D: int = HEAD_DIM, max_pos: Optional[int] = None) -> FusedCase:
    """The M new tokens of every sequence at their true offsets L-M .. L-1, with
    pre-norm Q/K/V ~ N(0,1) bf16 and norm weights ~ U(0.5, 1.5) bf16."""
    g = generator(seed)
    seq_lens = layout.seq_lens.tolist()
    B = len(seq_lens)
    T = B * M
    q = bf16_normal((T, Hq, D), g)
    k = bf16_normal((T, Hkv, D), g)
    v = bf16_normal((T, Hkv, D), g)
    qw = (0.5 + torch.rand((D,), generator=g)).to(torch.bfloat16)
    kw = (0.5 + torch.rand((D,), generator=g)).to(torch.bfloat16)
    pos = torch.cat([torch.arange(L - M, L) for L in seq_lens]).to(torch.int64)
    slots = torch.cat([layout.slots(b, torch.arange(L - M, L)) for b, L in enumerate(seq_lens)])
    mp = max_pos or int(max(seq_lens))
    return FusedCase(q, k, v, pos, qw, kw, rope_cos_sin(theta, mp, D), slots)


# ------------------------------------------------------------ the configs

CONFIGS = {
    1: "tiny single-layer global decode: B=1 M=1 L=256 ps=32",
    2: "single-layer verify: B=1 M=12 L=4096 ps=64, global and window 512",
    3: "48-layer verify step: [SW512 x3, G] x12, B=1 M=12 L=8192, ps 32|64",
    4: "long-context decode: 12 global layers, B=1 M=1 L=131072 ps=64, split 2048",
    5: "batched serving mix: B=64 L~U[1024,32768] M=12, 8 layers G/SW512, ps=32, fused norm+RoPE",
}


def cfg1_case(device="cpu") -> LayerCase:
    return layer_case(1001, [256], 1, 32, device=device)


def cfg2_case(window: Optional[int], device="cpu") -> LayerCase:
    return layer_case(1002, [4096], 12, 64, window=window, k_head_scale=(0.5, 2.0), device=device)


def cfg3_layer_kinds() -> List[Optional[int]]:
    """[SW, SW, SW, G] x 12: window 512 or None (global)."""
    return [512, 512, 512, None] * 12


def cfg3_case(layer: int, page_size: int, device="cpu") -> LayerCase:
    return layer_case(1003 * 100 + layer, [8192], 12, page_size,
                      window=cfg3_layer_kinds()[layer], device=device)


def cfg4_case(layer: int, device="cpu", seq_len: int = 131072, page_size: int = 64) -> LayerCase:
    return layer_case(1004 * 100 + layer, [seq_len], 1, page_size, outlier_frac=0.01, device=device)


def cfg5_seq_lens(B: int = 64) -> List[int]:
    g = generator(1005)
    return torch.randint(1024, 32768 + 1, (B,), generator=g).tolist()


def cfg5_layer_kinds() -> List[Optional[int]]:
    """G, SW, G, SW, ... over 8 layers."""
    return [None, 512] * 4


def cfg5_case(layer: int, device="cpu", seq_lens: Optional[List[int]] = None) -> LayerCase:
    lens = seq_lens or cfg5_seq_lens()
    return layer_case(1005 * 100 + layer, lens, 12, 32, window=cfg5_layer_kinds()[layer],
                      device=device)
