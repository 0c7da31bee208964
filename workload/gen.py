"""Seeded generators for the synthetic routed-MoE workloads.

Shapes follow the Gemma-4-26B-A4B-like configuration the TurboFieldfare
write-up streams (section "MoE needed parallel work, reuse, and coarse
overlap"; 128 experts per layer, top-8, one always-on shared expert, INT4
affine groups of 64 per section "Vectorization helped when it respected the
storage layout").

Canonical storage layout produced here (what a caller of the library holds):

* every projection is row-major ``[out][in]``;
* int4 values are unsigned 0..15, two per byte: byte ``m`` of a row holds
  element ``2m`` in its low nibble and ``2m+1`` in its high nibble;
* each run of ``group`` consecutive *input* elements of a row shares one fp16
  ``(scale, bias)`` pair, stored as ``sb[row][group_index][2]``;
* weight value = scale * q + bias.

The quantiser below (min/max affine per group) only encodes random weights
into that format; the method itself only ever decodes it.
"""

from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Shape:
    d: int            # hidden size
    f: int            # routed-expert intermediate size
    f_shared: int     # shared-expert intermediate size
    n_experts: int    # E
    top_k: int        # k
    group: int = 64   # int4 affine group length along the input dimension
    n_layers: int = 1

    def expert_bytes(self, f: int | None = None) -> int:
        f = self.f if f is None else f
        q = 3 * f * self.d // 2
        sb = (2 * f * (self.d // self.group) + self.d * (f // self.group)) * 4
        return q + sb


# Tiny single layer: d=256, f=128, E=8, top-2, shared f=128.
TINY = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2, group=64, n_layers=1)
# Full-shape layer: d=2816, f=704, E=128, top-8, shared f=2816, 30 layers.
FULL = Shape(d=2816, f=704, f_shared=2816, n_experts=128, top_k=8, group=64, n_layers=30)


def derive_seed(*parts) -> int:
    """Stable 63-bit seed from any tuple of ints/strings."""
    h = hashlib.sha256(repr(tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def quantise_rows(w: torch.Tensor, group: int):
    """Encode float rows ``w[..., rows, cols]`` as int4 affine groups.

    scale = fp16((max - min) / 15), bias = fp16(min),
    q = clamp(round_half_even((w - bias) / scale), 0, 15), q = 0 where scale == 0.
    Returns (packed uint8 [..., rows, cols/2], sb fp16 [..., rows, cols/group, 2]).
    """
    *lead, rows, cols = w.shape
    assert cols % group == 0 and cols % 2 == 0
    wg = w.reshape(*lead, rows, cols // group, group).float()
    mn = wg.amin(-1)
    mx = wg.amax(-1)
    s16 = ((mx - mn) / 15.0).to(torch.float16)
    b16 = mn.to(torch.float16)
    s = s16.float().unsqueeze(-1)
    b = b16.float().unsqueeze(-1)
    safe = torch.where(s > 0, s, torch.ones_like(s))
    q = torch.round((wg - b) / safe)
    q = torch.where(s > 0, q, torch.zeros_like(q)).clamp_(0, 15).to(torch.uint8)
    q = q.reshape(*lead, rows, cols)
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).contiguous()
    sb = torch.stack([s16, b16], dim=-1).contiguous()
    return packed, sb


def _gen_proj(lead, rows, cols, group, seed, device, std=0.02):
    g = _gen(seed, device)
    w = torch.randn(*lead, rows, cols, generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    out = quantise_rows(w, group)
    del w
    return out


def _gen_ffn(shape: Shape, lead, f: int, seed: int, layer: int, tag: str, device):
    d, grp = shape.d, shape.group
    gq, gsb = _gen_proj(lead, f, d, grp, derive_seed(seed, layer, tag, "gate"), device)
    uq, usb = _gen_proj(lead, f, d, grp, derive_seed(seed, layer, tag, "up"), device)
    dq, dsb = _gen_proj(lead, d, f, grp, derive_seed(seed, layer, tag, "down"), device)
    return {"gate_q": gq, "gate_sb": gsb, "up_q": uq, "up_sb": usb,
            "down_q": dq, "down_sb": dsb}


def gen_layer(shape: Shape, seed: int, layer: int, device="cpu", chunk: int = 16):
    """All weights of one MoE layer in canonical layout.

    Returns ``{"router_w": fp16 [E, d], "experts": {...stacked over E...},
    "shared": {...}}``; weights are N(0, 0.02) before int4 quantisation and
    the router is fp16 N(0, 0.02).  Experts are drawn in chunks of ``chunk``
    experts to bound temporary memory; each chunk has its own seed.
    """
    E = shape.n_experts
    g = _gen(derive_seed(seed, layer, "router"), device)
    router = (torch.randn(E, shape.d, generator=g, device=device) * 0.02).to(torch.float16)
    parts = []
    for c0 in range(0, E, chunk):
        n = min(chunk, E - c0)
        parts.append(_gen_ffn(shape, (n,), shape.f, seed, layer, ("experts", c0), device))
    experts = {k: torch.cat([p[k] for p in parts], 0) for k in parts[0]}
    shared = _gen_ffn(shape, (), shape.f_shared, seed, layer, "shared", device)
    return {"router_w": router, "experts": experts, "shared": shared}


def gen_hidden(n_tokens: int, d: int, seed: int, device="cpu", tag="hidden"):
    """bf16 N(0, 1) hidden states [n_tokens, d]."""
    g = _gen(derive_seed(seed, tag), device)
    return torch.randn(n_tokens, d, generator=g, device=device).to(torch.bfloat16)


def _zipf_probs(E: int, s: float) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    return p / p.sum()


def zipf_reuse_targets(n_tokens: int, n_layers: int, E: int, k: int, seed: int,
                       s: float = 1.1, p_reuse: float = 0.6) -> np.ndarray:
    """Expert targets [T, L, k] int32 for the slot-cache workload.

    Per layer a seeded permutation maps Zipf(s) ranks to experts.  For token 0
    every position draws fresh; afterwards position j reuses the previous
    token's expert at j with probability ``p_reuse``, else draws fresh;
    duplicates within a token are redrawn.
    """
    out = np.zeros((n_tokens, n_layers, k), dtype=np.int32)
    probs = _zipf_probs(E, s)
    for layer in range(n_layers):
        rng = np.random.Generator(np.random.Philox(derive_seed(seed, layer, "zipf-trace")))
        perm = rng.permutation(E)
        prev = None
        for t in range(n_tokens):
            chosen: list[int] = []
            for j in range(k):
                cand = -1
                if prev is not None and rng.random() < p_reuse:
                    cand = int(prev[j])
                while cand < 0 or cand in chosen:
                    cand = int(perm[rng.choice(E, p=probs)])
                chosen.append(cand)
            out[t, layer] = chosen
            prev = chosen
    return out


def mixture_targets(n_tokens: int, n_layers: int, E: int, k: int, seed: int,
                    s: float = 0.8) -> np.ndarray:
    """Expert targets [T, L, k]: k distinct draws per token, each from a 50/50
    mixture of uniform and Zipf(s) over a per-layer permutation."""
    out = np.zeros((n_tokens, n_layers, k), dtype=np.int32)
    probs = _zipf_probs(E, s)
    for layer in range(n_layers):
        rng = np.random.Generator(np.random.Philox(derive_seed(seed, layer, "mixture-trace")))
        perm = rng.permutation(E)
        coin = rng.random((n_tokens, 4 * k)) < 0.5
        uni = rng.integers(0, E, size=(n_tokens, 4 * k))
        zr = perm[rng.choice(E, size=(n_tokens, 4 * k), p=probs)]
        draws = np.where(coin, uni, zr)
        for t in range(n_tokens):
            chosen: list[int] = []
            for v in draws[t]:
                if int(v) not in chosen:
                    chosen.append(int(v))
                    if len(chosen) == k:
                        break
            while len(chosen) < k:
                v = int(rng.integers(0, E))
                if v not in chosen:
                    chosen.append(v)
            out[t, layer] = chosen
    return out


def bias_from_targets(targets: np.ndarray, E: int, value: float = 16.0) -> np.ndarray:
    """Logit bias [T, L, E] float32: ``value`` on each target expert, 0 elsewhere."""
    T, L, k = targets.shape
    bias = np.zeros((T, L, E), dtype=np.float32)
    ti = np.arange(T)[:, None, None]
    li = np.arange(L)[None, :, None]
    bias[ti, li, targets] = value
    return bias
