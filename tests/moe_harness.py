"""Shared test harness: build a libmoe context from generated weights, run it
through the C ABI, and compare against the CPU oracle."""

from __future__ import annotations

import numpy as np
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import Shape

# FFN tolerance: max|y_gpu - y_ref| <= 2e-3 * max|y_ref| (fp32 accumulation).
FFN_RTOL = 2e-3
GATE_RTOL = 1e-5


def bf16_to_f64(t) -> np.ndarray:
    b = oracle.as_bits(t).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_device(layer: dict, device="cuda") -> dict:
    out = {"router_w": layer["router_w"].to(device).contiguous()}
    for key in ("experts", "shared"):
        out[key] = {k: v.to(device).contiguous() for k, v in layer[key].items()}
    return out


def to_host(layer: dict) -> dict:
    out = {"router_w": layer["router_w"].cpu().contiguous()}
    for key in ("experts", "shared"):
        out[key] = {k: v.cpu().contiguous() for k, v in layer[key].items()}
    return out


class Ctx:
    """Owns one libmoe context."""

    def __init__(self, shape: Shape, n_layers=None, prenorm=0, max_tokens=32, gelu=0, eps=1e-6, device=0):
        self.shape = shape
        self.n_layers = n_layers or shape.n_layers
        self.cfg = moe.make_config(shape.d, shape.f, shape.f_shared, shape.n_experts, shape.top_k,
                                   n_layers=self.n_layers, gelu_variant=gelu, prenorm=prenorm,
                                   max_tokens=max_tokens, norm_eps=eps)
        st, self.h = moe.moe_create(self.cfg, device)
        if st != moe.MOE_OK:
            raise moe.MoeError(st, moe.moe_last_error(None))

    def init_layer(self, layer: int, weights: dict, residency=moe.MOE_RESIDENT_HBM):
        moe.check(moe.moe_init_layer(self.h, layer, weights["router_w"], weights["experts"], weights["shared"],
                                     residency), self.h)

    def decode(self, h_in, l0=0, l1=None, bias=None, trace=None, stream=None):
        l1 = self.n_layers if l1 is None else l1
        B = h_in.shape[0]
        h_out = torch.empty_like(h_in)
        y = torch.empty(B, self.shape.d, dtype=torch.float32, device=h_in.device)
        st, n = moe.moe_decode_step(self.h, h_in, B, l0, l1, bias, h_out, y, trace, stream)
        moe.check(st, self.h)
        return h_out, y, n

    def sync(self):
        moe.check(moe.moe_sync(self.h), self.h)

    def close(self):
        if self.h is not None:
            moe.moe_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


# B = 1 decode kernels a test can pin: the clustered persistent kernel, the
# per-SM persistent kernel, or the per-layer kernels.
DECODE_KERNELS = ("cluster", "per_sm", "layers")


def use_decode_kernel(ctx: "Ctx", which: str) -> None:
    if which == "layers":
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PERSISTENT, 0), ctx.h)
        return
    moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PERSISTENT, 1), ctx.h)
    moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_CLUSTER, 1 if which == "cluster" else 0), ctx.h)


def assert_ffn_close(y_gpu, y_ref, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    err = np.abs(y_gpu - y_ref).max()
    bound = FFN_RTOL * np.abs(y_ref).max()
    assert err <= bound, f"{what}: max err {err:.3e} > {bound:.3e}"
    return err / max(np.abs(y_ref).max(), 1e-30)
