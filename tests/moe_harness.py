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


INT64_MIN = np.iinfo(np.int64).min


def check_logits(got, ref, ids, what="", candidates_only=False):
    """Router logits (int64, 2^-40 units, bias included) bit for bit.  With
    candidates_only (the prefill router), experts its error bound ruled out read
    INT64_MIN; every other entry and every picked expert must be exact."""
    got = np.asarray(got, dtype=np.int64)
    ref = np.asarray(ref, dtype=np.int64)
    live = got != INT64_MIN if candidates_only else np.ones(got.shape, bool)
    assert live[np.asarray(ids)].all(), f"{what}: a picked expert has no exact logit"
    bad = np.nonzero(live & (got != ref))[0]
    assert bad.size == 0, f"{what}: logits differ at experts {bad[:8].tolist()}: {got[bad[:4]]} vs {ref[bad[:4]]}"
    if candidates_only:
        # a ruled-out expert must be strictly below the k-th largest logit
        kth = np.sort(ref)[::-1][len(ids) - 1]
        assert np.all(ref[~live] < kth), f"{what}: the bound ruled out an expert tied with the top-k"


def capture(ctx, L, B, logits=False):
    """Device buffers for the debug capture of the next call(s) over L layers, B tokens."""
    d, k, E = ctx.shape.d, ctx.shape.top_k, ctx.shape.n_experts
    cap = {"x": torch.zeros(L, B, d, dtype=torch.bfloat16, device="cuda"),
           "ids": torch.zeros(L, B, k, dtype=torch.int32, device="cuda"),
           "gates": torch.zeros(L, B, k, dtype=torch.float32, device="cuda"),
           "y": torch.zeros(L, B, d, dtype=torch.float32, device="cuda")}
    moe.check(moe.moe_set_debug(ctx.h, cap["x"], cap["ids"], cap["gates"], cap["y"], L), ctx.h)
    if logits:
        cap["logits"] = torch.full((L, B, E), 7, dtype=torch.int64, device="cuda")
        moe.check(moe.moe_set_debug_logits(ctx.h, cap["logits"]), ctx.h)
    return cap


def end_capture(ctx):
    moe.check(moe.moe_set_debug_logits(ctx.h), ctx.h)
    moe.check(moe.moe_set_debug(ctx.h), ctx.h)


def check_stack(weights, H, cap, h_out, top_k, ffn_layers=(), ffn_tokens=None, bias=None, prenorm=1,
                candidates_only=False, eps=1e-6):
    """Teacher-forced oracle check of a captured stack of L layers for every
    token of H [B, d]: x_l within one bf16 ulp of RMSNorm(h_l) (or equal to h_l
    without the norm), ids bit-exact, gates within GATE_RTOL, logits bit-exact
    (if captured), y_l against oracle.Layer on ffn_layers (tokens ffn_tokens,
    default all), and h_{l+1} = bf16(h_l + y_l) within one ulp, chained on the
    kernels' fp32 rule.  weights[l] holds at least router_w; full host weights
    on the FFN layers.  bias: [L, B, E] or None."""
    xs, ids, gs, ys = (cap[n].cpu() for n in ("x", "ids", "gates", "y"))
    lgs = cap["logits"].cpu().numpy() if "logits" in cap else None
    L, B = ids.shape[0], ids.shape[1]
    bias_np = None if bias is None else bias.cpu().numpy()
    ffn_tokens = range(B) if ffn_tokens is None else ffn_tokens
    lays = {l: oracle.Layer(weights[l], top_k) for l in ffn_layers}
    worst = 0.0
    for b in range(B):
        h = oracle.as_bits(H[b])
        for l in range(L):
            x_gpu = oracle.as_bits(xs[l, b])
            if prenorm:
                x_ref = oracle.rmsnorm_bf16(h, eps)
                dx = np.abs(bf16_to_f64(x_gpu) - bf16_to_f64(x_ref))
                assert np.all(dx <= np.abs(bf16_to_f64(x_ref)) * 2.0 ** -7 + 1e-30), f"token {b} layer {l}: x"
            else:
                assert np.array_equal(x_gpu, h), f"token {b} layer {l}: x must equal h without the norm"
            bl = None if bias_np is None else bias_np[l, b]
            lg, st = oracle.router_logits(oracle.as_bits(weights[l]["router_w"]), x_gpu, bl)
            assert st == 0
            rid = oracle.topk(lg, top_k)
            assert list(ids[l, b].numpy()) == list(rid), f"token {b} layer {l}: ids {ids[l, b].tolist()} vs {list(rid)}"
            assert np.allclose(gs[l, b].numpy(), oracle.gates(lg, rid), rtol=GATE_RTOL, atol=1e-7), \
                f"token {b} layer {l}: gates"
            if lgs is not None:
                check_logits(lgs[l, b], lg, rid, f"token {b} layer {l}", candidates_only)
            if l in lays and b in ffn_tokens:
                _, _, _, ry, _ = lays[l].forward(x_gpu, bl)
                worst = max(worst, assert_ffn_close(ys[l, b].numpy(), ry, f"token {b} layer {l}"))
            y32 = ys[l, b].numpy().astype(np.float32)
            h_ref = oracle.residual_bf16(h, y32.astype(np.float64))
            # the kernels form h + y in fp32 and round that to bf16; the fp64 sum
            # can round the other way on a tie of the fp32 result (one ulp), and a
            # one-ulp step would carry through the rest of the stack, so the chain
            # follows the fp32 rule after checking both agree within an ulp
            s32 = (bf16_to_f64(h).astype(np.float32) + y32).astype(np.float64)
            h = oracle.residual_bf16(np.zeros_like(h), s32)
            dh = np.abs(bf16_to_f64(h) - bf16_to_f64(h_ref))
            assert np.all(dh <= np.abs(bf16_to_f64(h_ref)) * 2.0 ** -7 + 1e-30), f"token {b} layer {l}: h + y"
        if h_out is not None:
            got = bf16_to_f64(oracle.as_bits(h_out[b]))
            ref = bf16_to_f64(h)
            assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30), f"token {b}: h_out"
    return worst
