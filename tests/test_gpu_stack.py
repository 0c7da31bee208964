"""Layer stacks: teacher-forced per-layer parity of the residual stream
(x_l = bf16(RMSNorm(h_l)), logits, ids, gates, y_l, h_{l+1} = bf16(h_l + y_l))
through the persistent one-token kernels, the per-layer kernels and, for 32
tokens, the tensor-core grouped GEMM path."""

import pytest
import torch

import bit_routed_expert_router_gb300 as moe
from workload import FULL, TINY, Shape, gen_hidden, gen_layer

from moe_harness import (DECODE_KERNELS, Ctx, assert_ffn_close, capture, check_stack, end_capture, to_host,
                         use_decode_kernel)

pytestmark = pytest.mark.gpu


def _check_stack(ctx, weights_host, H, L, ffn_layers, bias=None, ffn_tokens=None):
    B = H.shape[0]
    cap = capture(ctx, L, B, logits=True)
    h_out, y_last, _ = ctx.decode(H, 0, L, bias=bias)
    ctx.sync()
    end_capture(ctx)
    assert torch.equal(y_last, cap["y"][L - 1])
    check_stack(weights_host, H, cap, h_out, ctx.shape.top_k, ffn_layers, ffn_tokens, bias,
                candidates_only=B >= 2)


@pytest.mark.parametrize("kernel", DECODE_KERNELS)
def test_tiny_stack_eight_layers(kernel):
    L = 8
    ws = [gen_layer(TINY, seed=80, layer=l) for l in range(L)]
    with Ctx(TINY, n_layers=L, prenorm=1) as ctx:
        for l in range(L):
            ctx.init_layer(l, {"router_w": ws[l]["router_w"].cuda(),
                               "experts": {k: v.cuda() for k, v in ws[l]["experts"].items()},
                               "shared": {k: v.cuda() for k, v in ws[l]["shared"].items()}})
        use_decode_kernel(ctx, kernel)
        H = (gen_hidden(3, TINY.d, seed=80).float() * 2).to(torch.bfloat16).cuda()
        for t in range(3):
            _check_stack(ctx, ws, H[t:t + 1], L, ffn_layers=set(range(L)))
        # consecutive calls reuse the kernel's counters: run a few more and check again
        for t in range(5):
            ctx.decode(H[t % 3:t % 3 + 1])
        _check_stack(ctx, ws, H[1:2], L, ffn_layers={0, 7})


def test_full_stack_thirty_layers_one_token():
    L = 30
    sh = FULL
    hosts = []
    with Ctx(sh, n_layers=L, prenorm=1) as ctx:
        for l in range(L):
            w = gen_layer(sh, seed=2, layer=l, device="cuda")
            ctx.init_layer(l, w)
            keep = l in (0, 13, 29)
            hosts.append(to_host(w) if keep else {"router_w": w["router_w"].cpu()})
            del w
        H = gen_hidden(2, sh.d, seed=2, device="cuda")
        from workload import bias_from_targets, zipf_reuse_targets
        tg = zipf_reuse_targets(2, L, sh.n_experts, sh.top_k, seed=2)
        bias_all = torch.from_numpy(bias_from_targets(tg, sh.n_experts)).cuda()   # [T, L, E]
        for t in range(2):
            b = bias_all[t].unsqueeze(1).contiguous() if t == 1 else None        # [L, 1, E]
            _check_stack(ctx, hosts, H[t:t + 1], L, ffn_layers={0, 13, 29}, bias=b)


def test_persistent_and_layer_kernels_agree():
    L = 4
    sh = Shape(d=1024, f=256, f_shared=1024, n_experts=32, top_k=4)
    ws = [gen_layer(sh, seed=90, layer=l, device="cuda") for l in range(L)]
    with Ctx(sh, n_layers=L, prenorm=1) as ctx:
        for l in range(L):
            ctx.init_layer(l, ws[l])
        H = gen_hidden(6, sh.d, seed=90, device="cuda")
        outs = {}
        for kernel in DECODE_KERNELS:
            use_decode_kernel(ctx, kernel)
            ys = []
            for t in range(6):
                _, y, _ = ctx.decode(H[t:t + 1])
                ys.append(y.clone())
            ctx.sync()
            outs[kernel] = torch.cat(ys)
        for kernel in ("cluster", "per_sm"):
            for t in range(6):
                assert_ffn_close(outs[kernel][t].cpu().numpy(), outs["layers"][t].cpu().double().numpy(),
                                 f"{kernel} token {t}")


def _full_stack(seed, keep):
    """A 30-layer full-shape context (RMS pre-norm between layers) and the host
    weights: every router, and the full weights of the layers in keep."""
    L, sh = 30, FULL
    ctx = Ctx(sh, n_layers=L, prenorm=1)
    hosts = []
    for l in range(L):
        w = gen_layer(sh, seed=seed, layer=l, device="cuda")
        ctx.init_layer(l, w)
        hosts.append(to_host(w) if l in keep else {"router_w": w["router_w"].cpu()})
        del w
    return ctx, hosts


def test_full_stack_thirty_layers_batch32():
    """The batched workload (32 tokens, 30 layers, Zipf-reuse routing bias) through
    the tensor-core path: every token's logits, ids and gates on every layer,
    FFN outputs on sampled layers and tokens."""
    import os

    import oracle
    from workload import bias_from_targets, zipf_reuse_targets
    oracle.set_threads(os.cpu_count())
    L, B, sh = 30, 32, FULL
    ctx, hosts = _full_stack(seed=3, keep=(0, 14, 29))
    with ctx:
        H = gen_hidden(B, sh.d, seed=3, device="cuda")
        tg = zipf_reuse_targets(B, L, sh.n_experts, sh.top_k, seed=3)
        bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts).transpose(1, 0, 2).copy()).cuda()  # [L, B, E]
        _check_stack(ctx, hosts, H, L, ffn_layers={0, 14, 29}, bias=bias, ffn_tokens=(0, 9, 22, 31))
