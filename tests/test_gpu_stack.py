"""Layer stacks: teacher-forced per-layer parity of the residual stream
(x_l = bf16(RMSNorm(h_l)), y_l, h_{l+1} = bf16(h_l + y_l)) through the
persistent one-token kernel and the per-layer kernels."""

import numpy as np
import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, TINY, Shape, gen_hidden, gen_layer

from moe_harness import DECODE_KERNELS, GATE_RTOL, Ctx, assert_ffn_close, bf16_to_f64, to_host, use_decode_kernel

pytestmark = pytest.mark.gpu


def _capture(ctx, H, L, bias=None):
    B, d, k = H.shape[0], ctx.shape.d, ctx.shape.top_k
    xs = torch.zeros(L, B, d, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(L, B, k, dtype=torch.int32, device="cuda")
    gs = torch.zeros(L, B, k, dtype=torch.float32, device="cuda")
    ys = torch.zeros(L, B, d, dtype=torch.float32, device="cuda")
    moe.check(moe.moe_set_debug(ctx.h, xs, ids, gs, ys, L), ctx.h)
    h_out, y_last, _ = ctx.decode(H, 0, L, bias=bias)
    ctx.sync()
    moe.check(moe.moe_set_debug(ctx.h), ctx.h)
    return xs, ids, gs, ys, h_out, y_last


def _check_stack(ctx, weights_host, H, L, ffn_layers, bias=None):
    xs, ids, gs, ys, h_out, y_last = _capture(ctx, H, L, bias)
    assert torch.equal(y_last, ys[L - 1])
    B = H.shape[0]
    for b in range(B):
        h = oracle.as_bits(H[b])
        for l in range(L):
            x_gpu = oracle.as_bits(xs[l, b])
            x_ref = oracle.rmsnorm_bf16(h, 1e-6)
            dx = np.abs(bf16_to_f64(x_gpu) - bf16_to_f64(x_ref))
            assert np.all(dx <= np.abs(bf16_to_f64(x_ref)) * 2.0 ** -7 + 1e-30), f"layer {l}: x off by > 1 ulp"
            w = weights_host[l]
            rw = oracle.as_bits(w["router_w"])
            bl = None if bias is None else bias[l, b].cpu().numpy()
            lg, st = oracle.router_logits(rw, x_gpu, bl)
            assert st == 0
            rid = oracle.topk(lg, ctx.shape.top_k)
            assert list(ids[l, b].cpu().numpy()) == list(rid), f"token {b} layer {l}: ids"
            assert np.allclose(gs[l, b].cpu().numpy(), oracle.gates(lg, rid), rtol=GATE_RTOL, atol=1e-7)
            if l in ffn_layers:
                lay = oracle.Layer(w, ctx.shape.top_k)
                _, _, _, ry, _ = lay.forward(x_gpu, bl)
                assert_ffn_close(ys[l, b].cpu().numpy(), ry, f"token {b} layer {l}")
            y32 = ys[l, b].cpu().numpy().astype(np.float32)
            h_ref = oracle.residual_bf16(h, y32.astype(np.float64))
            # the kernels form h + y in fp32 and round that to bf16; the fp64 sum
            # can round the other way on a tie of the fp32 result (one ulp), and a
            # one-ulp step would carry through the rest of the stack, so the
            # chain follows the fp32 rule after checking both agree within an ulp
            s32 = (bf16_to_f64(h).astype(np.float32) + y32).astype(np.float64)
            h = oracle.residual_bf16(np.zeros_like(h), s32)
            dh = np.abs(bf16_to_f64(h) - bf16_to_f64(h_ref))
            assert np.all(dh <= np.abs(bf16_to_f64(h_ref)) * 2.0 ** -7 + 1e-30), f"layer {l}: h + y"
        got = bf16_to_f64(oracle.as_bits(h_out[b]))
        ref = bf16_to_f64(h)
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)


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
