"""GPU parity of the decode path (router logits, top-k, gates, int4
gate/up/GELU, down, combine) against the CPU oracle, through the C ABI."""

import os

import numpy as np
import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, TINY, Shape, gen_hidden, gen_layer

from moe_harness import (DECODE_KERNELS, GATE_RTOL, Ctx, assert_ffn_close, bf16_to_f64, capture, check_logits,
                         check_stack, end_capture, to_device, to_host, use_decode_kernel)

pytestmark = pytest.mark.gpu


def _check_layer_outputs(ctx, lay, H, bias=None):
    """Run H [B, d] through one layer with debug capture; compare every token."""
    B, d = H.shape
    k = ctx.shape.top_k
    dev = H.device
    xs = torch.zeros(1, B, d, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(1, B, k, dtype=torch.int32, device=dev)
    gs = torch.zeros(1, B, k, dtype=torch.float32, device=dev)
    ys = torch.zeros(1, B, d, dtype=torch.float32, device=dev)
    lgs = torch.full((1, B, ctx.shape.n_experts), 7, dtype=torch.int64, device=dev)
    moe.check(moe.moe_set_debug(ctx.h, xs, ids, gs, ys, 1), ctx.h)
    moe.check(moe.moe_set_debug_logits(ctx.h, lgs), ctx.h)
    h_out, y, _ = ctx.decode(H, 0, 1, bias=bias)
    ctx.sync()
    end_capture(ctx)
    lgs = lgs[0].cpu().numpy()
    assert torch.equal(y, ys[0])
    worst = 0.0
    for b in range(B):
        xb = oracle.as_bits(xs[0, b])
        bb = None if bias is None else bias[0, b].cpu().numpy()
        rid, rg, rlg, ry, st = lay.forward(xb, bb)
        assert st == 0
        assert list(ids[0, b].cpu().numpy()) == list(rid), f"token {b}: ids {ids[0, b].tolist()} vs {list(rid)}"
        assert np.allclose(gs[0, b].cpu().numpy(), rg, rtol=GATE_RTOL, atol=1e-7)
        # the grouped path (batches) evaluates only the candidates exactly
        check_logits(lgs[b], rlg, rid, f"token {b}", candidates_only=B >= 2)
        worst = max(worst, assert_ffn_close(y[b].cpu().numpy(), ry, f"token {b}"))
        # residual: h_out = bf16(h + y) from the GPU's own y
        ref_h = oracle.residual_bf16(oracle.as_bits(H[b]), y[b].cpu().double().numpy())
        got_h = oracle.as_bits(h_out[b])
        diff = np.abs(bf16_to_f64(got_h) - bf16_to_f64(ref_h))
        ulp = np.abs(bf16_to_f64(ref_h)) * 2.0 ** -7 + 1e-38
        assert np.all(diff <= ulp)
    return xs, worst


def _tiny_ctx(shape=TINY, prenorm=0, seed=0, gelu=0):
    w = gen_layer(shape, seed=seed, layer=0)
    ctx = Ctx(shape, n_layers=1, prenorm=prenorm, gelu=gelu)
    ctx.init_layer(0, to_device(w))
    return ctx, oracle.Layer(w, shape.top_k, gelu_variant=gelu)


@pytest.mark.parametrize("kernel", DECODE_KERNELS)
def test_tiny_layer_single_tokens(kernel):
    ctx, lay = _tiny_ctx()
    with ctx:
        use_decode_kernel(ctx, kernel)
        H = gen_hidden(16, TINY.d, seed=0).cuda()
        for t in range(16):
            _check_layer_outputs(ctx, lay, H[t:t + 1])


def use_batch_path(ctx, path):
    """small: small-batch grouped GEMVs (the default from 5 tokens on); tc:
    tcgen05 GEMMs from 16 tokens on, per-layer GEMVs below; gemv: per-layer
    GEMVs; loop: one clustered-kernel launch per token (the default for 2 to 4
    tokens).  All but loop switch the per-token launches off."""
    moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_TOKEN_LOOP, 1 if path == "loop" else 0), ctx.h)
    if path == "loop":
        return
    moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PREFILL_TC, 0 if path == "gemv" else 1), ctx.h)
    if path != "gemv":
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_SMALL_BATCH, 1 if path == "small" else 0), ctx.h)


@pytest.mark.parametrize("path", ["small", "tc", "gemv", "loop"])
@pytest.mark.parametrize("B", [2, 3, 8, 9, 31, 32])
def test_tiny_layer_batched(B, path):
    if path == "loop" and B > 4:
        pytest.skip("one launch per token covers 2 to 4 tokens")
    ctx, lay = _tiny_ctx()
    with ctx:
        use_batch_path(ctx, path)
        H = gen_hidden(B, TINY.d, seed=100 + B).cuda()
        _check_layer_outputs(ctx, lay, H)


def test_tiny_layer_batch_equals_single_tokens():
    ctx, lay = _tiny_ctx()
    with ctx:
        H = gen_hidden(12, TINY.d, seed=7).cuda()
        _, yb, _ = ctx.decode(H, 0, 1)
        for t in range(12):
            _, y1, _ = ctx.decode(H[t:t + 1], 0, 1)
            assert_ffn_close(y1[0].cpu().numpy(), yb[t].cpu().double().numpy(), f"token {t}")


@pytest.mark.parametrize("B", [2, 4])
def test_few_tokens_one_launch_each(B):
    """2 to 4 tokens take one clustered-kernel launch per token: each token's
    h_out, y and captured ids / gates equal its own single-token call bit for
    bit (two layers, full shape, a routing bias per token and layer)."""
    sh, L = FULL, 2
    with Ctx(sh, n_layers=L, prenorm=1) as ctx:
        for l in range(L):
            ctx.init_layer(l, gen_layer(sh, seed=9, layer=l, device="cuda"))
        H = gen_hidden(B, sh.d, seed=9, device="cuda")
        g = torch.Generator().manual_seed(9)
        bias = (torch.randn(L, B, sh.n_experts, generator=g) * 0.5).cuda()
        cap = capture(ctx, L, B)
        h_b, y_b, _ = ctx.decode(H, 0, L, bias=bias)
        ctx.sync()
        ids_b, gates_b = cap["ids"].clone(), cap["gates"].clone()
        end_capture(ctx)
        for t in range(B):
            cap1 = capture(ctx, L, 1)
            h1, y1, _ = ctx.decode(H[t:t + 1], 0, L, bias=bias[:, t:t + 1].contiguous())
            ctx.sync()
            assert torch.equal(h1[0].view(torch.int16), h_b[t].view(torch.int16)), f"token {t}: h_out"
            assert torch.equal(y1[0], y_b[t]), f"token {t}: y"
            assert torch.equal(cap1["ids"][:, 0], ids_b[:, t]), f"token {t}: ids"
            assert torch.equal(cap1["gates"][:, 0], gates_b[:, t]), f"token {t}: gates"
            end_capture(ctx)


def test_tanh_gelu_variant():
    ctx, lay = _tiny_ctx(gelu=1, seed=5)
    with ctx:
        H = gen_hidden(4, TINY.d, seed=5).cuda()
        _check_layer_outputs(ctx, lay, H)
        _check_layer_outputs(ctx, lay, H[1:2])


def test_prenorm_input_matches_oracle_rmsnorm():
    ctx, lay = _tiny_ctx(prenorm=1, seed=9)
    with ctx:
        H = (gen_hidden(6, TINY.d, seed=9).float() * 3.0).to(torch.bfloat16).cuda()
        xs, _ = _check_layer_outputs(ctx, lay, H)
        for b in range(6):
            ref = bf16_to_f64(oracle.rmsnorm_bf16(oracle.as_bits(H[b]), 1e-6))
            got = bf16_to_f64(oracle.as_bits(xs[0, b]))
            assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)


def test_odd_shapes_and_uneven_shared_chunks():
    # E not a multiple of 8, f/64 = 1 so the shared down splits into 3 chunks
    sh = Shape(d=192, f=64, f_shared=192, n_experts=5, top_k=3)
    ctx, lay = _tiny_ctx(sh, seed=21)
    with ctx:
        H = gen_hidden(5, sh.d, seed=21).cuda()
        _check_layer_outputs(ctx, lay, H)
        for t in range(5):
            _check_layer_outputs(ctx, lay, H[t:t + 1])


@pytest.mark.parametrize("path", ["small", "gemv"])
def test_long_rows_several_stages_per_task(path):
    # d/64 = 24 groups (gate/up tiles span 3 stages), f/64 = 13 (down tiles span 2 stages;
    # small-batch routed down stages of three 16-row tiles, the last stage short),
    # f_shared/64 = 23 (three shared down chunks, the last one short)
    sh = Shape(d=1536, f=832, f_shared=1472, n_experts=16, top_k=4)
    ctx, lay = _tiny_ctx(sh, seed=23)
    with ctx:
        use_batch_path(ctx, path)
        H = gen_hidden(20, sh.d, seed=23).cuda()
        for t in range(4):
            _check_layer_outputs(ctx, lay, H[t:t + 1])
        _check_layer_outputs(ctx, lay, H[:4])
        _check_layer_outputs(ctx, lay, H)      # up to 20 tokens on an expert: three token blocks


def test_router_ties_go_to_lower_index():
    sh = TINY
    w = gen_layer(sh, seed=31, layer=0)
    rw = w["router_w"].clone()
    rw[5] = rw[2]      # experts 2 and 5 always tie
    rw[7] = rw[0]      # experts 0 and 7 always tie
    w["router_w"] = rw
    ctx = Ctx(sh, n_layers=1)
    with ctx:
        ctx.init_layer(0, to_device(w))
        lay = oracle.Layer(w, sh.top_k)
        H = gen_hidden(32, sh.d, seed=31).cuda()
        _check_layer_outputs(ctx, lay, H)


def test_logit_bias_and_exact_ties_from_bias():
    sh = TINY
    w = gen_layer(sh, seed=41, layer=0)
    w["router_w"] = torch.zeros_like(w["router_w"])
    ctx = Ctx(sh, n_layers=1)
    with ctx:
        ctx.init_layer(0, to_device(w))
        lay = oracle.Layer(w, sh.top_k)
        H = gen_hidden(8, sh.d, seed=41).cuda()
        bias = torch.zeros(1, 8, sh.n_experts, dtype=torch.float32)
        bias[0, :, 3] = 16.0
        bias[0, :4, 6] = 16.0   # ties at 16 for the first four tokens -> expert 3 first
        _check_layer_outputs(ctx, lay, H, bias.cuda())


def test_dense_equivalence_invariant():
    """W_r = 0, k = E: ids = 0..E-1, gates 1/E, y = FFN_s + mean_e FFN_e."""
    sh = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=8)
    w = gen_layer(sh, seed=51, layer=0)
    w["router_w"] = torch.zeros_like(w["router_w"])
    ctx = Ctx(sh, n_layers=1)
    with ctx:
        ctx.init_layer(0, to_device(w))
        H = gen_hidden(3, sh.d, seed=51).cuda()
        _, y, _ = ctx.decode(H, 0, 1)
        for b in range(3):
            x = bf16_to_f64(oracle.as_bits(H[b]))
            ref = oracle.expert_ffn(w["shared"], x)
            for e in range(8):
                ref = ref + oracle.expert_ffn({k: v[e] for k, v in w["experts"].items()}, x) / 8.0
            assert_ffn_close(y[b].cpu().numpy(), ref, f"token {b}")


def test_host_weights_equal_device_weights():
    w = gen_layer(TINY, seed=61, layer=0)
    H = gen_hidden(4, TINY.d, seed=61).cuda()
    outs = []
    for src in ("cpu", "cuda"):
        ctx = Ctx(TINY, n_layers=1)
        with ctx:
            ctx.init_layer(0, to_device(w, src))
            _, y, _ = ctx.decode(H, 0, 1)
            ctx.sync()
            outs.append(y.clone())
    assert torch.equal(outs[0], outs[1])


def test_full_shape_layer_sampled_tokens():
    sh = FULL
    wd = gen_layer(sh, seed=1, layer=0, device="cuda")
    ctx = Ctx(sh, n_layers=1)
    with ctx:
        ctx.init_layer(0, wd)
        from moe_harness import to_host
        lay = oracle.Layer(to_host(wd), sh.top_k)
        H = gen_hidden(1024, sh.d, seed=1, device="cuda")
        # routing for many tokens through the batched path, bit-exact
        ids_all = []
        for t0 in range(0, 256, 32):
            k = sh.top_k
            ids = torch.zeros(1, 32, k, dtype=torch.int32, device="cuda")
            moe.check(moe.moe_set_debug(ctx.h, None, ids, None, None, 1), ctx.h)
            ctx.decode(H[t0:t0 + 32], 0, 1)
            ctx.sync()
            ids_all.append(ids[0].cpu().numpy())
        moe.check(moe.moe_set_debug(ctx.h), ctx.h)
        ids_all = np.concatenate(ids_all)
        rw = oracle.as_bits(wd["router_w"].cpu())
        for t in range(0, 256, 5):
            lg, st = oracle.router_logits(rw, oracle.as_bits(H[t]))
            assert list(ids_all[t]) == list(oracle.topk(lg, sh.top_k)), f"token {t}"
        # full FFN parity on sampled single tokens, at the bench launch shape (B = 1),
        # through the persistent kernel and through the per-layer kernels
        for t in (0, 1, 517, 1023):
            _check_layer_outputs(ctx, lay, H[t:t + 1])
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PERSISTENT, 0), ctx.h)
        for t in (2, 700):
            _check_layer_outputs(ctx, lay, H[t:t + 1])
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PERSISTENT, 1), ctx.h)
        # and a ragged batch
        _check_layer_outputs(ctx, lay, H[100:105])


def test_c1_thousand_tokens_through_the_clustered_kernel():
    """The one-token decode workload at full shape, 1024 tokens one at a time
    through the kernel the decode benchmark times: every token's int64 logits
    and ids bit-exact, every eighth token's FFN output (128 tokens)."""
    sh, T = FULL, 1024
    wd = gen_layer(sh, seed=11, layer=0, device="cuda")
    oracle.set_threads(os.cpu_count())
    with Ctx(sh, n_layers=1) as ctx:
        ctx.init_layer(0, wd)
        use_decode_kernel(ctx, "cluster")
        w = to_host(wd)
        del wd
        H = gen_hidden(T, sh.d, seed=11, device="cuda")
        k, E = sh.top_k, sh.n_experts
        ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
        lgs = torch.full((T, E), 7, dtype=torch.int64, device="cuda")
        y = torch.zeros(T, sh.d, dtype=torch.float32, device="cuda")
        h_out = torch.empty_like(H)
        for t in range(T):
            # each call captures into its own rows (one layer, one token)
            moe.check(moe.moe_set_debug(ctx.h, None, ids[t:t + 1], None, None, 1), ctx.h)
            moe.check(moe.moe_set_debug_logits(ctx.h, lgs[t:t + 1]), ctx.h)
            st, _ = moe.moe_decode_step(ctx.h, H[t:t + 1], 1, 0, 1, None, h_out[t:t + 1], y[t:t + 1], None, None)
            moe.check(st, ctx.h)
        ctx.sync()
        end_capture(ctx)
        ids, lgs, y = ids.cpu().numpy(), lgs.cpu().numpy(), y.cpu().numpy()
        rw = oracle.as_bits(w["router_w"])
        Hb = oracle.as_bits(H.cpu())
        for t in range(T):
            lg, st = oracle.router_logits(rw, Hb[t])
            assert st == 0
            rid = oracle.topk(lg, k)
            assert list(ids[t]) == list(rid), f"token {t}: ids {ids[t].tolist()} vs {list(rid)}"
            check_logits(lgs[t], lg, rid, f"token {t}")
        lay = oracle.Layer(w, k)
        worst = 0.0
        for t in range(0, T, 8):
            _, _, _, ry, st = lay.forward(Hb[t])
            assert st == 0
            worst = max(worst, assert_ffn_close(y[t], ry, f"token {t}"))


@pytest.mark.parametrize("path", ["small", "tc"])
def test_full_shape_batch32_grouped_paths(path):
    """32 tokens at full shape on the grouped path, with the small-batch GEMVs
    (one item per active expert, 44 k-groups per gate/up tile) or the tcgen05
    GEMMs (32-row token tiles): every token's ids, gates, candidate logits and
    FFN output on two layers against the oracle."""
    sh, L, B = FULL, 2, 32
    oracle.set_threads(os.cpu_count())
    with Ctx(sh, n_layers=L, prenorm=1) as ctx:
        use_batch_path(ctx, path)
        hosts = []
        for l in range(L):
            wd = gen_layer(sh, seed=12, layer=l, device="cuda")
            ctx.init_layer(l, wd)
            hosts.append(to_host(wd))
            del wd
        H = gen_hidden(B, sh.d, seed=12, device="cuda")
        cap = capture(ctx, L, B, logits=True)
        h_out, y_last, _ = ctx.decode(H, 0, L)
        ctx.sync()
        end_capture(ctx)
        assert torch.equal(y_last, cap["y"][L - 1])
        check_stack(hosts, H, cap, h_out, sh.top_k, ffn_layers={0, 1}, candidates_only=True)
