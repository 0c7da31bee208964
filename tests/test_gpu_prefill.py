"""GPU parity of the batched prefill (tcgen05 grouped GEMM path) against the
CPU oracle, through the C ABI: exact routing, gates, FFN output and residual
per token, teacher-forced per layer through the debug capture."""

import numpy as np
import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, TINY, Shape, bias_from_targets, gen_hidden, gen_layer, mixture_targets

from moe_harness import GATE_RTOL, Ctx, assert_ffn_close, bf16_to_f64, check_stack, to_device, to_host

pytestmark = pytest.mark.gpu

MEDIUM = Shape(d=512, f=192, f_shared=256, n_experts=16, top_k=4, group=64, n_layers=1)


def _run_prefill(ctx, H, n_layers=1, bias=None, tc=True):
    """Prefill H [T, d] through layers [0, n_layers) with debug capture of every layer."""
    T, d = H.shape
    k = ctx.shape.top_k
    dev = H.device
    moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PREFILL_TC, 1 if tc else 0), ctx.h)
    xs = torch.zeros(n_layers, T, d, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(n_layers, T, k, dtype=torch.int32, device=dev)
    gs = torch.zeros(n_layers, T, k, dtype=torch.float32, device=dev)
    ys = torch.zeros(n_layers, T, d, dtype=torch.float32, device=dev)
    moe.check(moe.moe_set_debug(ctx.h, xs, ids, gs, ys, n_layers), ctx.h)
    h_out = torch.empty_like(H)
    y = torch.empty(T, d, dtype=torch.float32, device=dev)
    moe.check(moe.moe_prefill(ctx.h, H, T, 0, n_layers, bias, h_out, y), ctx.h)
    ctx.sync()
    moe.check(moe.moe_set_debug(ctx.h), ctx.h)
    return h_out, y, xs, ids, gs, ys


def _check_tokens(lay, H_in, xs, ids, gs, ys, h_out, tokens, bias=None, prenorm=0):
    """Oracle check of one layer's outputs for the given tokens (teacher-forced on the GPU's x)."""
    worst = 0.0
    for t in tokens:
        xb = oracle.as_bits(xs[t])
        if prenorm:
            ref_x = bf16_to_f64(oracle.rmsnorm_bf16(oracle.as_bits(H_in[t]), 1e-6))
            got_x = bf16_to_f64(xb)
            assert np.all(np.abs(got_x - ref_x) <= np.abs(ref_x) * 2.0 ** -7 + 1e-30), f"token {t}: x"
        else:
            assert np.array_equal(xb, oracle.as_bits(H_in[t])), f"token {t}: x must equal h without the norm"
        bb = None if bias is None else bias[t].cpu().numpy()
        rid, rg, _, ry, st = lay.forward(xb, bb)
        assert st == 0
        assert list(ids[t].cpu().numpy()) == list(rid), f"token {t}: ids {ids[t].tolist()} vs {list(rid)}"
        assert np.allclose(gs[t].cpu().numpy(), rg, rtol=GATE_RTOL, atol=1e-7), f"token {t}: gates"
        worst = max(worst, assert_ffn_close(ys[t].cpu().numpy(), ry, f"token {t}"))
        if h_out is not None:
            ref_h = oracle.residual_bf16(oracle.as_bits(H_in[t]), ys[t].cpu().double().numpy())
            diff = np.abs(bf16_to_f64(oracle.as_bits(h_out[t])) - bf16_to_f64(ref_h))
            assert np.all(diff <= np.abs(bf16_to_f64(ref_h)) * 2.0 ** -7 + 1e-38), f"token {t}: residual"
    return worst


def _ctx(shape, n_layers=1, prenorm=0, max_tokens=512, seed=0, gelu=0):
    ctx = Ctx(shape, n_layers=n_layers, prenorm=prenorm, max_tokens=max_tokens, gelu=gelu)
    lays = []
    for l in range(n_layers):
        w = gen_layer(shape, seed=seed, layer=l)
        ctx.init_layer(l, to_device(w))
        lays.append(oracle.Layer(w, shape.top_k, gelu_variant=gelu))
    return ctx, lays


@pytest.mark.parametrize("T", [1, 7, 130, 300])
@pytest.mark.parametrize("prenorm", [0, 1])
def test_prefill_tiny_layer(T, prenorm):
    ctx, (lay,) = _ctx(TINY, prenorm=prenorm, seed=3)
    with ctx:
        H = gen_hidden(T, TINY.d, seed=100 + T).cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H)
        assert torch.equal(y, ys[0])
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(T), prenorm=prenorm)


def test_prefill_tanh_gelu():
    ctx, (lay,) = _ctx(TINY, seed=5, gelu=1)
    with ctx:
        H = gen_hidden(40, TINY.d, seed=5).cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H)
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(40))


def test_prefill_medium_shape_all_tokens():
    # 4 k-steps per raw stage with a ragged last stage (f/64 = 3), several items per expert
    ctx, (lay,) = _ctx(MEDIUM, seed=7)
    with ctx:
        H = gen_hidden(300, MEDIUM.d, seed=7).cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H)
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(300))


def test_prefill_concentrated_and_empty_experts():
    # every token routed to experts 3 and 5 (bias): two experts with 300 rows (three
    # 128-row items each), six experts with none
    ctx, (lay,) = _ctx(TINY, seed=11)
    with ctx:
        T = 300
        H = gen_hidden(T, TINY.d, seed=11).cuda()
        bias = torch.zeros(1, T, TINY.n_experts, dtype=torch.float32)
        bias[0, :, 3] = 16.0
        bias[0, :, 5] = 16.0
        bias = bias.cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H, bias=bias)
        assert set(ids[0].flatten().tolist()) == {3, 5}
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(T), bias=bias[0])


def test_prefill_tiny_stack_teacher_forced():
    L = 3
    ctx, lays = _ctx(TINY, n_layers=L, prenorm=1, seed=13)
    with ctx:
        T = 64
        H = gen_hidden(T, TINY.d, seed=13).cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H, n_layers=L)
        h_cur = H
        for l in range(L):
            _check_tokens(lays[l], h_cur, xs[l], ids[l], gs[l], ys[l], None, range(T), prenorm=1)
            # the next layer's input is this layer's residual output, rebuilt from the GPU's own y
            h_cur = torch.stack([torch.from_numpy(oracle.residual_bf16(oracle.as_bits(h_cur[t]),
                                                                        ys[l, t].cpu().double().numpy()).view(np.int16))
                                 for t in range(T)]).view(torch.bfloat16).cuda()
        # bf16(h + y) with the add in fp32 (GPU) vs fp64 (oracle): equal up to one bf16 ulp
        got = bf16_to_f64(oracle.as_bits(h_out.cpu()))
        ref = bf16_to_f64(oracle.as_bits(h_cur.cpu()))
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-38)
        assert torch.equal(y, ys[L - 1])


def test_prefill_equals_batched_decode_path():
    ctx, (lay,) = _ctx(MEDIUM, seed=17)
    with ctx:
        T = 200
        H = gen_hidden(T, MEDIUM.d, seed=17).cuda()
        out_tc = _run_prefill(ctx, H, tc=True)
        out_dec = _run_prefill(ctx, H, tc=False)
        assert torch.equal(out_tc[3], out_dec[3])                      # ids
        assert torch.allclose(out_tc[4], out_dec[4], rtol=1e-6, atol=0)  # gates
        for t in range(T):
            assert_ffn_close(out_tc[1][t].cpu().numpy(), out_dec[1][t].cpu().double().numpy(), f"token {t}")


def test_prefill_fp16_range_is_reported():
    ctx, _ = _ctx(TINY, seed=19)
    with ctx:
        H = gen_hidden(8, TINY.d, seed=19)
        H[3, 17] = 1.0e5     # outside fp16 without the norm
        H = H.cuda()
        h_out = torch.empty_like(H)
        moe.check(moe.moe_prefill(ctx.h, H, 8, 0, 1, None, h_out, None), ctx.h)
        st = moe.moe_sync(ctx.h)
        assert st == moe.MOE_EDOMAIN, moe.status_name(st)


def test_prefill_full_shape_sampled_tokens():
    """T = 4096 (the prefill workload: uniform-plus-Zipf routing bias) at full shape;
    sampled tokens against the oracle, every token's routing against the oracle's top-k."""
    sh = FULL
    wd = gen_layer(sh, seed=4, layer=0, device="cuda")
    ctx = Ctx(sh, n_layers=1, prenorm=1, max_tokens=4096)
    with ctx:
        ctx.init_layer(0, wd)
        lay = oracle.Layer(to_host(wd), sh.top_k)
        T = 4096
        H = gen_hidden(T, sh.d, seed=4, device="cuda")
        tg = mixture_targets(T, 1, sh.n_experts, sh.top_k, seed=4)
        bias = torch.from_numpy(np.ascontiguousarray(
            bias_from_targets(tg, sh.n_experts).astype(np.float32).transpose(1, 0, 2))).cuda()  # [L, T, E]
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H, bias=bias)
        rw = oracle.as_bits(wd["router_w"].cpu())
        ids_np = ids[0].cpu().numpy()
        for t in range(0, T, 97):
            lg, st = oracle.router_logits(rw, oracle.as_bits(xs[0, t]), bias[0, t].cpu().numpy())
            assert st == 0
            assert list(ids_np[t]) == list(oracle.topk(lg, sh.top_k)), f"token {t}"
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, (0, 1, 2047, 4095), bias=bias[0], prenorm=1)


def test_prefill_router_exact_ties_and_zero_rows():
    """Duplicated router rows tie exactly (ties go to the lower index) and an
    all-zero router with a bias that ties on some tokens: the candidate filter
    must keep every tied expert."""
    w = gen_layer(TINY, seed=31, layer=0)
    rw = w["router_w"].clone()
    rw[5] = rw[2]
    rw[7] = rw[0]
    w["router_w"] = rw
    ctx = Ctx(TINY, n_layers=1, max_tokens=512)
    with ctx:
        ctx.init_layer(0, to_device(w))
        lay = oracle.Layer(w, TINY.top_k)
        H = gen_hidden(200, TINY.d, seed=31).cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H)
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(200))
    w2 = gen_layer(TINY, seed=41, layer=0)
    w2["router_w"] = torch.zeros_like(w2["router_w"])
    ctx = Ctx(TINY, n_layers=1, max_tokens=512)
    with ctx:
        ctx.init_layer(0, to_device(w2))
        lay = oracle.Layer(w2, TINY.top_k)
        T = 40
        H = gen_hidden(T, TINY.d, seed=41).cuda()
        bias = torch.zeros(1, T, TINY.n_experts, dtype=torch.float32)
        bias[0, :, 3] = 16.0
        bias[0, :20, 6] = 16.0
        bias = bias.cuda()
        h_out, y, xs, ids, gs, ys = _run_prefill(ctx, H, bias=bias)
        _check_tokens(lay, H, xs[0], ids[0], gs[0], ys[0], h_out, range(T), bias=bias[0])


def test_small_batch_graph_replay_equals_direct_launches():
    """Calls of at most 512 tokens without debug capture replay a CUDA graph with
    the caller's buffers copied in and out; results equal the direct launches."""
    L = 2
    ctx, _ = _ctx(TINY, n_layers=L, prenorm=1, seed=23)
    with ctx:
        for T in (24, 100):
            H = gen_hidden(T, TINY.d, seed=23 + T).cuda()
            bias = torch.zeros(L, T, TINY.n_experts, dtype=torch.float32)
            bias[:, :, 1] = 16.0
            bias = bias.cuda()
            outs = []
            for rep in range(3):   # first call captures, later calls replay
                h_out = torch.empty_like(H)
                y = torch.empty(T, TINY.d, dtype=torch.float32, device="cuda")
                moe.check(moe.moe_prefill(ctx.h, H, T, 0, L, bias, h_out, y), ctx.h)
                ctx.sync()
                outs.append((h_out.clone(), y.clone()))
            ref = _run_prefill(ctx, H, n_layers=L, bias=bias)   # debug capture: direct launches
            for h_out, y in outs:
                assert torch.equal(h_out.view(torch.int16), ref[0].view(torch.int16))
                assert torch.equal(y, ref[1])
        # decode steps of 20+ tokens take the same path
        H = gen_hidden(24, TINY.d, seed=29).cuda()
        h1, y1, _ = ctx.decode(H, 0, L)
        ctx.sync()
        ref = _run_prefill(ctx, H, n_layers=L)
        assert torch.equal(y1, ref[1])


def _pool_prefill_ctx(shape, n_layers, residency, path, max_tokens, seed):
    ctx = Ctx(shape, n_layers=n_layers, prenorm=1, max_tokens=max_tokens)
    if residency == moe.MOE_FILE_POOL:
        moe.check(moe.moe_set_expert_file(ctx.h, str(path), 4, 0), ctx.h)
    for l in range(n_layers):
        ctx.init_layer(l, to_device(gen_layer(shape, seed=seed, layer=l)), residency=residency)
    return ctx


@pytest.mark.parametrize("residency", [moe.MOE_HOST_POOL, moe.MOE_FILE_POOL])
@pytest.mark.parametrize("T", [3, 300])
def test_chunked_prefill_through_the_pool(residency, T, tmp_path):
    # a host-pool (or expert-file) context prefills a chunk of T tokens layer by
    # layer: route, stage the union of the picked experts once, grouped GEMMs
    # over it.  Same kernels and bytes as the resident prefill, so every output
    # is bit-identical; the staged bytes are the per-layer unions' and the
    # decode slot cache is left alone.
    L = 3
    ref, _ = _ctx(MEDIUM, n_layers=L, prenorm=1, max_tokens=T, seed=31)
    pool = _pool_prefill_ctx(MEDIUM, L, residency, tmp_path / "experts.bin", T, seed=31)
    with ref, pool:
        H = gen_hidden(T, MEDIUM.d, seed=310 + T).cuda()
        r = _run_prefill(ref, H, n_layers=L)
        p = _run_prefill(pool, H, n_layers=L)
        for a, b, name in zip(r, p, ("h_out", "y_last", "x", "ids", "gates", "y")):
            assert torch.equal(a, b), name
        # and directly against the oracle, every token's routing, sampled tokens' FFN
        wh = [gen_layer(MEDIUM, seed=31, layer=l) for l in range(L)]
        check_stack(wh, H, {"x": p[2], "ids": p[3], "gates": p[4], "y": p[5]}, p[0], MEDIUM.top_k,
                    ffn_layers=range(L), ffn_tokens=range(T) if T < 10 else (0, 1, 150, T - 1))
        _, st = moe.moe_get_stats(pool.h)
        unions = [len(np.unique(r[3][l].cpu().numpy())) for l in range(L)]
        if T == 3:
            assert max(unions) < MEDIUM.n_experts      # a partial union is staged
        assert st.staged_bytes == sum(unions) * st.expert_bytes
        assert st.hits == 0 and st.misses == 0
        if residency == moe.MOE_FILE_POOL:
            assert st.file_read_bytes == st.staged_bytes
        # a second chunk through the same arena
        H2 = gen_hidden(T, MEDIUM.d, seed=320 + T).cuda()
        r2 = _run_prefill(ref, H2, n_layers=L)
        p2 = _run_prefill(pool, H2, n_layers=L)
        for a, b in zip(r2, p2):
            assert torch.equal(a, b)


def test_chunked_prefill_needs_the_tensor_core_path():
    pool = _pool_prefill_ctx(MEDIUM, 1, moe.MOE_HOST_POOL, None, 8, seed=32)
    with pool:
        moe.check(moe.moe_test_hook(pool.h, moe.HOOK_PREFILL_TC, 0), pool.h)
        H = gen_hidden(8, MEDIUM.d, seed=32).cuda()
        h_out = torch.empty_like(H)
        assert moe.moe_prefill(pool.h, H, 8, 0, 1, None, h_out, None) == moe.MOE_EINVAL
        assert moe.moe_prefill(pool.h, H, 9, 0, 1, None, h_out, None) == moe.MOE_EINVAL   # T > max_tokens
