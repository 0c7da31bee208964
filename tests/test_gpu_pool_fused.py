"""The host-pool step in one launch of the clustered decode kernel
(MOE_STAGING_FUSED; TurboFieldfare, "MoE needed parallel work, reuse, and
coarse overlap": persistent workers, the cache first, the shared expert
overlapped with the reads): router, top-k, the per-layer slot-cache step,
hits from the slots and misses read from the mapped pool by the consumer
warps.  Checks: traces and cache state bit-identical to the oracle's LRU and
LFU (hand-worked trace, random Zipf traces, full shape), outputs bit-identical
to a resident context's clustered kernel and close to the oracle, staged
bytes, argument and state errors."""

import json
import os

import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, Shape, bias_from_targets, gen_hidden, gen_layer, zipf_reuse_targets

from moe_harness import Ctx, assert_ffn_close, to_device, to_host, use_decode_kernel

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fused_ctx(shape, L, n_slots, weights, policy=moe.MOE_CACHE_LRU):
    ctx = Ctx(shape, n_layers=L, prenorm=1)
    for l in range(L):
        ctx.init_layer(l, weights[l], residency=moe.MOE_HOST_POOL)
    moe.check(moe.moe_set_slots(ctx.h, n_slots), ctx.h)
    moe.check(moe.moe_set_staging(ctx.h, moe.MOE_STAGING_FUSED), ctx.h)
    if policy != moe.MOE_CACHE_LRU:
        moe.check(moe.moe_set_cache_policy(ctx.h, policy), ctx.h)
    return ctx


def _step(ctx, h, L, bias=None):
    k = ctx.shape.top_k
    tr = (moe.MoeTraceRec * (L * k))()
    h_out, y, n = ctx.decode(h, 0, L, bias=bias, trace=tr)
    assert n == L * k
    return h_out, y, [(r.layer, r.k_pos, r.expert, r.hit, r.slot, r.evicted) for r in tr]


def test_fused_hand_worked_lru_trace():
    with open(os.path.join(GOLDEN, "lru_hand_trace.json")) as fh:
        g = json.load(fh)
    sh = Shape(d=128, f=64, f_shared=64, n_experts=g["n_experts"], top_k=g["top_k"])
    w = gen_layer(sh, seed=101, layer=0)
    with _fused_ctx(sh, 1, g["n_slots"], [to_device(w)]) as ctx:
        H = gen_hidden(len(g["steps"]), sh.d, seed=101).cuda()
        for t, st in enumerate(g["steps"]):
            bias = torch.zeros(1, 1, sh.n_experts, dtype=torch.float32)
            bias[0, 0, st["ids"][0]] = 32.0     # forces the pick and its order
            bias[0, 0, st["ids"][1]] = 16.0
            _, _, rec = _step(ctx, H[t:t + 1], 1, bias.cuda())
            assert [r[2] for r in rec] == st["ids"]
            assert [r[3] for r in rec] == st["hit"]
            assert [r[4] for r in rec] == st["slot"]
            assert [r[5] for r in rec] == st["evicted"]
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.hits == g["total_hits"] and stats.misses == g["total_misses"]
        assert stats.staged_bytes == g["total_misses"] * stats.expert_bytes
        _, eos, _ = moe.moe_get_cache_state(ctx.h, 0, g["n_slots"])
        assert list(eos) == g["final_expert_of_slot"]


@pytest.mark.parametrize("policy", [moe.MOE_CACHE_LRU, moe.MOE_CACHE_LFU])
def test_fused_random_traces_match_the_oracle(policy):
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=4)
    L, N, T = 3, 6, 40
    ws = [gen_layer(sh, seed=210, layer=l) for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=210)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts))          # [T, L, E]
    with _fused_ctx(sh, L, N, [to_device(w) for w in ws], policy) as ctx:
        H = gen_hidden(T, sh.d, seed=210).cuda()
        caches = [oracle.LRU(N) if policy == moe.MOE_CACHE_LRU else oracle.LFU(N, sh.n_experts)
                  for _ in range(L)]
        xs = torch.zeros(L, 1, sh.d, dtype=torch.bfloat16, device="cuda")
        ys = torch.zeros(L, 1, sh.d, dtype=torch.float32, device="cuda")
        lays = [oracle.Layer(w, sh.top_k) for w in ws]
        for t in range(T):
            moe.check(moe.moe_set_debug(ctx.h, xs, None, None, ys, L), ctx.h)
            _, _, rec = _step(ctx, H[t:t + 1], L, bias[t].unsqueeze(1).contiguous().cuda())
            ctx.sync()
            for l in range(L):
                rows = [r for r in rec if r[0] == l]
                ids = [r[2] for r in rows]
                hit, slot, ev = caches[l].step(ids, t)
                assert [r[3] for r in rows] == list(hit), f"t={t} l={l}"
                assert [r[4] for r in rows] == list(slot), f"t={t} l={l}"
                assert [r[5] for r in rows] == list(ev), f"t={t} l={l}"
                if t % 13 == 0:
                    rid, _, _, ry, _ = lays[l].forward(oracle.as_bits(xs[l, 0]), bias[t, l].numpy())
                    assert list(rid) == ids
                    assert_ffn_close(ys[l, 0].cpu().numpy(), ry, f"t={t} l={l}")
        moe.check(moe.moe_set_debug(ctx.h), ctx.h)
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.hits + stats.misses == T * L * sh.top_k and stats.misses > 0 and stats.hits > 0
        assert stats.steps == T
        assert stats.staged_bytes == stats.misses * stats.expert_bytes
        for l in range(L):
            _, eos, lu = moe.moe_get_cache_state(ctx.h, l, N)
            assert list(eos) == list(caches[l].expert_of_slot)
            assert list(lu) == list(caches[l].last_use)


def _resident_cluster_outputs(shape, weights, H, bias, L):
    with Ctx(shape, n_layers=L, prenorm=1) as ctx:
        for l in range(L):
            ctx.init_layer(l, weights[l])
        use_decode_kernel(ctx, "cluster")
        outs = []
        for t in range(H.shape[0]):
            h_out, y, _ = ctx.decode(H[t:t + 1], 0, L, bias=None if bias is None else bias[t])
            outs.append((h_out.clone(), y.clone()))
        ctx.sync()
        return outs


@pytest.mark.parametrize("n_slots", [4, 9, 16])
def test_fused_outputs_equal_the_resident_clustered_kernel(n_slots):
    # the same kernel and arithmetic; only where the routed weights come from
    # differs (slots, or the mapped pool on a miss): bit-identical outputs
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=4)
    L, T = 3, 12
    ws = [to_device(gen_layer(sh, seed=220, layer=l)) for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=220)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts)).cuda()   # [T, L, E]
    bias = [bias[t].unsqueeze(1).contiguous() for t in range(T)]
    H = gen_hidden(T, sh.d, seed=220).cuda()
    ref = _resident_cluster_outputs(sh, ws, H, bias, L)
    with _fused_ctx(sh, L, n_slots, ws) as ctx:
        for t in range(T):
            h_out, y, _ = _step(ctx, H[t:t + 1], L, bias[t])
            assert torch.equal(h_out.view(torch.int16), ref[t][0].view(torch.int16)), f"h_out, t={t}"
            assert torch.equal(y, ref[t][1]), f"y, t={t}"


def test_fused_full_shape_three_layers():
    sh = FULL
    L, N, T = 3, 16, 6
    wd = [gen_layer(sh, seed=230, layer=l, device="cuda") for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=230)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts))
    bias_d = [bias[t].unsqueeze(1).contiguous().cuda() for t in range(T)]
    H = gen_hidden(T, sh.d, seed=230, device="cuda")
    ref = _resident_cluster_outputs(sh, wd, H, bias_d, L)
    with _fused_ctx(sh, L, N, wd) as ctx:
        hosts = [to_host(w) for w in wd]
        del wd
        lrus = [oracle.LRU(N) for _ in range(L)]
        xs = torch.zeros(L, 1, sh.d, dtype=torch.bfloat16, device="cuda")
        ys = torch.zeros(L, 1, sh.d, dtype=torch.float32, device="cuda")
        for t in range(T):
            moe.check(moe.moe_set_debug(ctx.h, xs, None, None, ys, L), ctx.h)
            h_out, y, rec = _step(ctx, H[t:t + 1], L, bias_d[t])
            ctx.sync()
            assert torch.equal(y, ref[t][1]), f"y, t={t}"
            for l in range(L):
                rows = [r for r in rec if r[0] == l]
                hit, slot, ev = lrus[l].step([r[2] for r in rows], t)
                assert [r[3] for r in rows] == list(hit)
                assert [r[4] for r in rows] == list(slot)
                assert [r[5] for r in rows] == list(ev)
            if t in (0, T - 1):
                l = t % L
                lay = oracle.Layer(hosts[l], sh.top_k)
                rid, _, _, ry, _ = lay.forward(oracle.as_bits(xs[l, 0]), bias[t, l].numpy())
                assert list(rid) == [r[2] for r in rec if r[0] == l]
                assert_ffn_close(ys[l, 0].cpu().numpy(), ry, f"t={t} l={l}")
        moe.check(moe.moe_set_debug(ctx.h), ctx.h)
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.staged_bytes == stats.misses * stats.expert_bytes > 0


def test_fused_staging_state_errors(tmp_path):
    sh = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2)
    w = to_device(gen_layer(sh, seed=240, layer=0))
    H = gen_hidden(4, sh.d, seed=240).cuda()
    with _fused_ctx(sh, 1, 2, [w]) as ctx:
        assert moe.moe_set_staging(ctx.h, 3) == moe.MOE_EINVAL
        ys = [ctx.decode(H[t:t + 1], 0, 1)[1].clone() for t in range(4)]   # no trace: returns at once
        ctx.sync()
        # back to host staging (cache emptied): the per-layer kernels decide the same way
        moe.check(moe.moe_set_staging(ctx.h, moe.MOE_STAGING_HOST), ctx.h)
        moe.check(moe.moe_set_staging(ctx.h, moe.MOE_STAGING_FUSED), ctx.h)
        for t in range(4):
            assert torch.equal(ctx.decode(H[t:t + 1], 0, 1)[1], ys[t])
    res = Ctx(sh, n_layers=1)
    with res:
        res.init_layer(0, w)
        assert moe.moe_set_staging(res.h, moe.MOE_STAGING_FUSED) == moe.MOE_ESTATE   # resident context
    fctx = Ctx(sh, n_layers=1, prenorm=1)
    with fctx:
        moe.check(moe.moe_set_expert_file(fctx.h, str(tmp_path / "e.bin"), 2, 0), fctx.h)
        fctx.init_layer(0, w, residency=moe.MOE_FILE_POOL)
        assert moe.moe_set_staging(fctx.h, moe.MOE_STAGING_FUSED) == moe.MOE_ESTATE  # file reads are host I/O
