"""Host-pool contexts: the per-layer LRU expert-slot cache (TurboFieldfare,
"MoE needed parallel work, reuse, and coarse overlap": a bounded per-layer
cache of routed experts; goinfer, "When the model doesn't fit": LRU slots).

Checks: the cache trace and counters are bit-identical to the oracle's LRU;
misses are staged from the pinned pool; outputs do not depend on the slot
count; host-side failures (argument errors, budget, a failed staging copy, a
timed-out wait) are reported and poison the context as documented."""

import json
import os

import numpy as np
import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, Shape, bias_from_targets, gen_hidden, gen_layer, zipf_reuse_targets

from moe_harness import Ctx, assert_ffn_close, capture, check_stack, end_capture, to_device, to_host

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pool_ctx(shape, L, n_slots, weights, prenorm=1):
    ctx = Ctx(shape, n_layers=L, prenorm=prenorm)
    for l in range(L):
        ctx.init_layer(l, weights[l], residency=moe.MOE_HOST_POOL)
    moe.check(moe.moe_set_slots(ctx.h, n_slots), ctx.h)
    return ctx


def _decode_trace(ctx, h, L, bias):
    k = ctx.shape.top_k
    tr = (moe.MoeTraceRec * (L * k))()
    _, y, n = ctx.decode(h, 0, L, bias=bias, trace=tr)
    assert n == L * k
    return y, [(r.layer, r.k_pos, r.expert, r.hit, r.slot, r.evicted) for r in tr]


def test_hand_worked_lru_trace():
    with open(os.path.join(GOLDEN, "lru_hand_trace.json")) as fh:
        g = json.load(fh)
    sh = Shape(d=128, f=64, f_shared=64, n_experts=g["n_experts"], top_k=g["top_k"])
    w = gen_layer(sh, seed=101, layer=0)
    with _pool_ctx(sh, 1, g["n_slots"], [to_device(w)]) as ctx:
        H = gen_hidden(len(g["steps"]), sh.d, seed=101).cuda()
        for t, st in enumerate(g["steps"]):
            bias = torch.zeros(1, 1, sh.n_experts, dtype=torch.float32)
            bias[0, 0, st["ids"][0]] = 32.0     # forces the pick and its order
            bias[0, 0, st["ids"][1]] = 16.0
            _, rec = _decode_trace(ctx, H[t:t + 1], 1, bias.cuda())
            assert [r[2] for r in rec] == st["ids"]
            assert [r[3] for r in rec] == st["hit"]
            assert [r[4] for r in rec] == st["slot"]
            assert [r[5] for r in rec] == st["evicted"]
        st_, stats = moe.moe_get_stats(ctx.h)
        assert stats.hits == g["total_hits"] and stats.misses == g["total_misses"]
        assert stats.staged_bytes == g["total_misses"] * stats.expert_bytes
        _, eos, _ = moe.moe_get_cache_state(ctx.h, 0, g["n_slots"])
        assert list(eos) == g["final_expert_of_slot"]


def test_random_traces_match_oracle_lru_and_outputs_match_oracle():
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=4)
    L, N, T = 3, 6, 40
    ws = [gen_layer(sh, seed=110, layer=l) for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=110)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts))          # [T, L, E]
    with _pool_ctx(sh, L, N, [to_device(w) for w in ws]) as ctx:
        H = gen_hidden(T, sh.d, seed=110).cuda()
        lrus = [oracle.LRU(N) for _ in range(L)]
        xs = torch.zeros(L, 1, sh.d, dtype=torch.bfloat16, device="cuda")
        ys = torch.zeros(L, 1, sh.d, dtype=torch.float32, device="cuda")
        lays = [oracle.Layer(w, sh.top_k) for w in ws]
        for t in range(T):
            moe.check(moe.moe_set_debug(ctx.h, xs, None, None, ys, L), ctx.h)
            _, rec = _decode_trace(ctx, H[t:t + 1], L, bias[t].unsqueeze(1).contiguous().cuda())
            ctx.sync()
            for l in range(L):
                rows = [r for r in rec if r[0] == l]
                ids = [r[2] for r in rows]
                hit, slot, ev = lrus[l].step(ids, t)
                assert [r[3] for r in rows] == list(hit), f"t={t} l={l}"
                assert [r[4] for r in rows] == list(slot), f"t={t} l={l}"
                assert [r[5] for r in rows] == list(ev), f"t={t} l={l}"
                if t % 13 == 0:
                    rid, _, _, ry, _ = lays[l].forward(oracle.as_bits(xs[l, 0]), bias[t, l].numpy())
                    assert list(rid) == ids
                    assert_ffn_close(ys[l, 0].cpu().numpy(), ry, f"t={t} l={l}")
        moe.check(moe.moe_set_debug(ctx.h), ctx.h)
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.hits + stats.misses == T * L * sh.top_k
        assert stats.steps == T
        assert stats.staged_bytes == stats.misses * stats.expert_bytes
        for l in range(L):
            _, eos, lu = moe.moe_get_cache_state(ctx.h, l, N)
            assert list(eos) == list(lrus[l].expert_of_slot)
            assert list(lu) == list(lrus[l].last_use)


def test_outputs_do_not_depend_on_slot_count():
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=4)
    L, T = 2, 12
    ws = [gen_layer(sh, seed=120, layer=l) for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=120)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts)).cuda()
    H = gen_hidden(T, sh.d, seed=120).cuda()
    outs = {}
    for n_slots in (4, 7, 16, None):
        if n_slots is None:
            ctx = Ctx(sh, n_layers=L, prenorm=1)
            for l in range(L):
                ctx.init_layer(l, to_device(ws[l]))
            moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_PERSISTENT, 0), ctx.h)
        else:
            ctx = _pool_ctx(sh, L, n_slots, [to_device(w) for w in ws])
        with ctx:
            res = []
            for t in range(T):
                h_out, y, _ = ctx.decode(H[t:t + 1], 0, L, bias=bias[t].unsqueeze(1).contiguous())
                res.append((h_out.clone(), y.clone()))
            ctx.sync()
            outs[n_slots] = res
    for n_slots in (7, 16, None):
        for t in range(T):
            assert torch.equal(outs[n_slots][t][0], outs[4][t][0]), f"h_out differs, N={n_slots} t={t}"
            assert torch.equal(outs[n_slots][t][1], outs[4][t][1]), f"y differs, N={n_slots} t={t}"


@pytest.mark.parametrize("staging", [moe.MOE_STAGING_HOST, moe.MOE_STAGING_DEVICE])
def test_full_shape_pool_three_layers(staging):
    sh = FULL
    L, N, T = 3, 16, 6
    wd = [gen_layer(sh, seed=130, layer=l, device="cuda") for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=130)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts))
    with _pool_ctx(sh, L, N, wd) as ctx:
        moe.check(moe.moe_set_staging(ctx.h, staging), ctx.h)
        hosts = [to_host(w) for w in wd]
        del wd
        H = gen_hidden(T, sh.d, seed=130, device="cuda")
        lrus = [oracle.LRU(N) for _ in range(L)]
        xs = torch.zeros(L, 1, sh.d, dtype=torch.bfloat16, device="cuda")
        ys = torch.zeros(L, 1, sh.d, dtype=torch.float32, device="cuda")
        for t in range(T):
            moe.check(moe.moe_set_debug(ctx.h, xs, None, None, ys, L), ctx.h)
            _, rec = _decode_trace(ctx, H[t:t + 1], L, bias[t].unsqueeze(1).contiguous().cuda())
            ctx.sync()
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


def _small_pool(n_slots=4):
    sh = Shape(d=128, f=64, f_shared=64, n_experts=8, top_k=2)
    ws = [to_device(gen_layer(sh, seed=140, layer=0))]
    return sh, _pool_ctx(sh, 1, n_slots, ws)


def test_argument_and_state_errors():
    sh, ctx = _small_pool()
    with ctx:
        assert moe.moe_set_slots(ctx.h, 1) == moe.MOE_EINVAL          # fewer than top_k
        assert moe.moe_set_slots(ctx.h, 9) == moe.MOE_EINVAL          # more than n_experts
        H = gen_hidden(2, sh.d, seed=140).cuda()
        out = torch.empty_like(H)
        st, _ = moe.moe_decode_step(ctx.h, H, 2, 0, 1, None, out)     # one token per call
        assert st == moe.MOE_EINVAL
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 2, None, out)     # layer range
        assert st == moe.MOE_EINVAL
        ctx.decode(H[:1])                                              # still usable
    with Ctx(sh, n_layers=1) as res:
        res.init_layer(0, to_device(gen_layer(sh, seed=141, layer=0)))
        assert moe.moe_set_slots(res.h, 4) == moe.MOE_ESTATE           # resident context


def test_budget_is_checked_before_allocating():
    sh, ctx = _small_pool(4)
    with ctx:
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_FREE_BYTES, 1 << 20), ctx.h)
        assert moe.moe_set_slots(ctx.h, 8) == moe.MOE_ENOMEM
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_FREE_BYTES, -1), ctx.h)
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.n_slots == 4                                      # unchanged
        H = gen_hidden(1, sh.d, seed=142).cuda()
        ctx.decode(H)                                                  # still usable


def test_failed_staging_copy_poisons_the_context():
    sh, ctx = _small_pool(4)
    with ctx:
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_FAIL_NEXT_COPY, 1), ctx.h)
        H = gen_hidden(1, sh.d, seed=143).cuda()
        out = torch.empty_like(H)
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 1, None, out)
        assert st == moe.MOE_ECUDA                                     # first token misses
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 1, None, out)
        assert st == moe.MOE_ESTATE
        assert moe.moe_sync(ctx.h) == moe.MOE_ESTATE
        torch.cuda.synchronize()


def test_timed_out_wait_poisons_the_context():
    sh, ctx = _small_pool(4)
    with ctx:
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_WAIT_LIMIT_US, -1), ctx.h)
        H = gen_hidden(1, sh.d, seed=144).cuda()
        out = torch.empty_like(H)
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 1, None, out)
        assert st == moe.MOE_ETIMEOUT
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 1, None, out)
        assert st == moe.MOE_ESTATE
        torch.cuda.synchronize()


def test_reset_cache_empties_slots():
    sh, ctx = _small_pool(4)
    with ctx:
        H = gen_hidden(3, sh.d, seed=145).cuda()
        for t in range(3):
            ctx.decode(H[t:t + 1])
        moe.check(moe.moe_reset_cache(ctx.h), ctx.h)
        _, eos, lu = moe.moe_get_cache_state(ctx.h, 0, 4)
        assert list(eos) == [-1] * 4 and list(lu) == [-1] * 4
        _, stats = moe.moe_get_stats(ctx.h)
        assert stats.hits == 0 and stats.misses == 0 and stats.steps == 0


# ----------------------------------------------------------------- LFU eviction

def test_hand_worked_lfu_traces():
    with open(os.path.join(GOLDEN, "lfu_hand_traces.json")) as fh:
        g = json.load(fh)
    for ti, tr in enumerate(g["traces"]):
        sh = Shape(d=128, f=64, f_shared=64, n_experts=tr["n_experts"], top_k=tr["top_k"])
        w = gen_layer(sh, seed=150 + ti, layer=0)
        with _pool_ctx(sh, 1, tr["n_slots"], [to_device(w)]) as ctx:
            moe.check(moe.moe_set_cache_policy(ctx.h, moe.MOE_CACHE_LFU), ctx.h)
            H = gen_hidden(len(tr["steps"]), sh.d, seed=150 + ti).cuda()
            for t, st in enumerate(tr["steps"]):
                bias = torch.zeros(1, 1, sh.n_experts, dtype=torch.float32)
                for j, e in enumerate(st["ids"]):
                    bias[0, 0, e] = 32.0 - 16.0 * j     # forces the picks and their order
                _, rec = _decode_trace(ctx, H[t:t + 1], 1, bias.cuda())
                assert [r[2] for r in rec] == st["ids"]
                assert [r[3] for r in rec] == st["hit"], (ti, t)
                assert [r[4] for r in rec] == st["slot"], (ti, t)
                assert [r[5] for r in rec] == st["evicted"], (ti, t)
            _, stats = moe.moe_get_stats(ctx.h)
            assert stats.hits == tr["total_hits"] and stats.misses == tr["total_misses"]
            _, eos, _ = moe.moe_get_cache_state(ctx.h, 0, tr["n_slots"])
            assert list(eos) == tr["final_expert_of_slot"]


def test_random_traces_match_oracle_lfu():
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=4)
    L, N, T = 2, 6, 60
    ws = [gen_layer(sh, seed=160, layer=l) for l in range(L)]
    tg = zipf_reuse_targets(T, L, sh.n_experts, sh.top_k, seed=160)
    bias = torch.from_numpy(bias_from_targets(tg, sh.n_experts))          # [T, L, E]
    with _pool_ctx(sh, L, N, [to_device(w) for w in ws]) as ctx:
        moe.check(moe.moe_set_cache_policy(ctx.h, moe.MOE_CACHE_LFU), ctx.h)
        H = gen_hidden(T, sh.d, seed=160).cuda()
        lfus = [oracle.LFU(N, sh.n_experts) for _ in range(L)]
        for t in range(T):
            _, rec = _decode_trace(ctx, H[t:t + 1], L, bias[t].unsqueeze(1).contiguous().cuda())
            for l in range(L):
                rows = [r for r in rec if r[0] == l]
                hit, slot, ev = lfus[l].step([r[2] for r in rows], t)
                assert [r[3] for r in rows] == list(hit), f"t={t} l={l}"
                assert [r[4] for r in rows] == list(slot), f"t={t} l={l}"
                assert [r[5] for r in rows] == list(ev), f"t={t} l={l}"
        ctx.sync()
        for l in range(L):
            _, eos, lu = moe.moe_get_cache_state(ctx.h, l, N)
            assert list(eos) == list(lfus[l].expert_of_slot)
            assert list(lu) == list(lfus[l].last_use)
        # switching the policy empties the cache
        moe.check(moe.moe_set_cache_policy(ctx.h, moe.MOE_CACHE_LRU), ctx.h)
        _, eos, _ = moe.moe_get_cache_state(ctx.h, 0, N)
        assert list(eos) == [-1] * N


def test_cache_policy_argument_errors():
    sh = Shape(d=128, f=64, f_shared=64, n_experts=8, top_k=2)
    w = to_device(gen_layer(sh, seed=170, layer=0))
    with _pool_ctx(sh, 1, 4, [w]) as ctx:
        assert moe.moe_set_cache_policy(ctx.h, 7) == moe.MOE_EINVAL
    res = Ctx(sh, n_layers=1)
    with res:
        res.init_layer(0, w)
        assert moe.moe_set_cache_policy(res.h, moe.MOE_CACHE_LFU) == moe.MOE_ESTATE


def _file_run(shape, L, ws, H, n_slots, path=None, n_host=0, staging=None):
    ctx = Ctx(shape, n_layers=L, prenorm=1)
    with ctx:
        if path is not None:
            moe.check(moe.moe_set_expert_file(ctx.h, str(path), 4, 65536), ctx.h)
        for l in range(L):
            ctx.init_layer(l, ws[l], residency=moe.MOE_FILE_POOL if path is not None else moe.MOE_HOST_POOL)
        if n_host:
            moe.check(moe.moe_set_file_cache(ctx.h, n_host), ctx.h)
        moe.check(moe.moe_set_slots(ctx.h, n_slots), ctx.h)
        if staging is not None:
            moe.check(moe.moe_set_staging(ctx.h, staging), ctx.h)
        ys, trs = [], []
        for t in range(H.shape[0]):
            y, tr = _decode_trace(ctx, H[t:t + 1], L, None)
            ys.append(y.clone())
            trs.append(tr)
        ctx.sync()
        status, st = moe.moe_get_stats(ctx.h)
        moe.check(status, ctx.h)
        return torch.cat(ys), trs, st


def test_file_pool_matches_host_pool(tmp_path):
    # the expert file tier (misses read by parallel pread into pinned staging)
    # stages the same bytes as the pinned host pool: identical traces and outputs
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=2)
    L = 3
    ws = [to_device(gen_layer(sh, seed=150, layer=l)) for l in range(L)]
    H = gen_hidden(12, sh.d, seed=150).cuda()
    y_h, tr_h, st_h = _file_run(sh, L, ws, H, 3)
    path = tmp_path / "experts.bin"
    y_f, tr_f, st_f = _file_run(sh, L, ws, H, 3, path)
    assert tr_h == tr_f
    assert torch.equal(y_h, y_f)
    assert st_f.misses == st_h.misses > 0 and st_f.staged_bytes == st_h.staged_bytes
    assert st_f.host_pool_bytes == 0 and st_h.host_pool_bytes > 0
    rec = (st_h.expert_bytes + 4095) // 4096 * 4096
    assert os.path.getsize(path) == (L * sh.n_experts - 1) * rec + st_h.expert_bytes


@pytest.mark.parametrize("tier", ["host", "file", "file+host"])
def test_pool_outputs_match_oracle(tier, tmp_path):
    # a slot cache smaller than the working set, misses staged from the pinned
    # pool or read from the expert file (with or without the pinned host tier):
    # every layer's logits, ids, gates, FFN output and residual against the oracle
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=2)
    L, N, NH, T = 3, 3, 6, 10
    wh = [gen_layer(sh, seed=154, layer=l) for l in range(L)]
    ctx = Ctx(sh, n_layers=L, prenorm=1)
    with ctx:
        if tier != "host":
            moe.check(moe.moe_set_expert_file(ctx.h, str(tmp_path / "experts.bin"), 4, 65536), ctx.h)
        for l in range(L):
            ctx.init_layer(l, to_device(wh[l]), residency=moe.MOE_HOST_POOL if tier == "host" else moe.MOE_FILE_POOL)
        if tier == "file+host":
            moe.check(moe.moe_set_file_cache(ctx.h, NH), ctx.h)
        moe.check(moe.moe_set_slots(ctx.h, N), ctx.h)
        H = gen_hidden(T, sh.d, seed=154).cuda()
        for t in range(T):
            cap = capture(ctx, L, 1, logits=True)
            h_out, _, _ = ctx.decode(H[t:t + 1], 0, L)
            ctx.sync()
            end_capture(ctx)
            check_stack(wh, H[t:t + 1], cap, h_out, sh.top_k, ffn_layers=range(L))
        _, st = moe.moe_get_stats(ctx.h)
        assert st.misses > 0 and st.hits > 0
        if tier == "file":
            assert st.file_read_bytes == st.misses * st.expert_bytes
        if tier == "file+host":
            assert st.host_tier_hits > 0


def test_file_pool_state_and_io_errors(tmp_path):
    sh = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2)
    w = to_device(gen_layer(sh, seed=151, layer=0))
    ctx = Ctx(sh, n_layers=1, prenorm=1)
    with ctx:
        # a file-pool layer needs the file first; bad arguments are rejected
        assert moe.moe_init_layer(ctx.h, 0, w["router_w"], w["experts"], w["shared"],
                                  moe.MOE_FILE_POOL) == moe.MOE_ESTATE
        assert moe.moe_set_expert_file(ctx.h, str(tmp_path / "e.bin"), 0, 0) == moe.MOE_EINVAL
        assert moe.moe_set_expert_file(ctx.h, str(tmp_path / "e.bin"), 4, 1000) == moe.MOE_EINVAL
        assert moe.moe_set_expert_file(ctx.h, str(tmp_path / "no_dir" / "e.bin"), 4, 0) == moe.MOE_EINVAL
        moe.check(moe.moe_set_expert_file(ctx.h, str(tmp_path / "e.bin"), 4, 0), ctx.h)
        assert moe.moe_set_expert_file(ctx.h, str(tmp_path / "e2.bin"), 4, 0) == moe.MOE_EINVAL   # once only
        ctx.init_layer(0, w, residency=moe.MOE_FILE_POOL)
        moe.check(moe.moe_set_slots(ctx.h, 2), ctx.h)
        # a file cut short under the context: the next miss is a short read, MOE_EIO, and poisons
        os.truncate(tmp_path / "e.bin", 4096)
        H = gen_hidden(1, sh.d, seed=151).cuda()
        h_out = torch.empty_like(H)
        st, _ = moe.moe_decode_step(ctx.h, H, 1, 0, 1, None, h_out, None, None, None)
        assert st == moe.MOE_EIO
        assert moe.moe_set_slots(ctx.h, 2) == moe.MOE_ESTATE      # poisoned


def test_file_host_tier_follows_oracle_lru(tmp_path):
    # two-tier cache (file -> pinned host records -> HBM slots): a slot-cache
    # miss that the host tier holds is copied from it, any other is read from
    # the file; the host tier runs the oracle's LRU rules over each step's miss
    # list (top-k order).  Slot traces and outputs stay those of the host pool.
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=2)
    L, N, NH = 3, 3, 6
    ws = [to_device(gen_layer(sh, seed=152, layer=l)) for l in range(L)]
    H = gen_hidden(16, sh.d, seed=152).cuda()
    y_h, tr_h, st_h = _file_run(sh, L, ws, H, N)
    y_f, tr_f, st_f = _file_run(sh, L, ws, H, N, tmp_path / "experts.bin", n_host=NH)
    assert tr_h == tr_f
    assert torch.equal(y_h, y_f)
    host = [oracle.LRU(NH) for _ in range(L)]
    hits = reads = 0
    for t, tr in enumerate(tr_f):
        for l in range(L):
            miss = [r[2] for r in sorted(r for r in tr if r[0] == l) if not r[3]]
            if miss:
                h, _, _ = host[l].step(miss, t)
                hits += int(h.sum())
                reads += len(miss) - int(h.sum())
    assert st_f.misses == st_h.misses == hits + reads
    assert st_f.host_tier_hits == hits > 0 and reads > 0
    assert st_f.file_read_bytes == reads * st_f.expert_bytes
    rec = (st_f.expert_bytes + 4095) // 4096 * 4096
    assert st_f.host_tier_bytes == L * NH * rec


def test_file_host_tier_argument_errors(tmp_path):
    sh = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2)
    w = to_device(gen_layer(sh, seed=153, layer=0))
    with _pool_ctx(sh, 1, 4, [w]) as ctx:
        assert moe.moe_set_file_cache(ctx.h, 4) == moe.MOE_ESTATE      # host pool: no expert file
    ctx = Ctx(sh, n_layers=1, prenorm=1)
    with ctx:
        moe.check(moe.moe_set_expert_file(ctx.h, str(tmp_path / "e.bin"), 2, 0), ctx.h)
        ctx.init_layer(0, w, residency=moe.MOE_FILE_POOL)
        assert moe.moe_set_file_cache(ctx.h, 1) == moe.MOE_EINVAL       # below top_k
        assert moe.moe_set_file_cache(ctx.h, 9) == moe.MOE_EINVAL       # above n_experts
        moe.check(moe.moe_set_file_cache(ctx.h, 8), ctx.h)
        moe.check(moe.moe_set_file_cache(ctx.h, 0), ctx.h)              # removed again
        moe.check(moe.moe_set_slots(ctx.h, 2), ctx.h)
        _, st = moe.moe_get_stats(ctx.h)
        assert st.host_tier_bytes == 0


def test_device_staging_matches_host_staging():
    # device-driven staging (a kernel copies the misses from the mapped host
    # pool, no host round trip per layer) makes the same cache decisions and
    # outputs as the host-driven copies, bit for bit
    sh = Shape(d=256, f=128, f_shared=128, n_experts=16, top_k=2)
    L = 3
    ws = [to_device(gen_layer(sh, seed=154, layer=l)) for l in range(L)]
    H = gen_hidden(16, sh.d, seed=154).cuda()
    y_h, tr_h, st_h = _file_run(sh, L, ws, H, 3)
    y_d, tr_d, st_d = _file_run(sh, L, ws, H, 3, staging=moe.MOE_STAGING_DEVICE)
    assert tr_h == tr_d
    assert torch.equal(y_h, y_d)
    assert st_d.hits == st_h.hits and st_d.misses == st_h.misses > 0
    assert st_d.staged_bytes == st_h.staged_bytes == st_h.misses * st_h.expert_bytes


def test_device_staging_without_trace_and_errors(tmp_path):
    sh = Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2)
    w = to_device(gen_layer(sh, seed=155, layer=0))
    H = gen_hidden(4, sh.d, seed=155).cuda()
    with _pool_ctx(sh, 1, 2, [w]) as ctx:
        assert moe.moe_set_staging(ctx.h, 3) == moe.MOE_EINVAL
        moe.check(moe.moe_set_staging(ctx.h, moe.MOE_STAGING_DEVICE), ctx.h)
        ys = [ctx.decode(H[t:t + 1], 0, 1)[1].clone() for t in range(4)]   # no trace: returns at once
        ctx.sync()
        moe.check(moe.moe_set_staging(ctx.h, moe.MOE_STAGING_HOST), ctx.h)
        for t in range(4):
            assert torch.equal(ctx.decode(H[t:t + 1], 0, 1)[1], ys[t])
    res = Ctx(sh, n_layers=1)
    with res:
        res.init_layer(0, w)
        assert moe.moe_set_staging(res.h, moe.MOE_STAGING_DEVICE) == moe.MOE_ESTATE   # resident context
    fctx = Ctx(sh, n_layers=1, prenorm=1)
    with fctx:
        moe.check(moe.moe_set_expert_file(fctx.h, str(tmp_path / "e.bin"), 2, 0), fctx.h)
        fctx.init_layer(0, w, residency=moe.MOE_FILE_POOL)
        assert moe.moe_set_staging(fctx.h, moe.MOE_STAGING_DEVICE) == moe.MOE_ESTATE  # file reads are host I/O


def test_host_read_rate():
    # plain loads of pinned host memory from every SM (the pool line's link peak);
    # pageable memory is refused
    buf = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    st, gbs = moe.moe_host_read_rate(buf, buf.numel(), 3, torch.cuda.current_stream())
    assert st == moe.MOE_OK and 1.0 < gbs < 2000.0, (st, gbs)
    pageable = torch.empty(1 << 20, dtype=torch.uint8)
    st, _ = moe.moe_host_read_rate(pageable, pageable.numel(), 1, None)
    assert st == moe.MOE_EINVAL

