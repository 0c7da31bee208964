"""The allocation-free routing entry point against the regular decode path.

moe_route_noalloc exists for callers that cannot call cudaMalloc where they
route (a host that reserves all device memory up front, a real-time loop that
cannot afford cudaMalloc's blocking or implicit synchronisation).  Its scratch
is a fixed device array shared by every call, so this test makes two calls in
a row and checks both against moe_decode_step's routing.  The file name sorts
last so that a run stopping at the first failure has run every other test.
"""

import numpy as np
import pytest
import torch

import bit_routed_expert_router_gb300 as moe
import oracle
from workload import FULL, Shape, gen_hidden, gen_layer

from moe_harness import GATE_RTOL, Ctx

pytestmark = pytest.mark.gpu


def _decode_routing(ctx, H, bias):
    B, k = H.shape[0], ctx.shape.top_k
    ids = torch.zeros(1, B, k, dtype=torch.int32, device="cuda")
    gs = torch.zeros(1, B, k, dtype=torch.float32, device="cuda")
    moe.check(moe.moe_set_debug(ctx.h, None, ids, gs, None, 1), ctx.h)
    ctx.decode(H, 0, 1, bias=None if bias is None else bias.unsqueeze(0))
    ctx.sync()
    moe.check(moe.moe_set_debug(ctx.h), ctx.h)
    return ids[0], gs[0]


def test_route_noalloc_matches_decode_routing_on_consecutive_calls():
    sh = FULL
    w = gen_layer(sh, seed=71, layer=0, device="cuda")
    with Ctx(sh, n_layers=1, prenorm=1) as ctx:
        ctx.init_layer(0, w)
        cases = [(32, None), (7, True)]
        for call, (B, with_bias) in enumerate(cases):
            H = (gen_hidden(B, sh.d, seed=900 + call, device="cuda").float() * (1 + call)).to(torch.bfloat16)
            bias = None
            if with_bias:
                bias = torch.zeros(B, sh.n_experts, dtype=torch.float32, device="cuda")
                bias[:, 5] = 16.0
                bias[:, 77] = 16.0
            ref_ids, ref_g = _decode_routing(ctx, H, bias)
            ids = torch.full((B, sh.top_k), -1, dtype=torch.int32, device="cuda")
            gates = torch.zeros(B, sh.top_k, dtype=torch.float32, device="cuda")
            st = moe.moe_route_noalloc(ctx.cfg, w["router_w"], H, B, bias, ids, gates)
            assert st == moe.MOE_OK
            torch.cuda.synchronize()
            assert torch.equal(ids, ref_ids), f"call {call}: ids differ"
            assert np.allclose(gates.cpu().numpy(), ref_g.cpu().numpy(), rtol=GATE_RTOL, atol=1e-7)


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    sh = FULL
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k)
    rw = torch.zeros(sh.n_experts, sh.d, dtype=torch.float16, device="cuda")
    B = moe.ROUTE_NOALLOC_MAX_B + 1
    H = torch.zeros(B, sh.d, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(B, sh.top_k, dtype=torch.int32, device="cuda")
    gates = torch.zeros(B, sh.top_k, dtype=torch.float32, device="cuda")
    assert moe.moe_route_noalloc(cfg, rw, H, B, None, ids, gates) == moe.MOE_EINVAL
    big = moe.make_config(sh.d, sh.f, sh.f_shared, 300, sh.top_k)
    assert moe.moe_route_noalloc(big, rw, H, 1, None, ids, gates) == moe.MOE_EINVAL


def test_route_noalloc_small_shape_without_norm_against_the_oracle():
    # prenorm 0, 13 experts (the last CTA's expert range runs past E), top-k 3,
    # two calls in a row through the same scratch; ids bit-exact and gates
    # against the oracle's router on x = h
    sh = Shape(d=256, f=128, f_shared=128, n_experts=13, top_k=3)
    rw = gen_layer(sh, seed=72, layer=0)["router_w"]
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, prenorm=0)
    rw_d = rw.cuda()
    for call, B in enumerate((5, 64)):
        H = gen_hidden(B, sh.d, seed=920 + call, device="cuda")
        bias = None
        if call == 1:
            bias = torch.zeros(B, sh.n_experts, dtype=torch.float32, device="cuda")
            bias[:, 12] = 16.0       # the last expert wins whenever the bias decides
        ids = torch.full((B, sh.top_k), -1, dtype=torch.int32, device="cuda")
        gates = torch.zeros(B, sh.top_k, dtype=torch.float32, device="cuda")
        assert moe.moe_route_noalloc(cfg, rw_d, H, B, bias, ids, gates) == moe.MOE_OK
        torch.cuda.synchronize()
        Hb = oracle.as_bits(H.cpu())
        for b in range(B):
            lg, st = oracle.router_logits(rw, Hb[b], None if bias is None else bias[b].cpu().numpy())
            assert st == 0
            rid = oracle.topk(lg, sh.top_k)
            assert list(ids[b].cpu().numpy()) == list(rid), f"call {call} token {b}"
            assert np.allclose(gates[b].cpu().numpy(), oracle.gates(lg, rid), rtol=GATE_RTOL, atol=1e-7)


def test_route_noalloc_rejects_misaligned_rows():
    sh = Shape(d=256, f=128, f_shared=128, n_experts=13, top_k=3)
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k)
    rw = torch.zeros(sh.n_experts * sh.d + 8, dtype=torch.float16, device="cuda")
    H = torch.zeros(2 * sh.d + 8, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(2, sh.top_k, dtype=torch.int32, device="cuda")
    gates = torch.zeros(2, sh.top_k, dtype=torch.float32, device="cuda")
    # the host rejects these before any launch
    assert moe.moe_route_noalloc(cfg, rw[1:1 + sh.n_experts * sh.d], H[:2 * sh.d], 2, None, ids, gates) == \
        moe.MOE_EINVAL
    assert moe.moe_route_noalloc(cfg, rw[:sh.n_experts * sh.d], H[4:4 + 2 * sh.d], 2, None, ids, gates) == \
        moe.MOE_EINVAL
