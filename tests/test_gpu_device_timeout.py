"""A device-side wait that runs out.  Every wait of the two persistent decode
kernels is bounded by a cycle limit the host sets (test hook 10).  With a
limit of one cycle the first wait that is not already satisfied gives up: the
kernel sets the abort flag and the error word, every CTA drains its own copies
in flight and leaves, and the last CTA out puts the launch words back at rest.
The host then sees MOE_ETIMEOUT from moe_sync, the context is poisoned, the
device is still usable, and a fresh context decodes correctly.  No wait is left
unbounded and nothing faults: the failure is a limit that runs out."""

import pytest
import torch

import bit_routed_expert_router_gb300 as moe
from workload import TINY, gen_hidden, gen_layer

from moe_harness import Ctx, capture, check_stack, end_capture, to_device, use_decode_kernel

pytestmark = pytest.mark.gpu

L = 8


def _ctx(ws, kernel):
    ctx = Ctx(TINY, n_layers=L, prenorm=1)
    for l in range(L):
        ctx.init_layer(l, to_device(ws[l]))
    use_decode_kernel(ctx, kernel)
    return ctx


@pytest.mark.parametrize("kernel", ["cluster", "per_sm"])
def test_device_wait_that_runs_out_poisons_only_its_context(kernel):
    ws = [gen_layer(TINY, seed=95, layer=l) for l in range(L)]
    H = gen_hidden(3, TINY.d, seed=95).cuda()
    with _ctx(ws, kernel) as ctx:
        ctx.decode(H[0:1])
        ctx.sync()
        assert moe.moe_test_hook(ctx.h, moe.HOOK_AT_REST, 0) == moe.MOE_OK
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_SPIN_LIMIT, 1), ctx.h)
        h_out = torch.empty_like(H[1:2])
        st, _ = moe.moe_decode_step(ctx.h, H[1:2], 1, 0, L, None, h_out, None, None, None)
        assert st == moe.MOE_OK                       # the launch itself is fine
        st = moe.moe_sync(ctx.h)
        assert st == moe.MOE_ETIMEOUT, moe.status_name(st)
        assert "wait" in moe.moe_last_error(ctx.h)
        st, _ = moe.moe_decode_step(ctx.h, H[1:2], 1, 0, L, None, h_out, None, None, None)
        assert st == moe.MOE_ESTATE                   # poisoned
        # the aborted launch left its exit counter, abort flag, counters and sums at rest
        assert moe.moe_test_hook(ctx.h, moe.HOOK_AT_REST, 0) == moe.MOE_OK
        if kernel == "cluster":
            # and recorded which wait ran out first (a site and a CTA of the grid)
            import ctypes
            word = ctypes.c_uint32(0)
            assert moe.moe_test_hook(ctx.h, moe.HOOK_WAIT_DIAG, ctypes.addressof(word)) == moe.MOE_OK
            assert 1 <= word.value >> 16 <= 16, hex(word.value)
    torch.cuda.synchronize()                          # the device still answers
    with _ctx(ws, kernel) as ctx:
        for t in range(3):
            cap = capture(ctx, L, 1, logits=True)
            h_out, _, _ = ctx.decode(H[t:t + 1])
            ctx.sync()
            end_capture(ctx)
            check_stack(ws, H[t:t + 1], cap, h_out, TINY.top_k, ffn_layers=(0, L - 1))


def test_default_limit_is_restored():
    ws = [gen_layer(TINY, seed=96, layer=l) for l in range(L)]
    H = gen_hidden(1, TINY.d, seed=96).cuda()
    with _ctx(ws, "cluster") as ctx:
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_SPIN_LIMIT, 1), ctx.h)
        moe.check(moe.moe_test_hook(ctx.h, moe.HOOK_SPIN_LIMIT, 0), ctx.h)   # back to the default
        for _ in range(3):
            ctx.decode(H)
        ctx.sync()
        assert moe.moe_test_hook(ctx.h, moe.HOOK_AT_REST, 0) == moe.MOE_OK
