"""The expert file tier's host tier (pinned records in front of the file) on the
CPU: its bookkeeping is the slot cache's LRU rules one level down, so it must
reproduce the oracle's LRU, and the hand-worked LRU trace, on the stream of
slot-cache misses it is given.  The product's host-only file-tier code is
built here with the host compiler."""

import ctypes as C
import json
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_routed_expert_router_gb300", "csrc")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def shim(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("host_tier") / "libhosttier.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-x", "c++",
                           os.path.join(CSRC, "expert_file.cu"), os.path.join(os.path.dirname(__file__),
                                                                              "host_tier_shim.cpp"),
                           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-o", so, "-lpthread"])
    lib = C.CDLL(so)
    lib.shim_host_tier_lru_step.restype = C.c_int
    lib.shim_host_tier_lru_step.argtypes = [C.c_int] + [C.c_void_p] * 4 + [C.c_int, C.c_int64] + [C.c_void_p] * 4
    return lib


class Tier:
    def __init__(self, lib, n_rec, n_experts):
        self.lib, self.n = lib, n_rec
        self.eor = np.full(n_rec, -1, dtype=np.int32)
        self.lu = np.full(n_rec, -1, dtype=np.int64)
        self.roe = np.full(n_experts, -1, dtype=np.int32)
        self.touched = np.zeros(n_rec, dtype=np.int8)

    def step(self, ids, t):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        n = len(ids)
        rec, hit, ev = (np.zeros(max(n, 1), dtype=np.int32) for _ in range(3))
        p = lambda a: a.ctypes.data_as(C.c_void_p)
        r = self.lib.shim_host_tier_lru_step(self.n, p(self.eor), p(self.lu), p(self.roe), p(ids), n, t, p(rec),
                                             p(hit), p(ev), p(self.touched))
        return r, hit[:n], rec[:n], ev[:n]


def test_hand_worked_lru_trace(shim):
    with open(os.path.join(GOLDEN, "lru_hand_trace.json")) as fh:
        g = json.load(fh)
    tier = Tier(shim, g["n_slots"], g["n_experts"])
    for st in g["steps"]:
        n_new, hit, rec, ev = tier.step(st["ids"], st["t"])
        assert list(hit) == st["hit"] and list(rec) == st["slot"] and list(ev) == st["evicted"]
        assert n_new == len(st["ids"]) - sum(st["hit"])
    assert list(tier.eor) == g["final_expert_of_slot"]


@pytest.mark.parametrize("n_rec,n_experts,k", [(2, 6, 2), (5, 16, 3), (8, 32, 8)])
def test_random_miss_streams_match_the_oracle_lru(shim, n_rec, n_experts, k):
    rng = np.random.default_rng(n_rec * 100 + k)
    tier = Tier(shim, n_rec, n_experts)
    ref = oracle.LRU(n_rec)
    for t in range(400):
        m = int(rng.integers(0, k + 1))
        ids = rng.choice(n_experts, size=m, replace=False).astype(np.int32)
        n_new, hit, rec, ev = tier.step(ids, t)
        if m == 0:
            assert n_new == 0
            continue
        rh, rs, rev = ref.step(ids, t)
        assert list(hit) == list(rh) and list(rec) == list(rs) and list(ev) == list(rev), f"t={t}"
        assert list(tier.eor) == list(ref.expert_of_slot) and list(tier.lu) == list(ref.last_use)
        for r, e in enumerate(tier.eor):
            if e >= 0:
                assert tier.roe[e] == r
        assert int((tier.roe >= 0).sum()) == int((tier.eor >= 0).sum())


def test_more_requests_than_records_is_refused(shim):
    tier = Tier(shim, 2, 8)
    assert tier.step([1, 2, 3], 0)[0] == -1
