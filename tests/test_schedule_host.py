"""The clustered decode kernel deals a layer's units to clusters: routed unit i
to cluster i mod n_cl, and the shared expert's units round-robin over all
clusters, those with fewer routed units first (shared units run before the
routing is known, in the wait for it, so each cluster takes one before any
takes two).  The rule, from kernels.h, is built here with the host compiler."""

import ctypes as C
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_routed_expert_router_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"


@pytest.fixture(scope="module")
def owner(tmp_path_factory):
    if not os.path.isdir(CUDA_INC):
        pytest.skip("no CUDA headers")
    so = str(tmp_path_factory.mktemp("sched") / "libsched.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
                           os.path.join(os.path.dirname(__file__), "schedule_shim.cpp"), "-I", CSRC,
                           "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC, "-o", so])
    lib = C.CDLL(so)
    lib.shim_cluster_unit_owner_shared.restype = C.c_int
    lib.shim_cluster_unit_owner_shared.argtypes = [C.c_int, C.c_int, C.c_int]
    return lib.shim_cluster_unit_owner_shared


@pytest.mark.parametrize("n_cl,k,groups,shared_groups", [(36, 8, 11, 44), (36, 2, 2, 2), (36, 8, 9, 36),
                                                         (15, 8, 11, 44), (36, 4, 9, 72), (36, 8, 11, 30)])
def test_shared_units_spread_over_every_cluster_light_ones_first(owner, n_cl, k, groups, shared_groups):
    Ur = k * groups
    routed = [0] * n_cl
    for i in range(Ur):
        routed[i % n_cl] += 1
    shared = [0] * n_cl
    for G in range(shared_groups):
        c = owner(G, Ur, n_cl)
        assert 0 <= c < n_cl
        shared[c] += 1
    # every cluster within one shared unit of every other ...
    assert max(shared) - min(shared) <= 1 and sum(shared) == shared_groups
    # ... and the clusters holding the larger count are the lightest in routed units first
    light = {c for c in range(n_cl) if routed[c] == min(routed)}
    more = {c for c in range(n_cl) if shared[c] == max(shared)} if max(shared) != min(shared) else set()
    if more:
        assert more <= light or light <= more


def test_full_shape_layer_has_at_most_four_units_per_cluster(owner):
    # 88 routed and 44 shared units over 36 clusters: 16 clusters take 3 routed
    # + 1 shared, 8 take 2 + 2 and 12 take 2 + 1
    n_cl, Ur = 36, 8 * 11
    tot = [0] * n_cl
    for i in range(Ur):
        tot[i % n_cl] += 1
    for G in range(44):
        tot[owner(G, Ur, n_cl)] += 1
    assert max(tot) == 4 and sorted(tot).count(3) == 12
