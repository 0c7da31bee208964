"""The clustered decode kernel deals a layer's units to clusters: routed unit i
to cluster i mod n_cl, and the shared expert's units evenly over the clusters
that got fewer routed units (they run before the routing is known, so they
fill the clusters that finish their routed work first).  The rule, from
kernels.h, is built here with the host compiler."""

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
                                                         (15, 8, 11, 44), (36, 4, 9, 72)])
def test_shared_units_fill_the_clusters_with_fewer_routed_units(owner, n_cl, k, groups, shared_groups):
    Ur = k * groups
    routed = [0] * n_cl
    for i in range(Ur):
        routed[i % n_cl] += 1
    shared = [0] * n_cl
    for G in range(shared_groups):
        c = owner(G, Ur, n_cl)
        assert 0 <= c < n_cl
        shared[c] += 1
    fewest = min(routed)
    light = [c for c in range(n_cl) if routed[c] == fewest]
    # every shared unit sits on a cluster with the fewest routed units ...
    assert all(shared[c] == 0 for c in range(n_cl) if routed[c] != fewest)
    # ... spread evenly over them
    got = [shared[c] for c in light]
    assert max(got) - min(got) <= 1 and sum(got) == shared_groups
