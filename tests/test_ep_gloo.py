"""Expert-parallel split of a layer, on CPU: G ranks each sum the 2^-32-grid
values of the units they own (their routed experts, their chunk of the shared
expert), one integer all-reduce adds the d-vectors, and the result has the
same bits as one rank summing every unit.  Two gloo ranks run the all-reduce;
the unit outputs come from the oracle."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_routed_expert_router_gb300 import ep

SHAPE = dict(d=256, f=128, f_shared=320, n_experts=8, top_k=3)   # 5 shared groups: an uneven split
N_TOK = 4


def _units(seed=7):
    """Per token: [(kind, key, output fp64 [d])] for every unit of the layer,
    plus the oracle's whole-layer y."""
    import oracle
    from workload import Shape, gen_hidden, gen_layer
    sh = Shape(**SHAPE)
    w = gen_layer(sh, seed=seed, layer=0)
    lay = oracle.Layer(w, sh.top_k)
    H = oracle.as_bits(gen_hidden(N_TOK, sh.d, seed=seed))
    s = {k: oracle.as_np(v) if k.endswith("_q") else oracle.as_bits(v) for k, v in w["shared"].items()}
    out = []
    for t in range(N_TOK):
        ids, gates, _, y_ref, st = lay.forward(H[t])
        assert st == 0
        x = oracle.bf16_bits_to_f64(H[t])
        units = []
        for j, e in enumerate(ids):
            ex = {k: v[int(e)] for k, v in w["experts"].items()}
            units.append(("routed", int(e), gates[j] * oracle.expert_ffn(ex, x)))
        n_groups = sh.f_shared // 64
        for G in range(n_groups):
            r0, r1 = 64 * G, 64 * (G + 1)
            g = oracle.matvec(s["gate_q"][r0:r1], s["gate_sb"][r0:r1], x)
            u = oracle.matvec(s["up_q"][r0:r1], s["up_sb"][r0:r1], x)
            a = np.array([oracle.gelu(v) for v in g]) * u
            dn = oracle.matvec(np.ascontiguousarray(s["down_q"][:, 32 * G:32 * (G + 1)]),
                               np.ascontiguousarray(s["down_sb"][:, G:G + 1]), a)
            units.append(("shared", G, dn))
        out.append((ids, units, y_ref))
    return out


def _grid(y):
    return np.rint(np.asarray(y, dtype=np.float64) * 2.0 ** ep.GRID_BITS).astype(np.int64)   # half to even


def _rank_sum(ids, units, rank, world):
    n_groups = SHAPE["f_shared"] // 64
    g0, g1 = ep.shared_chunks(n_groups, rank, world)
    mine = {e for _, e in ep.owned_experts(ids, rank, world)}
    v = np.zeros(SHAPE["d"], dtype=np.int64)
    for kind, key, y in units:
        if (kind == "routed" and key in mine) or (kind == "shared" and g0 <= key < g1):
            v += _grid(y)
    return v


def test_shared_chunks_sum_to_the_shared_expert():
    # pins the slicing used above: the chunks' down outputs add up to the
    # oracle's whole shared FFN
    import oracle
    from workload import Shape, gen_hidden, gen_layer
    sh = Shape(**SHAPE)
    w = gen_layer(sh, seed=7, layer=0)
    x = oracle.bf16_bits_to_f64(oracle.as_bits(gen_hidden(1, sh.d, seed=7))[0])
    whole = oracle.expert_ffn(w["shared"], x)
    s = {k: oracle.as_np(v) if k.endswith("_q") else oracle.as_bits(v) for k, v in w["shared"].items()}
    tot = np.zeros(sh.d)
    for G in range(sh.f_shared // 64):
        r0, r1 = 64 * G, 64 * (G + 1)
        g = oracle.matvec(s["gate_q"][r0:r1], s["gate_sb"][r0:r1], x)
        u = oracle.matvec(s["up_q"][r0:r1], s["up_sb"][r0:r1], x)
        a = np.array([oracle.gelu(v) for v in g]) * u
        tot += oracle.matvec(np.ascontiguousarray(s["down_q"][:, 32 * G:32 * (G + 1)]),
                             np.ascontiguousarray(s["down_sb"][:, G:G + 1]), a)
    assert np.allclose(tot, whole, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 16])
def test_every_unit_has_exactly_one_owner(world):
    E, k, n_groups = 128, 8, 44
    rng = np.random.default_rng(world)
    for _ in range(20):
        ids = rng.choice(E, size=k, replace=False)
        owners = [r for r in range(world) for _ in ep.owned_experts(ids, r, world)]
        assert len(owners) == k
        covered = []
        for r in range(world):
            g0, g1 = ep.shared_chunks(n_groups, r, world)
            covered += list(range(g0, g1))
            assert g1 - g0 in (n_groups // world, n_groups // world + 1)
        assert covered == list(range(n_groups))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for t, (ids, units, _) in enumerate(_units()):
            v = torch.from_numpy(_rank_sum(ids, units, rank, world))
            ep.allreduce_fixed(v)
            out[(rank, t)] = v.numpy().tobytes()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_give_the_single_rank_bits():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        for t, (ids, units, y_ref) in enumerate(_units()):
            single = _rank_sum(ids, units, 0, 1)
            for rank in range(world):
                got = np.frombuffer(out[(rank, t)], dtype=np.int64)
                assert np.array_equal(got, single), f"token {t} rank {rank}"
            # and the grid sum is the oracle's layer output up to the grid's rounding
            y = single.astype(np.float64) * 2.0 ** -ep.GRID_BITS
            assert np.max(np.abs(y - y_ref)) <= len(units) * 2.0 ** -(ep.GRID_BITS + 1) + 1e-12 * np.abs(y_ref).max()
