// Clustered persistent decode kernel: one cooperative launch runs a B = 1 token
// through every layer of a resident context, on clusters of four CTAs.
//
// The routed-MoE FFN of a layer is cut along the groups of 64 intermediate
// rows that the int4 quantisation already defines.  A unit is (source, group):
// the source is the shared expert or one of the top-k positions, and the unit
// holds the group's 64 gate and 64 up rows (eight gate/up tiles of 8 + 8 rows)
// and the matching 64-column block of the down projection (all d output rows,
// one int4 group).  The down product of a unit needs only the unit's own 64
// values of a = GELU(gate) * up, so a cluster that owns whole units never waits
// on another cluster between gate/up and down:
//
//   CTA rank r of the cluster computes gate/up tiles 2r and 2r + 1 of the unit
//   (16 intermediate rows), writes their 16 values of a (as bf16 hi + lo
//   mma.sync B fragments) and their sums into the shared memory of every CTA of
//   the cluster (distributed shared memory), and arrives on each CTA's
//   mbarrier for the unit; then it multiplies output rows [r d/4, (r+1) d/4) of
//   the unit's down block by the 64 values once all eight tiles have arrived.
//
// The grid-wide exchanges left per layer are the router logits (one router
// row per CTA, published with a per-launch tag inside each 64-bit word, so a
// reader polls the data itself) and the layer output: each CTA sums its units'
// down partials (gate-weighted, fixed order) for its d/4 rows, rounds them onto
// a 2^-32 fixed-point grid and adds them into the layer's int64 output vector
// with one bulk reduction (TMA engine, integer adds in L2, so the result does
// not depend on the order in which CTAs arrive), then bumps the layer's
// counter.  Every CTA then reads the vector, adds it to its own copy of the
// residual stream and normalises it for the next layer.
//
// Roles per CTA (18 warps):
//   warp 0, lane 0 (producer): the router row, then every stage of the CTA's
//     units (gate/up tiles by 1-D bulk copy, down slices by a 3-D TMA tile load
//     that gathers one group of d/64 consecutive 16-row tiles) into a ring of
//     six shared-memory slots; routing-independent units (shared expert) come
//     first, routed units after the top-k is known.
//   warps 1..16 (consumers): four quads of four warps; stage u of the CTA goes
//     to quad u mod 4 (gate/up: 11-group chunks per warp, the last warp of the
//     quad runs the epilogue and the push; down: row tiles split by warp).
//   warp 17 (top-k): polls the layer's tagged logits, takes the top-k and the
//     softmax gates and releases the producer.
// Every wait is bounded and gives up through an abort flag and the device
// error word (MOE_ETIMEOUT from moe_sync); the last CTA to leave zeroes the
// counters for the next launch.
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

#include <cstddef>

namespace moe {

namespace {

constexpr int kCl = kCCluster;                    // CTAs per cluster
constexpr int kNC = 16;                           // consumer warps
constexpr int kQW = 4;                            // warps per quad (one stage each)
constexpr int kNQ = kNC / kQW;                    // quads
constexpr int kNS = kCStages;                     // ring slots
constexpr int kMaxG = kPMaxD / 64;                // int4 groups along d
constexpr int kSlotBytes = kMaxG * kGroupBytes;   // one gate/up tile or one down slice
constexpr int kMaxU = kCMaxUnits;                 // units per cluster and layer
constexpr int kMaxRows = kPMaxD / kCl;            // down output rows per CTA
constexpr int kMaxTasks = 3 * kMaxU + 1;
constexpr unsigned kFull = 0xFFFFFFFFu;

static_assert(kCThreads == 32 * (kNC + 2), "producer warp, 16 consumer warps, top-k warp");
static_assert(kCl == 4, "the a push maps 32 lanes onto 4 ranks x 8 fragment words; 8 tiles = 4 ranks x 2");

enum : int { K_GU = 0, K_DN = 1, K_TOPK = 2 };

struct CTask {
  int8_t kind;           // K_GU, K_DN, or the top-k marker
  int8_t tt;             // K_GU: tile 0 or 1 of this CTA's two tiles of the unit
  int8_t ui;             // unit index within the layer (a-slot, down partial buffer)
  int8_t pad;
  int16_t src;           // -1 shared expert, else top-k position j
  int16_t G;             // group (64 intermediate rows)
};

struct Smem {
  alignas(128) uint8_t ring[kNS][kSlotBytes];     // bulk / TMA targets
  alignas(16) uint16_t rrow[kPMaxD];               // this CTA's router row (fp16)
  alignas(16) uint16_t h[kPMaxD];                  // residual stream (bf16), the same in every CTA
  alignas(16) uint16_t xs[kPMaxD];                 // FFN input x (bf16)
  alignas(16) uint16_t xp[kPMaxD];                 // x as mma B fragments
  alignas(16) float xg[kMaxG];                     // per-group sums of x
  alignas(16) uint32_t abuf[2 * kMaxU][64];        // per unit: a as down B fragments (hi/lo), pushed by the cluster
  alignas(16) float tsum[2 * kMaxU][8];            // per unit: sum of a (hi + lo) of each of the 8 gate/up tiles
  alignas(16) float dn_part[kMaxU][kMaxRows];      // per unit: down partials of this CTA's rows
  alignas(16) long long yq[kMaxRows];              // fixed-point layer output rows, bulk-reduce source
  alignas(16) float gu_part[kNS][kQW][8][2];       // gate/up chunk partials [slot][warp][row][gate/up]
  alignas(8) uint64_t full[kNS];
  alignas(8) uint64_t empty[kNS];
  alignas(8) uint64_t a_full[2 * kMaxU];           // 8 remote arrivals per use (4 ranks x 2 tiles)
  alignas(8) uint64_t rrow_full;
  alignas(8) uint64_t rrow_empty;
  alignas(8) uint64_t topk_bar;                    // one phase per layer
  alignas(8) uint64_t cbar;                        // consumer-warp barrier
  alignas(16) DevCallArgs args;
  CTask tasks[kMaxTasks];
  int n_tasks, n_units, n_stages;
  int unit_src[kMaxU];
  int gu_cnt[kNS];
  int finisher;
  float red[kNC];
  long long rlog[kNC];
  int32_t ids[2][32];
  float gates[2][32];
};

static_assert(offsetof(Smem, ring) % 128 == 0 && kSlotBytes % 128 == 0, "TMA targets 128-byte aligned");
static_assert(offsetof(Smem, rrow) % 16 == 0 && offsetof(Smem, yq) % 16 == 0, "bulk copy ends 16-byte aligned");
static_assert(offsetof(Smem, abuf) % 16 == 0, "B fragments read as uint4");

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_idx() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_count() {
  unsigned r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* local, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void arrive_peer(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait for an mbarrier phase completed by arrivals from other CTAs of
// the cluster (acquire at cluster scope).
__device__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kSpinLimitCycles) {
      atomicOr(err, ERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// 3-D tiled TMA load (no swizzle) completing on `bar`; x must be 16-byte aligned.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// dst[i] += src[i] (int64, in L2) for bytes / 8 elements; waits until done.
__device__ __forceinline__ void bulk_reduce_add_s64(long long* dst, const long long* src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u64 [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ ulonglong2 ld_volatile_u64x2(const unsigned long long* p) {
  ulonglong2 v;
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile_u64x2(unsigned long long* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ bool aborted(const CParams& p) {
  return *reinterpret_cast<volatile unsigned*>(p.abort_flag) != 0;
}

__device__ __forceinline__ void raise_abort(const CParams& p) {
  atomicOr(p.err, ERR_WAIT_TIMEOUT);
  atomicExch(p.abort_flag, 1u);
}

// The whole warp waits until *ctr >= target (acquire); warp-uniform polling
// (a loop run by one lane while the others wait leaves the warp diverged and
// slows every later warp-wide instruction).  False on abort or timeout.
__device__ bool warp_wait_counter(const CParams& p, const unsigned* ctr, unsigned target) {
  if (__all_sync(kFull, ld_acquire(ctr) >= target)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    __nanosleep(32);
    if (__all_sync(kFull, ld_acquire(ctr) >= target)) return true;
    if ((it & 255) == 0) {
      if (__any_sync(kFull, aborted(p))) return false;
      if (__any_sync(kFull, clock64() - t0 > kSpinLimitCycles)) {
        if ((threadIdx.x & 31) == 0) raise_abort(p);
        return false;
      }
    }
  }
}

// Consumer-warp barrier: one arrival per consumer warp; round r (from 1)
// completes phase r - 1.  False on timeout.
__device__ bool consumer_barrier(const CParams& p, Smem& S, int round) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbarrier_arrive(&S.cbar);
  const bool ok = mbar_wait_bounded(&S.cbar, static_cast<uint32_t>(round - 1) & 1u, p.err);
  if (!ok) raise_abort(p);
  __syncwarp();
  return ok;
}

__device__ __forceinline__ float gelu_p(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

// ------------------------------------------------------------------ timeline (optional)

// Event times (%globaltimer, ns) of the call's third layer (the last one if
// fewer), row blockIdx.x of the caller's buffer: first occurrence, or latest
// for the *_LAST events.
enum : int { EV_Y_SEEN, EV_X_READY, EV_LOGIT_OUT, EV_LOGITS_IN, EV_TOPK_DONE, EV_ROUTED_ISSUE, EV_SHARED_DATA,
             EV_ROUTED_DATA, EV_PUSH_LAST, EV_DN_LAST, EV_STAGES_DONE, EV_REDUCED, EV_ISSUE_LAST, EV_DATA_LAST,
             EV_DN_A_FIRST, EV_A_WAIT_LAST };

__device__ __forceinline__ void stamp(const CParams& p, int rel, int ev, bool latest = false) {
  if (!p.timeline) return;
  const int n_rel = p.l1 - p.l0;
  if (rel != (n_rel > 2 ? 2 : n_rel - 1)) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  unsigned long long* q = p.timeline + static_cast<size_t>(blockIdx.x) * 16 + ev;
  if (latest) atomicMax(q, t);
  else atomicCAS(q, 0ull, t);
}

// ------------------------------------------------------------------ units and stages

// The cluster's units of a layer (the same for every layer: only the experts
// behind the top-k positions change).  Units are numbered routed first
// (position j, group G -> j * f/64 + G), then shared (k * f/64 + G), and dealt
// round-robin over the clusters, so a cluster with one routed unit more than
// another gets one shared unit fewer; a cluster runs its shared units first.
// Returns the number of units (> kMaxU: does not fit).
__device__ int build_tasks(const CParams& p, Smem& S, int cl, int n_cl) {
  const int nGf = p.f / 64, nGs = p.fs / 64, Ur = p.k * nGf;
  int n = 0, t = 0;
  auto add_unit = [&](int src, int G) {
    if (n < kMaxU) {
      S.unit_src[n] = src;
      for (int s = 0; s < 3; ++s) {
        CTask e;
        e.kind = static_cast<int8_t>(s < 2 ? K_GU : K_DN);
        e.tt = static_cast<int8_t>(s < 2 ? s : 0);
        e.ui = static_cast<int8_t>(n);
        e.pad = 0;
        e.src = static_cast<int16_t>(src);
        e.G = static_cast<int16_t>(G);
        S.tasks[t++] = e;
      }
    }
    ++n;
  };
  for (int G = 0; G < nGs; ++G)
    if ((Ur + G) % n_cl == cl) add_unit(-1, G);
  if (n <= kMaxU) {
    CTask m{};
    m.kind = K_TOPK;
    S.tasks[t++] = m;
  }
  for (int i = 0; i < Ur; ++i)
    if (i % n_cl == cl) add_unit(i / nGf, i % nGf);
  S.n_tasks = t;
  S.n_units = n < kMaxU ? n : kMaxU;
  S.n_stages = 3 * S.n_units;
  return n;
}

// ------------------------------------------------------------------ producer

__device__ void producer(const CParams& p, Smem& S, unsigned rank) {
  const int n_rel = p.l1 - p.l0;
  const uint32_t tile_bytes = static_cast<uint32_t>(p.d / 64) * kGroupBytes;   // gate/up tile = down slice
  const int R = p.d / 64;                                                     // 16-row down tiles per CTA
  uint32_t u_issued = 0;
  bool rrow_issued = false;
  bool stop = false;
  for (int rel = 0; rel < n_rel && !stop; ++rel) {
    const CLayer* L = p.layers + (p.l0 + rel);
    if (static_cast<int>(blockIdx.x) < p.E) {
      if (!mbar_wait_bounded(&S.rrow_empty, (static_cast<uint32_t>(rel) & 1u) ^ 1u, p.err)) {
        raise_abort(p);
        break;
      }
      const uint16_t* rw = L->router_w;
      mbar_arrive_expect_tx(&S.rrow_full, static_cast<uint32_t>(p.d) * 2u);
      bulk_g2s(S.rrow, rw + static_cast<size_t>(blockIdx.x) * p.d, static_cast<uint32_t>(p.d) * 2u, &S.rrow_full);
      rrow_issued = true;
    }
    int s = 0;
    for (int i = 0; i < S.n_tasks; ++i) {
      const CTask t = S.tasks[i];
      if (t.kind == K_TOPK) {
        if (!mbar_wait_bounded(&S.topk_bar, static_cast<uint32_t>(rel) & 1u, p.err)) {
          raise_abort(p);
          stop = true;
          break;
        }
        continue;
      }
      const uint32_t u = static_cast<uint32_t>(rel) * S.n_stages + s++;
      const int slot = u % kNS;
      if (!mbar_wait_bounded(&S.empty[slot], ((u / kNS) & 1u) ^ 1u, p.err)) {
        raise_abort(p);
        stop = true;
        break;
      }
      const int e = t.src < 0 ? 0 : S.ids[rel & 1][t.src];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&S.full[slot], tile_bytes);
      if (t.kind == K_GU) {
        const uint8_t* base = t.src < 0 ? L->shared : L->experts + static_cast<long long>(e) * p.expert_stride;
        const size_t tile = static_cast<size_t>(8 * t.G + 2 * static_cast<int>(rank) + t.tt);
        bulk_g2s(S.ring[slot], base + tile * tile_bytes, tile_bytes, &S.full[slot]);
      } else {
        tma_load_3d(S.ring[slot], t.src < 0 ? &L->dn_shared : &L->dn_routed, t.G * (kGroupBytes / 4),
                    R * static_cast<int>(rank), e, &S.full[slot]);
      }
      u_issued = u + 1;
      if (t.src >= 0) stamp(p, rel, EV_ROUTED_ISSUE);
      stamp(p, rel, EV_ISSUE_LAST, true);
    }
  }
  // after an abort, the last min(u_issued, kNS) stages and the router row may
  // still be in flight into this CTA's shared memory: wait for each, bounded
  if (aborted(p)) {
    for (uint32_t v = (u_issued > static_cast<uint32_t>(kNS) ? u_issued - kNS : 0); v < u_issued; ++v)
      mbar_wait_bounded(&S.full[v % kNS], (v / kNS) & 1u, p.err);
    if (rrow_issued) {
      // the newest router-row phase: consumers may not have waited for it
      for (uint32_t par = 0; par < 2; ++par)
        if (mbar_try_wait(&S.rrow_full, par)) break;
    }
  }
}

// ------------------------------------------------------------------ top-k

// Polls layer l's tagged logits until every entry carries this launch's tag,
// then takes the top-k (ties to the lower index) and the softmax gates.  Each
// lane holds up to 8 logits sorted by (value desc, index asc); a round picks
// the warp-wide best head with three warp reductions on the order-preserving
// unsigned image of the int64 logit and on the index.
__device__ bool topk_layer(const CParams& p, int l, int32_t* ids, float* gates) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* lg = p.tlog + static_cast<size_t>(l) * p.E * 2;
  unsigned long long key[8];
  int idx[8];
  int n = 0;
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    bool ok = true;
    n = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0ull;
      idx[i] = 0x7fffffff;
      if (e < p.E) {
        const ulonglong2 v = ld_volatile_u64x2(lg + 2 * e);
        ok = ok && static_cast<unsigned>(v.x >> 32) == p.tag && static_cast<unsigned>(v.y >> 32) == p.tag;
        key[i] = ((v.y << 32) | (v.x & 0xFFFFFFFFull)) ^ 0x8000000000000000ull;
        idx[i] = e;
        ++n;
      }
    }
    if (__all_sync(kFull, ok)) {
      if (lane == 0) stamp(p, l - p.l0, EV_LOGITS_IN);
      break;
    }
    __nanosleep(32);
    if ((it & 255) == 255) {
      if (__any_sync(kFull, aborted(p))) return false;
      if (__any_sync(kFull, clock64() - t0 > kSpinLimitCycles)) {
        if (lane == 0) raise_abort(p);
        return false;
      }
    }
  }
#pragma unroll
  for (int i = 1; i < 8; ++i) {
#pragma unroll
    for (int j = i; j > 0; --j) {
      if (key[j] > key[j - 1]) {
        const unsigned long long tk = key[j];
        key[j] = key[j - 1];
        key[j - 1] = tk;
        const int ti = idx[j];
        idx[j] = idx[j - 1];
        idx[j - 1] = ti;
      }
    }
  }
  int head = 0, my_id = 0;
  long long my_v = 0;
  for (int j = 0; j < p.k; ++j) {
    unsigned long long hk = 0ull;
    int he = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i == head) {
        hk = key[i];
        he = idx[i];
      }
    const bool has = head < n;
    const unsigned hi = has ? static_cast<unsigned>(hk >> 32) : 0u;
    const unsigned lo = has ? static_cast<unsigned>(hk) : 0u;
    const unsigned mh = __reduce_max_sync(kFull, hi);
    const bool c1 = has && hi == mh;
    const unsigned ml = __reduce_max_sync(kFull, c1 ? lo : 0u);
    const bool c2 = c1 && lo == ml;
    const unsigned me = __reduce_min_sync(kFull, c2 ? static_cast<unsigned>(he) : 0xFFFFFFFFu);
    if (c2 && static_cast<unsigned>(he) == me) ++head;
    if (lane == j) {
      my_id = static_cast<int>(me);
      my_v = static_cast<long long>((static_cast<unsigned long long>(mh) << 32 | ml) ^ 0x8000000000000000ull);
    }
  }
  const long long top = __shfl_sync(kFull, my_v, 0);
  float ex = 0.f;
  if (lane < p.k) ex = expf(__ll2float_rn(my_v - top) * 9.094947017729282e-13f);
  float sum = 0.f;
  for (int j = 0; j < p.k; ++j) sum += __shfl_sync(kFull, ex, j);
  if (lane < p.k) {
    ids[lane] = my_id;
    gates[lane] = ex / sum;
  }
  __syncwarp();
  return true;
}

__device__ void topk_warp(const CParams& p, Smem& S) {
  const int lane = threadIdx.x & 31;
  const int n_rel = p.l1 - p.l0;
  for (int rel = 0; rel < n_rel; ++rel) {
    int32_t* sid = S.ids[rel & 1];
    float* sg = S.gates[rel & 1];
    if (!topk_layer(p, p.l0 + rel, sid, sg)) return;
    if (lane == 0) stamp(p, rel, EV_TOPK_DONE);
    if (blockIdx.x == 0 && lane < p.k && rel < S.args.dbg_layers) {
      const DevCallArgs* A = &S.args;
      const size_t o = (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.k + lane;
      if (A->dbg_ids) A->dbg_ids[o] = sid[lane];
      if (A->dbg_gates) A->dbg_gates[o] = sg[lane];
    }
    __syncwarp();
    if (lane == 0) mbarrier_arrive(&S.topk_bar);
  }
}

// ------------------------------------------------------------------ consumers

// Layer input: wait for the previous layer's output vector, add it to this
// CTA's copy of the residual stream, RMS norm in a fixed order (every CTA gets
// the same x), x as plain bf16, as mma B fragments and as per-group sums.
__device__ bool prep(const CParams& p, Smem& S, int cw, int rel, int& round) {
  const int lane = threadIdx.x & 31;
  const int d = p.d, nGd = d / 64;
  const DevCallArgs* A = &S.args;
  const long long* yin = nullptr;
  if (rel > 0) {
    if (cw == 0 && !warp_wait_counter(p, p.y_cnt + (rel - 1), gridDim.x)) return false;
    if (cw == 0 && lane == 0) stamp(p, rel, EV_Y_SEEN);
    if (!consumer_barrier(p, S, ++round)) return false;
    yin = p.ybuf + static_cast<size_t>((rel - 1) % 3) * d;
    // this CTA's share of the vector layer rel + 1 adds into: its last reader
    // was the input step of layer rel - 1, which every CTA finished before the
    // counter just waited for
    long long* yz = p.ybuf + static_cast<size_t>((rel + 1) % 3) * d;
    const int share = (d + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int j = cw * 32 + lane, i = static_cast<int>(blockIdx.x) * share + j;
    if (j < share && i < d) yz[i] = 0;
  }
  // warp cw takes groups G = cw, cw + kNC, ...; lane holds elements 64G + 2*lane, +1
  uint32_t hv[(kMaxG + kNC - 1) / kNC];
  float ss = 0.f;
  int ng = 0;
  const bool dbg_y = blockIdx.x == 0 && rel > 0 && A->dbg_y && rel - 1 < A->dbg_layers;
  for (int G = cw; G < nGd; G += kNC, ++ng) {
    uint32_t v;
    if (rel == 0) {
      v = __ldcg(reinterpret_cast<const unsigned*>(A->h_in + 64 * G) + lane);
    } else {
      v = reinterpret_cast<const uint32_t*>(S.h)[32 * G + lane];
      const longlong2 yy = __ldcg(reinterpret_cast<const longlong2*>(yin + 64 * G + 2 * lane));
      const float y0 = __ll2float_rn(yy.x) * 2.3283064365386963e-10f;   // 2^-32
      const float y1 = __ll2float_rn(yy.y) * 2.3283064365386963e-10f;
      const float a = bf16_bits_to_float(static_cast<uint16_t>(v & 0xFFFFu)) + y0;
      const float b = bf16_bits_to_float(static_cast<uint16_t>(v >> 16)) + y1;
      v = static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
      if (dbg_y) {
        float* dy = A->dbg_y + (static_cast<size_t>(rel - 1) * A->tok_total + A->tok_off) * d + 64 * G + 2 * lane;
        dy[0] = y0;
        dy[1] = y1;
      }
    }
    reinterpret_cast<uint32_t*>(S.h)[32 * G + lane] = v;
    hv[ng] = v;
    const float a = bf16_bits_to_float(static_cast<uint16_t>(v & 0xFFFFu));
    const float b = bf16_bits_to_float(static_cast<uint16_t>(v >> 16));
    ss += a * a;
    ss += b * b;
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(kFull, ss, m);
  if (lane == 0) S.red[cw] = ss;
  if (!consumer_barrier(p, S, ++round)) return false;   // red[] complete, the previous layer's stages all done
  float r = 1.f;
  if (p.prenorm) {
    float tot = 0.f;
    for (int w = 0; w < kNC; ++w) tot += S.red[w];
    r = 1.0f / sqrtf(tot / static_cast<float>(d) + p.eps);
  }
  ng = 0;
  for (int G = cw; G < nGd; G += kNC, ++ng) {
    uint32_t xv = hv[ng];
    if (p.prenorm) {
      const float a = bf16_bits_to_float(static_cast<uint16_t>(xv & 0xFFFFu)) * r;
      const float b = bf16_bits_to_float(static_cast<uint16_t>(xv >> 16)) * r;
      xv = static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
    }
    reinterpret_cast<uint32_t*>(S.xs)[32 * G + lane] = xv;
    // B fragments: element e = 2*lane of the group lands in (t4, st, pos)
    const int e = 2 * lane, st = e >> 4, w = e & 15;
    const int t4 = (w & 7) >> 1, hi = w >> 3;
    reinterpret_cast<uint32_t*>(S.xp)[((G * 4 + t4) * 4 + st) * 2 + hi] = xv;
    float gs = bf16_bits_to_float(static_cast<uint16_t>(xv & 0xFFFFu)) +
               bf16_bits_to_float(static_cast<uint16_t>(xv >> 16));
#pragma unroll
    for (int m = 16; m; m >>= 1) gs += __shfl_xor_sync(kFull, gs, m);
    if (lane == 0) S.xg[G] = gs;
    if (blockIdx.x == 0 && A->dbg_x && rel < A->dbg_layers)
      reinterpret_cast<uint32_t*>(A->dbg_x + (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * d)[32 * G + lane] = xv;
  }
  const bool ok = consumer_barrier(p, S, ++round);   // x complete
  if (cw == 0 && lane == 0) stamp(p, rel, EV_X_READY);
  return ok;
}

// Router row blockIdx.x of layer rel (exact fixed-point logit, all consumer
// warps), published with this launch's tag in both 64-bit words.
__device__ bool router(const CParams& p, Smem& S, int cw, int rel, int& round) {
  if (static_cast<int>(blockIdx.x) >= p.E) return true;
  const int lane = threadIdx.x & 31;
  if (!mbar_wait_bounded(&S.rrow_full, static_cast<uint32_t>(rel) & 1u, p.err)) {
    raise_abort(p);
    return false;
  }
  const uint4* wr = reinterpret_cast<const uint4*>(S.rrow);
  const uint4* xv4 = reinterpret_cast<const uint4*>(S.xs);
  Fix40 fx;
  bool bad = false;
  for (int c0 = cw * 32; c0 < p.d / 8; c0 += 32 * kNC) {
    const int c = min(c0 + lane, p.d / 8 - 1);
    const bool live = c0 + lane < p.d / 8;   // the clamped lanes of a ragged tail add nothing
    uint4 wv = wr[c];
    const uint4 xv = xv4[c];
    if (!live) wv = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float pw = hh ? half_hi(wa[i]) : half_lo(wa[i]);
        const float px = bf16_bits_to_float(static_cast<uint16_t>(hh ? (xa[i] >> 16) : (xa[i] & 0xFFFFu)));
        const float prod = pw * px;  // exact: 11-bit x 8-bit significands
        const bool ok = fabsf(prod) < 2048.f;
        bad |= !ok;
        fix40_add(fx, ok ? prod * 1099511627776.0f : 0.f);  // RNE onto the 2^-40 grid, summed exactly
      }
    }
  }
  long long acc = fix40_value(fx);
#pragma unroll
  for (int m = 16; m; m >>= 1) acc += shfl_xor_i64(acc, m);
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(p.err, ERR_ROUTER_DOMAIN);
  if (lane == 0) S.rlog[cw] = acc;
  if (!consumer_barrier(p, S, ++round)) return false;   // every warp is done with the row and rlog[] is complete
  if (cw != 0) return true;
  acc = 0;
  for (int w = 0; w < kNC; ++w) acc += S.rlog[w];
  if (lane == 0) {
    mbarrier_arrive(&S.rrow_empty);
    const DevCallArgs* A = &S.args;
    if (A->bias) {
      const float bv = A->bias[(static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.E + blockIdx.x];
      if (!(fabsf(bv) < 1048576.f)) atomicOr(p.err, ERR_ROUTER_DOMAIN);
      else acc += __float2ll_rn(bv * 1099511627776.0f);
    }
    const unsigned long long tg = static_cast<unsigned long long>(p.tag) << 32;
    const unsigned long long ua = static_cast<unsigned long long>(acc);
    st_volatile_u64x2(p.tlog + (static_cast<size_t>(p.l0 + rel) * p.E + blockIdx.x) * 2, (ua & 0xFFFFFFFFull) | tg,
                      (ua >> 32) | tg);
    stamp(p, rel, EV_LOGIT_OUT);
  }
  return true;
}

// One chunk (<= 11 groups) of a gate/up tile: partial gate and up sums of row g.
__device__ void gu_chunk(Smem& S, const uint8_t* chunk, int g0, int ng, float& ga, float& ua) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  for (int i = 0; i < ng; ++i) {
    const int G = g0 + i;
    const uint8_t* blk = chunk + i * kGroupBytes;
    const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
    const uint4* xf = reinterpret_cast<const uint4*>(S.xp) + (G * 4 + t4) * 2;
    const uint4 x01 = xf[0], x23 = xf[1];
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t a[4];
    nibbles_to_bf16x2(q.x, a);
    mma_bf16(c0, a, x01.x, x01.y);
    nibbles_to_bf16x2(q.y, a);
    mma_bf16(c1, a, x01.z, x01.w);
    nibbles_to_bf16x2(q.z, a);
    mma_bf16(c0, a, x23.x, x23.y);
    nibbles_to_bf16x2(q.w, a);
    mma_bf16(c1, a, x23.z, x23.w);
    const float X = S.xg[G];
    const float sg = half_lo(sbv.x), bg = half_hi(sbv.x), su = half_lo(sbv.y), bu = half_hi(sbv.y);
    ga += sg * (c0[0] + c1[0]) + fmaf(-128.f, sg, bg) * X;
    ua += su * (c0[2] + c1[2]) + fmaf(-128.f, su, bu) * X;
  }
}

// Epilogue of gate/up tile tt of a unit: a = GELU(gate) * up for its 8 rows,
// split into bf16 hi + lo, written as down B fragments into the unit's a-slot
// of every CTA of the cluster, with the tile's sum of a; then one remote
// arrival on each CTA's a_full barrier.  Tile tt of rank r holds the unit's
// intermediate rows 16r + 8tt + g, i.e. k16 step r, in-step rows 8tt + g.
__device__ void gu_push(const CParams& p, Smem& S, int rel, const CTask& t, unsigned rank, float ga, float ua) {
  const int lane = threadIdx.x & 31;
  const float av = gelu_p(ga, p.gelu) * ua;
  const uint32_t hi = float_to_bf16_bits(av);
  const uint32_t lo = float_to_bf16_bits(av - bf16_bits_to_float(static_cast<uint16_t>(hi)));
  float sh = bf16_bits_to_float(static_cast<uint16_t>(hi)), sl = bf16_bits_to_float(static_cast<uint16_t>(lo));
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    sh += __shfl_xor_sync(kFull, sh, m);
    sl += __shfl_xor_sync(kFull, sl, m);
  }
  // lane = (destination rank, hi/lo column, t4): fragment word t4 of that
  // column packs rows 2*t4 and 2*t4 + 1 (held by lanes 8*t4 and 8*t4 + 4)
  const int dr = lane >> 3, par = (lane >> 2) & 1, t4w = lane & 3;
  const uint32_t h0 = __shfl_sync(kFull, hi, 8 * t4w), h1 = __shfl_sync(kFull, hi, 8 * t4w + 4);
  const uint32_t l0 = __shfl_sync(kFull, lo, 8 * t4w), l1 = __shfl_sync(kFull, lo, 8 * t4w + 4);
  const uint32_t word = par ? (l0 | (l1 << 16)) : (h0 | (h1 << 16));
  const int aslot = (rel & 1) * kMaxU + t.ui;
  const int wpos = ((par * 4 + t4w) * 4 + static_cast<int>(rank)) * 2 + t.tt;
  st_peer_u32(peer_addr(&S.abuf[aslot][wpos], static_cast<unsigned>(dr)), word);
  if (lane < kCl) st_peer_f32(peer_addr(&S.tsum[aslot][2 * rank + t.tt], static_cast<unsigned>(lane)), sh + sl);
  fence_acq_rel_cluster();
  __syncwarp();
  if (lane < kCl) arrive_peer(peer_addr(&S.a_full[aslot], static_cast<unsigned>(lane)));
  if (lane == 0) stamp(p, rel, EV_PUSH_LAST, true);
}

// Gate/up stage: warp qw of the quad takes groups [qw * cgu, ...); the last
// warp of the quad to finish sums the four partials in warp order and pushes a.
__device__ void stage_gu(const CParams& p, Smem& S, int qw, int rel, int slot, const CTask& t, unsigned rank) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nGd = p.d / 64, cgu = (nGd + kQW - 1) / kQW;
  const int g0 = qw * cgu, ng = min(cgu, nGd - g0);
  float ga = 0.f, ua = 0.f;
  if (ng > 0) gu_chunk(S, S.ring[slot] + static_cast<size_t>(g0) * kGroupBytes, g0, ng, ga, ua);
  if (t4 == 0) {
    S.gu_part[slot][qw][g][0] = ga;
    S.gu_part[slot][qw][g][1] = ua;
  }
  __threadfence_block();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&S.gu_cnt[slot], 1) == kQW - 1;
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __threadfence_block();
  ga = 0.f;
  ua = 0.f;
  for (int w = 0; w < kQW; ++w) {
    ga += reinterpret_cast<volatile float*>(S.gu_part[slot][w][g])[0];
    ua += reinterpret_cast<volatile float*>(S.gu_part[slot][w][g])[1];
  }
  __syncwarp();
  if (lane == 0) S.gu_cnt[slot] = 0;
  gu_push(p, S, rel, t, rank, ga, ua);
}

// Down stage: this CTA's d/64 row tiles of the unit's group, warp qw taking
// tiles qw, qw + 4, ...; every tile uses the same 64 values of a.
__device__ bool stage_dn(const CParams& p, Smem& S, int qw, int rel, int slot, const CTask& t) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int aslot = (rel & 1) * kMaxU + t.ui;
  if (!mbar_wait_cluster(&S.a_full[aslot], (static_cast<uint32_t>(rel) >> 1) & 1u, p.err)) return false;
  if (lane == 0) {
    stamp(p, rel, EV_DN_A_FIRST);
    stamp(p, rel, EV_A_WAIT_LAST, true);
  }
  float As = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) As += S.tsum[aslot][i];
  const uint4* bf = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(S.abuf[aslot]) +
                                                   ((g & 1) * 4 + t4) * 32);
  const uint4 b01 = bf[0], b23 = bf[1];
  const int R = p.d / 64;
  float* out = S.dn_part[t.ui];
  for (int T = qw; T < R; T += kQW) {
    const uint8_t* blk = S.ring[slot] + static_cast<size_t>(T) * kGroupBytes;
    const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t a[4];
    nibbles_to_bf16x2(q.x, a);
    mma_bf16(c0, a, b01.x, b01.y);
    nibbles_to_bf16x2(q.y, a);
    mma_bf16(c1, a, b01.z, b01.w);
    nibbles_to_bf16x2(q.z, a);
    mma_bf16(c0, a, b23.x, b23.y);
    nibbles_to_bf16x2(q.w, a);
    mma_bf16(c1, a, b23.z, b23.w);
    const float s0 = half_lo(sbv.x), o0 = half_hi(sbv.x), s1 = half_lo(sbv.y), o1 = half_hi(sbv.y);
    const float y0 = s0 * ((c0[0] + c1[0]) + (c0[1] + c1[1])) + fmaf(-128.f, s0, o0) * As;
    const float y1 = s1 * ((c0[2] + c1[2]) + (c0[3] + c1[3])) + fmaf(-128.f, s1, o1) * As;
    if (t4 == 0) {
      out[T * 16 + g] = y0;
      out[T * 16 + g + 8] = y1;
    }
  }
  return true;
}

// End of layer rel: gate-weighted sum of the units' partials in unit order,
// onto the 2^-32 grid, one bulk reduction into the layer's output vector, and
// the layer counter.  The CTA whose increment completes the last layer reads
// the final vector (finish()).
__device__ bool layer_end(const CParams& p, Smem& S, int cw, int rel, int& round, unsigned rank) {
  const int lane = threadIdx.x & 31;
  if (!mbar_wait_bounded(&S.topk_bar, static_cast<uint32_t>(rel) & 1u, p.err)) {   // gates of this layer
    raise_abort(p);
    return false;
  }
  if (!consumer_barrier(p, S, ++round)) return false;   // every down partial of the layer written
  if (cw == 0 && lane == 0) stamp(p, rel, EV_STAGES_DONE);
  const int rows = p.d / kCl;
  const float* gts = S.gates[rel & 1];
  bool bad = false;
  for (int i0 = 0; i0 < rows; i0 += kNC * 32) {
    const int i = i0 + cw * 32 + lane;
    if (i < rows) {
      float y = 0.f;
      for (int u = 0; u < S.n_units; ++u) {
        const int src = S.unit_src[u];
        y = fmaf(src < 0 ? 1.f : gts[src], S.dn_part[u][i], y);
      }
      const bool ok = fabsf(y) < 16777216.f;   // |y| < 2^24: the int64 sum over all CTAs cannot overflow
      bad |= !ok;
      S.yq[i] = ok ? __float2ll_rn(y * 4294967296.f) : 0ll;
    }
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(p.err, ERR_Y_RANGE);
  fence_proxy_async_smem();   // yq is read by the bulk reduction (async proxy)
  if (!consumer_barrier(p, S, ++round)) return false;
  if (cw != 0) return true;
  unsigned old = 0;
  if (lane == 0) {
    if (S.n_units > 0) {
      fence_proxy_async_global();   // the zeroing of this vector (generic stores, other CTAs) came first
      bulk_reduce_add_s64(p.ybuf + static_cast<size_t>(rel % 3) * p.d + static_cast<size_t>(rank) * rows, S.yq,
                          static_cast<uint32_t>(rows) * 8u);
      fence_proxy_async_global();
    }
    stamp(p, rel, EV_REDUCED);
    __threadfence();
    old = atom_add_acq_rel(p.y_cnt + rel, 1u);
  }
  old = __shfl_sync(kFull, old, 0);
  if (lane == 0) S.finisher = old == gridDim.x - 1 ? 1 : 0;
  return true;
}

// Run by the CTA that completed the last layer: h_out = bf16(h + y), y_last,
// the last layer's debug y, and the output vectors zeroed for the next launch.
__device__ void finish(const CParams& p, Smem& S, int cw, int rel, int& round) {
  const int lane = threadIdx.x & 31;
  if (!consumer_barrier(p, S, ++round)) return;
  if (!S.finisher) return;
  const DevCallArgs* A = &S.args;
  const int d = p.d;
  long long* yv = p.ybuf + static_cast<size_t>(rel % 3) * d;
  const bool dbg_y = A->dbg_y && rel < A->dbg_layers;
  for (int j0 = 0; j0 < d / 2; j0 += kNC * 32) {
    const int j = j0 + cw * 32 + lane;
    if (j < d / 2) {
      const longlong2 yy = __ldcg(reinterpret_cast<const longlong2*>(yv + 2 * j));
      const float y0 = __ll2float_rn(yy.x) * 2.3283064365386963e-10f;
      const float y1 = __ll2float_rn(yy.y) * 2.3283064365386963e-10f;
      const uint32_t hv = reinterpret_cast<const uint32_t*>(S.h)[j];
      const float a = bf16_bits_to_float(static_cast<uint16_t>(hv & 0xFFFFu)) + y0;
      const float b = bf16_bits_to_float(static_cast<uint16_t>(hv >> 16)) + y1;
      reinterpret_cast<uint32_t*>(A->h_out)[j] =
          static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
      if (A->y_last) {
        A->y_last[2 * j] = y0;
        A->y_last[2 * j + 1] = y1;
      }
      if (dbg_y) {
        float* dy = A->dbg_y + (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * d + 2 * j;
        dy[0] = y0;
        dy[1] = y1;
      }
      *reinterpret_cast<longlong2*>(yv + 2 * j) = make_longlong2(0, 0);
      if (rel > 0) {
        long long* yp = p.ybuf + static_cast<size_t>((rel - 1) % 3) * d;
        *reinterpret_cast<longlong2*>(yp + 2 * j) = make_longlong2(0, 0);
      }
    }
  }
}

__device__ void consumer(const CParams& p, Smem& S, int cw, unsigned rank) {
  const int lane = threadIdx.x & 31;
  const int quad = cw / kQW, qw = cw % kQW;
  const int n_rel = p.l1 - p.l0;
  int round = 0;
  for (int rel = 0; rel < n_rel; ++rel) {
    if (!prep(p, S, cw, rel, round)) return;
    if (!router(p, S, cw, rel, round)) return;
    int s = 0;
    for (int i = 0; i < S.n_tasks; ++i) {
      const CTask t = S.tasks[i];
      if (t.kind == K_TOPK) continue;
      const uint32_t u = static_cast<uint32_t>(rel) * S.n_stages + s++;
      if (static_cast<int>(u % kNQ) != quad) continue;
      const int slot = u % kNS;
      if (!mbar_wait_bounded(&S.full[slot], (u / kNS) & 1u, p.err)) {
        raise_abort(p);
        return;
      }
      if (lane == 0) {
        stamp(p, rel, t.src < 0 ? EV_SHARED_DATA : EV_ROUTED_DATA);
        stamp(p, rel, EV_DATA_LAST, true);
      }
      if (t.kind == K_GU) {
        stage_gu(p, S, qw, rel, slot, t, rank);
      } else if (!stage_dn(p, S, qw, rel, slot, t)) {
        raise_abort(p);
        return;
      }
      __syncwarp();
      if (lane == 0) mbarrier_arrive(&S.empty[slot]);
    }
    if (!layer_end(p, S, cw, rel, round, rank)) return;
  }
  finish(p, S, cw, n_rel - 1, round);
}

// 18 warps put five on two of the SM's four schedulers; each scheduler has 16 K
// registers, so a thread may hold at most 96 (launch bounds give exactly that).
__global__ void __launch_bounds__(kCThreads, 1) k_decode_cluster(CParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const unsigned rank = cluster_rank();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kQW);
    }
    for (int i = 0; i < 2 * kMaxU; ++i) mbar_init(&S.a_full[i], 2 * kCl);
    mbar_init(&S.rrow_full, 1);
    mbar_init(&S.rrow_empty, 1);
    mbar_init(&S.topk_bar, 1);
    mbar_init(&S.cbar, kNC);
    fence_mbar_init();
    S.args = *p.args;
    S.finisher = 0;
    if (build_tasks(p, S, static_cast<int>(cluster_idx()), static_cast<int>(cluster_count())) > kMaxU)
      raise_abort(p);
  }
  if (threadIdx.x < kNS) S.gu_cnt[threadIdx.x] = 0;
  __syncthreads();
  cluster_sync_all();   // every CTA's barriers exist before any remote arrival
  if (!aborted(p)) {
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) producer(p, S, rank);
    } else if (warp <= kNC) {
      consumer(p, S, warp - 1, rank);
    } else {
      topk_warp(p, S);
    }
  }
  __syncthreads();
  cluster_sync_all();   // no CTA leaves while a peer may still write into its shared memory
  // the last CTA out zeroes the counters (and, after an abort, the output vectors)
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(p.exit_cnt, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.y_cnt[i] = 0;
    if (aborted(p))
      for (int i = threadIdx.x; i < 3 * p.d; i += blockDim.x) p.ybuf[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      *p.abort_flag = 0;
      *p.exit_cnt = 0;
      __threadfence();
    }
  }
}

}  // namespace

size_t cluster_smem() { return sizeof(Smem); }

int cluster_max_units() { return kMaxU; }

cudaError_t cluster_attrs() {
  return cudaFuncSetAttribute((const void*)k_decode_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(Smem)));
}

// Clusters of kCCluster CTAs (one per SM) that can be resident at once.
cudaError_t cluster_max_active(int* n_clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCCluster);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n_clusters, (const void*)k_decode_cluster, &cfg);
}

cudaError_t launch_cluster(CParams& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_decode_cluster, p);
}

}  // namespace moe
