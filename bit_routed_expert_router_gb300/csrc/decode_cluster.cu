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
//   (16 intermediate rows) and writes their 16 values of a (as fp16 hi + lo
//   mma.sync B fragments) and their sums into the shared memory of every CTA of
//   the cluster (distributed shared memory) with asynchronous remote stores
//   that count their bytes on that CTA's barrier for the unit; then it
//   multiplies output rows [r d/4, (r+1) d/4) of the unit's down block by the
//   64 values once all eight tiles' bytes have arrived.
//
// The grid-wide exchanges left per layer are the router logits (one router
// row per CTA, published with a per-launch tag inside each 64-bit word into
// one replica per cluster, so a cluster's top-k warps poll their own copy
// and the readers do not crowd a single set of lines) and the layer output: each CTA sums its units'
// down partials (gate-weighted, fixed order) for its d/4 rows, rounds them onto
// a 2^-32 fixed-point grid and adds (v << 8) + 1 per row into the layer's int64
// output vector with one bulk reduction (TMA engine, integer adds in L2, so the
// result does not depend on the order in which CTAs arrive).  The low byte of
// a row counts its contributions, so a reader polls the rows themselves: every
// CTA polls the whole vector, adds it to its copy of the residual stream and
// normalises it for the next layer.
//
// Roles per CTA (18 warps):
//   warp 0, lane 0 (producer): the router row, then every stage of the CTA's
//     units (gate/up tiles by 1-D bulk copy, down slices by a 3-D TMA tile load
//     that gathers one group of d/64 consecutive 16-row tiles) into a ring of
//     seven shared-memory slots; routing-independent units (shared expert) come
//     first, routed units after the top-k is known.
//   warps 1..16 (consumers): four quads of four warps; stage u of the CTA goes
//     to quad u mod 4 (gate/up: a quarter of the groups per warp, the last
//     warp of the quad to finish sums the partials in warp order and runs the
//     epilogue and the push; down: row tiles strided by warp).  A unit's down
//     stage is queued after the next two units' gate/up stages, so its 64
//     values of a have normally arrived from the other CTAs of the cluster.
//   warp 17 (top-k, in the cluster's rank-0 CTA): once its CTA's stages of the
//     previous layer are done, polls the layer's tagged logits, takes the top-k
//     (publishing each rank for the cluster's producers as soon as it is
//     picked) and the softmax gates.
// Every wait is bounded and gives up through an abort flag and the device
// error word (MOE_ETIMEOUT from moe_sync).  Output vectors rotate over three
// buffers, each zeroed (in shares, by every CTA) once everyone has read it.
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

#include <cstddef>

namespace moe {

namespace {

constexpr int kCl = kCCluster;                    // CTAs per cluster
constexpr int kNC = 16;                           // consumer warps
constexpr int kQW = 4;                            // warps per quad (one work item each)
constexpr int kNQ = kNC / kQW;                    // quads
constexpr int kNS = kCStages;                     // ring slots
constexpr int kMaxD = kCMaxD;                     // largest d this kernel's buffers hold
constexpr int kMaxG = kMaxD / 64;                 // int4 groups along d
constexpr int kSlotBytes = kMaxG * kGroupBytes;   // one gate/up tile or one down slice
constexpr int kMaxU = kCMaxUnits;                 // units per cluster and layer
constexpr int kMaxRows = kMaxD / kCl;             // down output rows per CTA
constexpr int kMaxTasks = 3 * kMaxU + 1;
constexpr unsigned kFull = 0xFFFFFFFFu;

static_assert(kCThreads == 32 * (kNC + 2), "producer warp, 16 consumer warps, top-k warp");
static_assert(kCl == 4, "the a push maps 32 lanes onto 4 ranks x 8 fragment words; 8 tiles = 4 ranks x 2");
constexpr uint32_t kAPushBytes = 2 * kCl * (8 * 4 + 4);   // a unit's pushes into one CTA: 8 tiles x (8 words + sum)

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
  alignas(16) uint16_t rrow[kMaxD];                // this CTA's router row (fp16)
  alignas(16) uint16_t h[kMaxD];                   // residual stream (bf16), the same in every CTA
  alignas(16) uint16_t xp[kMaxD];                  // x as fp16 mma B fragments
  alignas(16) float xg[kMaxG];                     // per-group sums of the fp16 x
  alignas(16) uint32_t abuf[2 * kMaxU][64];        // per unit: a as B-fragment words, block (2 rank + tile) of 8
                                                   // words (4 * hi/lo column + t4) per sending tile
  alignas(16) float tsum[2 * kMaxU][8];            // per unit: sum of a (hi + lo) of each of the 8 gate/up tiles
  alignas(16) float dn_acc[kNQ][kMaxRows];         // per quad: its down stages' gate-weighted rows, in stage order
  alignas(16) long long yq[kMaxRows];              // fixed-point layer output rows, bulk-reduce source
  alignas(16) float gu_part[kNS][kQW][8][2];       // gate/up partials [slot][warp of the quad][row][gate/up]
  alignas(8) uint64_t full[kNS];
  alignas(8) uint64_t empty[kNS];
  alignas(8) uint64_t a_full[2 * kMaxU];           // per use: this CTA's expect of 8 x 36 bytes, and the bytes
  alignas(8) uint64_t rrow_full;
  alignas(8) uint64_t rrow_empty;
  alignas(8) uint64_t topk_bar;                    // one phase per layer
  alignas(8) uint64_t zero_bar;                    // one phase per layer: this CTA's share of the next vector zeroed
  alignas(8) uint64_t end_bar;                     // one phase per layer: this CTA's stages of the layer are done
  alignas(8) uint64_t cbar;                        // consumer-warp barrier
  alignas(16) DevCallArgs args;
  CTask tasks[kMaxTasks];
  int n_tasks, n_units, n_stages;
  int unit_src[kMaxU];
  int unit_G[kMaxU];
  int gu_cnt[kNS];
  float red[kNC];
  long long rlog[kNC];
  int32_t ids[2][32];
  float gates[2][32];
  alignas(8) long long topv[32];                   // top-k logits in rank order
  int last_out;                                    // this CTA is the last to leave the launch
  unsigned rank_word[32];                          // rank j of the top-k: (64 * layer + j + 1) << 8 | expert
  // host-pool mode: the producer's copy of the layer's plan words, and per
  // ring slot the stage a consumer warp fills from the mapped pool (a miss)
  unsigned long long plan_w[32];
  const uint8_t* fill_src[kNS];                    // host-pool address of the stage's data, or null (copied by TMA)
  uint8_t* fill_dst[kNS];                          // the same bytes' place in the device slot
  int fill_stride[kNS];                            // 0: one contiguous tile; else bytes between 576-byte row tiles
};

static_assert(offsetof(Smem, ring) % 128 == 0 && kSlotBytes % 128 == 0, "TMA targets 128-byte aligned");
static_assert(offsetof(Smem, rrow) % 16 == 0 && offsetof(Smem, yq) % 16 == 0, "bulk copy ends 16-byte aligned");
static_assert(offsetof(Smem, abuf) % 16 == 0, "B fragments read as uint4");
static_assert(sizeof(Smem) <= 227 * 1024, "shared memory per CTA (the kernel has no static shared memory)");

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
__device__ __forceinline__ unsigned cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
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
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void arrive_peer(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ bool aborted(const CParams& p);

// Wait sites, recorded with the CTA in p.diag by the first wait that runs out
// (the others then see the abort flag and leave without recording).
enum : unsigned { W_CBAR = 1, W_Y_POLL, W_RROW_EMPTY, W_P_TOPK, W_EMPTY, W_LOGITS, W_CLBAR, W_RROW_FULL, W_A_FULL,
                  W_DN_TOPK, W_END_TOPK, W_FINISH, W_FULL, W_ZERO, W_PLAN, W_END_STAGES };
__device__ __forceinline__ void note_timeout(const CParams& p, unsigned site) {
  atomicOr(p.err, ERR_WAIT_TIMEOUT);
  if (p.diag) atomicCAS(p.diag, 0u, (site << 16) | (blockIdx.x & 0xFFFFu));
}

// Bounded wait for an mbarrier phase completed by arrivals from other CTAs of
// the cluster (acquire at cluster scope), by a whole warp: the lanes decide
// together (a vote per poll), so a warp never splits between going on and
// giving up.  False after p.spin_limit cycles or once another CTA has aborted.
__device__ bool mbar_wait_cluster(const CParams& p, uint64_t* bar, uint32_t parity, unsigned site) {
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (__all_sync(kFull, ok != 0)) return true;
    if (__any_sync(kFull, clock64() - t0 > p.spin_limit)) {
      if ((threadIdx.x & 31) == 0) note_timeout(p, site);
      return false;
    }
    if ((it & 15) == 15 && __any_sync(kFull, aborted(p))) return false;
  }
}

// Bounded wait on a phase of a local mbarrier (this CTA's threads or copies)
// by a whole warp, deciding together as above.
__device__ bool wait_warp(const CParams& p, uint64_t* bar, uint32_t parity, unsigned site) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(kFull, clock64() - t0 > p.spin_limit)) {
      if ((threadIdx.x & 31) == 0) note_timeout(p, site);
      return false;
    }
    if ((it & 15) == 0 && __any_sync(kFull, aborted(p))) return false;
  }
}

// The same wait by a single thread (the producer).
__device__ bool wait_one(const CParams& p, uint64_t* bar, uint32_t parity, unsigned site) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > p.spin_limit) {
      note_timeout(p, site);
      return false;
    }
    if ((it & 15) == 0 && aborted(p)) return false;
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

// Relaxed (gpu scope) 2 x 64-bit accesses; each 64-bit element is single-copy
// atomic, which is what the tagged and counted words rely on.
__device__ __forceinline__ ulonglong2 ld_volatile_u64x2(const unsigned long long* p) {
  ulonglong2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile_u64x2(unsigned long long* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ bool aborted(const CParams& p) {
  return *reinterpret_cast<volatile unsigned*>(p.abort_flag) != 0;
}

__device__ __forceinline__ void raise_abort(const CParams& p) {
  atomicOr(p.err, ERR_WAIT_TIMEOUT);
  atomicExch(p.abort_flag, 1u);
}

// Consumer-warp barrier: one arrival per consumer warp; round r (from 1)
// completes phase r - 1.  False on timeout.
__device__ bool consumer_barrier(const CParams& p, Smem& S, int round) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbarrier_arrive(&S.cbar);
  const bool ok = wait_warp(p, &S.cbar, static_cast<uint32_t>(round - 1) & 1u, W_CBAR);
  if (!ok) raise_abort(p);
  __syncwarp();
  return ok;
}

// v * 2^-32 rounded to fp32 (the same value as a 64-bit integer conversion
// scaled by 2^-32) with 32-bit conversions only: conversions from and to
// 64-bit integers run on this part's narrow FP64 path, which measured slow
// enough to matter in the layer's hot loops.  For |v| < 2^48 both halves are
// exact in fp32 and the one rounding of their sum is the correct one.
__device__ __forceinline__ float grid_to_float(long long v) {
  const long long q = v >> 24;
  if (q > -(1ll << 24) && q < (1ll << 24))
    return fmaf(static_cast<float>(static_cast<int>(q)), 0.00390625f,                       // 2^-8
                static_cast<float>(static_cast<unsigned>(v & 0xFFFFFF)) * 5.9604644775390625e-08f * 3.90625e-3f);
  return __ll2float_rn(v) * 2.3283064365386963e-10f;                                         // 2^-32
}

// RN(v) as fp32 (the value of a 64-bit integer conversion) with 32-bit
// conversions for |v| < 2^48: v = q 2^24 + r with both parts exact in fp32
// and one rounding of their fused sum.
__device__ __forceinline__ float ll_to_float(long long v) {
  const long long q = v >> 24;
  if (q > -(1ll << 24) && q < (1ll << 24))
    return fmaf(static_cast<float>(static_cast<int>(q)), 16777216.f, static_cast<float>(static_cast<unsigned>(v & 0xFFFFFF)));
  return __ll2float_rn(v);
}

// RNE(b * 2^40) for |b| < 2^20 (the bias domain) with 32-bit conversions:
// a = |b| 2^40 is an exact fp32 value below 2^60; its multiples of 2^32 and
// its remainder (at most 24 significant bits) are exact, and the remainder is
// rounded to an integer, ties to even, by the one 32-bit conversion.
__device__ __forceinline__ long long bias_fix40(float b) {
  const float a = fabsf(b) * 1099511627776.0f;                      // 2^40
  const float h = floorf(a * 2.3283064365386963e-10f);              // 2^-32
  const float r = fmaf(-h, 4294967296.0f, a);                       // exact
  const long long m = static_cast<long long>(static_cast<unsigned>(h)) * 4294967296ll +
                      static_cast<long long>(__float2uint_rn(r));
  return b < 0.f ? -m : m;
}

// Layer outputs carry their completeness: every CTA adds (v << 8) + 1 into
// each of its rows (v = the row's partial on the 2^-32 grid), so a row is final
// once its low byte equals the number of clusters (one CTA of each cluster
// adds into every row).  The warp polls the two rows each lane holds (bounded)
// and returns their values.  False on abort or timeout.
// Lanes with valid == false take part in the warp-wide votes only.
__device__ bool poll_rows(const CParams& p, const long long* rows2, bool valid, float& y0, float& y1, unsigned site) {
  const unsigned n_cl = gridDim.x / kCl;
  const unsigned long long* src = reinterpret_cast<const unsigned long long*>(rows2);
  const long long t0 = clock64();
  y0 = y1 = 0.f;
  for (unsigned it = 0;; ++it) {
    const ulonglong2 v = valid ? ld_volatile_u64x2(src) : make_ulonglong2(n_cl, n_cl);
    const bool ok = (v.x & 0xFFull) == n_cl && (v.y & 0xFFull) == n_cl;
    if (__all_sync(kFull, ok)) {
      y0 = grid_to_float(static_cast<long long>(v.x) >> 8);
      y1 = grid_to_float(static_cast<long long>(v.y) >> 8);
      return true;
    }
    __nanosleep(64);
    if ((it & 255) == 255) {
      if (__any_sync(kFull, aborted(p))) return false;
      if (__any_sync(kFull, clock64() - t0 > p.spin_limit)) {
        if ((threadIdx.x & 31) == 0) {
          note_timeout(p, site);
          raise_abort(p);
        }
        return false;
      }
    }
  }
}

__device__ __forceinline__ float gelu_p(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

// ------------------------------------------------------------------ timeline (optional)

// Event times (%globaltimer, ns) of the call's third layer (the last one if
// fewer), row blockIdx.x (32 columns) of the caller's buffer: first
// occurrence, or latest for the *_LAST events.
enum : int { EV_Y_SEEN, EV_X_READY, EV_LOGIT_OUT, EV_LOGITS_IN, EV_TOPK_DONE, EV_ROUTED_ISSUE, EV_SHARED_DATA,
             EV_ROUTED_DATA, EV_PUSH_LAST, EV_DN_LAST, EV_STAGES_DONE, EV_REDUCED, EV_ISSUE_LAST, EV_DATA_LAST,
             EV_DN_A_FIRST, EV_A_WAIT_LAST, EV_PREP_B1, EV_PREP_Y, EV_PREP_B2, EV_ROUTER_B, EV_TOPK_SORTED,
             EV_BULK_ISSUED, EV_OPS_READY, EV_RANKS_OUT };
constexpr int kTlCols = 32;            // timeline row: events 0..23, accumulators 24..31

__device__ __forceinline__ void stamp(const CParams& p, int rel, int ev, bool latest = false) {
  if (!p.timeline) return;
  const int n_rel = p.l1 - p.l0;
  if (rel != (n_rel > 2 ? 2 : n_rel - 1)) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  unsigned long long* q = p.timeline + static_cast<size_t>(blockIdx.x) * kTlCols + ev;
  if (latest) atomicMax(q, t);
  else atomicCAS(q, 0ull, t);
}

// Accumulated times of the stamped layer at columns 24.. of row blockIdx.x:
// [0] gate/up compute, [1] down compute, [2] down wait for a, [3] data wait
// (routed stages), [4] gate/up stages, [5] down stages, [6] data wait
// (shared stages), [7] wait at the layer's end for the other warps' stages,
// all in ns summed over the CTA's consumer warps.
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void acc(const CParams& p, int rel, int slot, unsigned long long v) {
  if (!p.timeline) return;
  const int n_rel = p.l1 - p.l0;
  if (rel != (n_rel > 2 ? 2 : n_rel - 1)) return;
  atomicAdd(p.timeline + static_cast<size_t>(blockIdx.x) * kTlCols + 24 + slot, v);
}

// ------------------------------------------------------------------ units and stages

// The cluster's units of a layer (the same for every layer: only the experts
// behind the top-k positions change).  Routed unit i (position j, group G,
// i = j * f/64 + G) goes to cluster i mod n_cl; shared units go round-robin
// over every cluster, those with fewer routed units first
// (cluster_unit_owner_shared): routed work waits for the top-k and sets the
// layer's length, shared work fills the wait, which holds one or two units.
// A cluster runs its shared units first.
// Within each list a unit's down stage follows the gate/up stages of the next
// two units, so the other CTAs' values of a have normally arrived by the time
// a quad takes it.  Returns the number of units (> kMaxU: does not fit).
__device__ int build_tasks(const CParams& p, Smem& S, int cl, int n_cl) {
  const int nGf = p.f / 64, nGs = p.fs / 64, Ur = p.k * nGf;
  int n = 0, t = 0;
  int pend = -1, pend2 = -1;   // units whose down stages are still to be queued, oldest first
  auto push = [&](int kind, int tt, int ui) {
    CTask e;
    e.kind = static_cast<int8_t>(kind);
    e.tt = static_cast<int8_t>(tt);
    e.ui = static_cast<int8_t>(ui);
    e.pad = 0;
    e.src = static_cast<int16_t>(ui >= 0 ? S.unit_src[ui] : 0);
    e.G = static_cast<int16_t>(ui >= 0 ? S.unit_G[ui] : 0);
    S.tasks[t++] = e;
  };
  auto add_unit = [&](int src, int G) {
    if (n < kMaxU) {
      S.unit_src[n] = src;
      S.unit_G[n] = G;
      push(K_GU, 0, n);
      push(K_GU, 1, n);
      if (pend >= 0) push(K_DN, 0, pend);
      pend = pend2;
      pend2 = n;
    }
    ++n;
  };
  auto flush = [&]() {
    if (pend >= 0 && n <= kMaxU) push(K_DN, 0, pend);
    if (pend2 >= 0 && n <= kMaxU) push(K_DN, 0, pend2);
    pend = pend2 = -1;
  };
  for (int G = 0; G < nGs; ++G)
    if (cluster_unit_owner_shared(G, Ur, n_cl) == cl) add_unit(-1, G);
  flush();
  if (n <= kMaxU) push(K_TOPK, 0, -1);
  for (int i = 0; i < Ur; ++i)
    if (i % n_cl == cl) add_unit(i / nGf, i % nGf);
  flush();
  S.n_tasks = t;
  S.n_units = n < kMaxU ? n : kMaxU;
  S.n_stages = 3 * S.n_units;
  return n;
}

// ------------------------------------------------------------------ producer

// The producer's bounded wait for rank j of layer rel of the top-k, read
// from the rank word of the cluster's rank-0 CTA (whose top-k warp picks it);
// returns the expert, or -1 on abort or timeout.  The tag and the expert share
// one 32-bit word, so the word alone carries its own readiness (no fence on
// either side).
__device__ int wait_rank(const CParams& p, const Smem& S, int rel, int j) {
  const unsigned tag = 64u * static_cast<unsigned>(rel) + static_cast<unsigned>(j) + 1u;
  const uint32_t src = peer_addr(&S.rank_word[j], 0);
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    unsigned v;
    asm volatile("ld.volatile.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(src) : "memory");
    if ((v >> 8) == tag) return static_cast<int>(v & 0xFFu);
    if (clock64() - t0 > p.spin_limit) {
      note_timeout(p, W_P_TOPK);
      return -1;
    }
    if ((it & 15) == 15 && aborted(p)) return -1;
    __nanosleep(32);
  }
}

// Host-pool mode: the producer's bounded wait for layer l's plan word of rank
// j (published by cluster 0 after its slot-cache step; the launch's tag in the
// high half carries its readiness).  Returns the word, or 0 on abort or timeout.
__device__ unsigned long long wait_plan(const CParams& p, int l, int j) {
  const unsigned long long* src = p.plan + static_cast<size_t>(l) * 32 + j;
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(src) : "memory");
    if (static_cast<unsigned>(w >> 32) == p.tag) return w;
    if (clock64() - t0 > p.spin_limit) {
      note_timeout(p, W_PLAN);
      return 0ull;
    }
    if ((it & 15) == 15 && aborted(p)) return 0ull;
    __nanosleep(64);
  }
}

template <bool kPool>
__device__ void producer(const CParams& p, Smem& S, unsigned rank) {
  const int n_rel = p.l1 - p.l0;
  const uint32_t tile_bytes = static_cast<uint32_t>(p.d / 64) * kGroupBytes;   // gate/up tile = down slice
  const int R = p.d / 64;                                                     // 16-row down tiles per CTA
  uint32_t u_issued = 0;
  int rrow_last = -1;      // layer of the last router-row copy
  bool stop = false;
  for (int rel = 0; rel < n_rel && !stop; ++rel) {
    const CLayer* L = p.layers + (p.l0 + rel);
    // the layer's addresses once, before any wait, and its down tensor maps
    // into the TMA unit's descriptor cache
    const uint8_t* const Lsh = L->shared;
    const uint8_t* const Lex = L->experts;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L->dn_shared)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L->dn_routed)) : "memory");
    if (static_cast<int>(blockIdx.x) < p.E) {
      if (!wait_one(p, &S.rrow_empty, (static_cast<uint32_t>(rel) & 1u) ^ 1u, W_RROW_EMPTY)) {
        raise_abort(p);
        break;
      }
      const uint16_t* rw = L->router_w;
      mbar_arrive_expect_tx(&S.rrow_full, static_cast<uint32_t>(p.d) * 2u);
      bulk_g2s(S.rrow, rw + static_cast<size_t>(blockIdx.x) * p.d, static_cast<uint32_t>(p.d) * 2u, &S.rrow_full);
      rrow_last = rel;
    }
    int s = 0;
    unsigned plan_known = 0;   // host pool: ranks whose plan word this layer has been read
    for (int i = 0; i < S.n_tasks; ++i) {
      const CTask t = S.tasks[i];
      if (t.kind == K_TOPK) continue;
      // a routed stage needs only its own rank of the top-k
      const int e = t.src < 0 ? 0 : wait_rank(p, S, rel, t.src);
      if (e < 0) {
        raise_abort(p);
        stop = true;
        break;
      }
      // host pool: where the expert is (a slot, filled by this step if a miss)
      int se = e;
      bool miss = false;
      if (kPool && t.src >= 0) {
        if (!(plan_known & (1u << t.src))) {
          const unsigned long long w = wait_plan(p, p.l0 + rel, t.src);
          if (w == 0ull) {
            raise_abort(p);
            stop = true;
            break;
          }
          S.plan_w[t.src] = w;
          plan_known |= 1u << t.src;
        }
        const unsigned long long w = S.plan_w[t.src];
        se = static_cast<int>((w >> 16) & 0xFFFFu);
        miss = ((w >> 8) & 1u) == 0u;
      }
      const uint32_t u = static_cast<uint32_t>(rel) * S.n_stages + s++;
      const int slot = u % kNS;
      if (!wait_one(p, &S.empty[slot], ((u / kNS) & 1u) ^ 1u, W_EMPTY)) {
        raise_abort(p);
        stop = true;
        break;
      }
      if (miss) {
        // the consumers copy this stage from the mapped pool into the ring and
        // into the slot (plain loads: no bulk copy reads host memory)
        const long long gu_r = static_cast<long long>(p.f / 8) * R * kGroupBytes;
        const uint8_t* src = L->pool + static_cast<long long>(e) * p.expert_stride;
        uint8_t* dst = const_cast<uint8_t*>(Lex) + static_cast<long long>(se) * p.expert_stride;
        long long off;
        int fstride;
        if (t.kind == K_GU) {
          off = static_cast<long long>(8 * t.G + 2 * static_cast<int>(rank) + t.tt) * tile_bytes;
          fstride = 0;
        } else {
          off = gu_r + (static_cast<long long>(R) * rank * (p.f / 64) + t.G) * kGroupBytes;
          fstride = (p.f / 64) * kGroupBytes;
        }
        S.fill_src[slot] = src + off;
        S.fill_dst[slot] = dst + off;
        S.fill_stride[slot] = fstride;
        mbarrier_arrive(&S.full[slot]);
      } else {
        if (kPool) S.fill_src[slot] = nullptr;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&S.full[slot], tile_bytes);
        if (t.kind == K_GU) {
          const uint8_t* base = t.src < 0 ? Lsh : Lex + static_cast<long long>(se) * p.expert_stride;
          const size_t tile = static_cast<size_t>(8 * t.G + 2 * static_cast<int>(rank) + t.tt);
          bulk_g2s(S.ring[slot], base + tile * tile_bytes, tile_bytes, &S.full[slot]);
        } else {
          tma_load_3d(S.ring[slot], t.src < 0 ? &L->dn_shared : &L->dn_routed, t.G * (kGroupBytes / 4),
                      R * static_cast<int>(rank), se, &S.full[slot]);
        }
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
    // the last router-row copy completes phase rrow_last of rrow_full (its
    // consumers may have given up before waiting for it)
    if (rrow_last >= 0) mbar_wait_bounded(&S.rrow_full, static_cast<uint32_t>(rrow_last) & 1u, p.err);
  }
}

// ------------------------------------------------------------------ top-k

// Polls the cluster's replica of layer l's tagged logits until every entry
// carries this launch's tag, then takes the top-k (ties to the lower index)
// and the softmax gates.  Each lane holds up to NPL logits (4 for at most 128
// experts, else 8) sorted by (value desc, index asc); a round picks the
// warp-wide best head with one reduction on the high 32 bits of the
// order-preserving unsigned image of the int64 logit, and further reductions
// (low bits, then index) only when several heads tie there; the winning lane
// records it directly.
template <int NPL>
__device__ bool topk_layer(const CParams& p, Smem& S, int l, int32_t* ids, float* gates, unsigned seq_base) {
  const int lane = threadIdx.x & 31;
  const unsigned cl = cluster_idx(), n_cl = cluster_count();
  const unsigned long long* lg = p.tlog + (static_cast<size_t>(l) * n_cl + cl) * p.E * 2;
  unsigned long long key[NPL];
  int idx[NPL];
  // two polls in flight: the next one is issued before this one is checked
  const ulonglong2 absent = make_ulonglong2(static_cast<unsigned long long>(p.tag) << 32,
                                            static_cast<unsigned long long>(p.tag) << 32);
  ulonglong2 cur[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) cur[i] = lane + 32 * i < p.E ? ld_volatile_u64x2(lg + 2 * (lane + 32 * i)) : absent;
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    ulonglong2 nxt[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) nxt[i] = lane + 32 * i < p.E ? ld_volatile_u64x2(lg + 2 * (lane + 32 * i)) : absent;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      const ulonglong2 v = cur[i];
      ok = ok && static_cast<unsigned>(v.x >> 32) == p.tag && static_cast<unsigned>(v.y >> 32) == p.tag;
      key[i] = e < p.E ? ((v.y << 32) | (v.x & 0xFFFFFFFFull)) ^ 0x8000000000000000ull : 0ull;
      idx[i] = e < p.E ? e : 0x7fffffff;
    }
    if (__all_sync(kFull, ok)) {
      if (lane == 0) stamp(p, l - p.l0, EV_LOGITS_IN);
      break;
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) cur[i] = nxt[i];
    if ((it & 63) == 63) {
      if (__any_sync(kFull, aborted(p))) return false;
      if (__any_sync(kFull, clock64() - t0 > p.spin_limit)) {
        if (lane == 0) {
          note_timeout(p, W_LOGITS);
          raise_abort(p);
        }
        return false;
      }
    }
  }
  // absent entries (key 0, index max) sort last and are never picked (k <= E)
#pragma unroll
  for (int i = 1; i < NPL; ++i) {
#pragma unroll
    for (int j = i; j > 0; --j) {
      const bool sw = key[j] > key[j - 1];
      const unsigned long long tk = sw ? key[j] : key[j - 1];
      key[j] = sw ? key[j - 1] : key[j];
      key[j - 1] = tk;
      const int ti = sw ? idx[j] : idx[j - 1];
      idx[j] = sw ? idx[j - 1] : idx[j];
      idx[j - 1] = ti;
    }
  }
  if (lane == 0) stamp(p, l - p.l0, EV_TOPK_SORTED);
  int head = 0;
  for (int j = 0; j < p.k; ++j) {
    unsigned long long hk = 0ull;
    int he = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i == head) {
        hk = key[i];
        he = idx[i];
      }
    const unsigned hi = static_cast<unsigned>(hk >> 32), lo = static_cast<unsigned>(hk);
    const unsigned mh = __reduce_max_sync(kFull, hi);
    bool c = hi == mh;
    unsigned bal = __ballot_sync(kFull, c);
    if (__popc(bal) > 1) {
      const unsigned ml = __reduce_max_sync(kFull, c ? lo : 0u);
      c = c && lo == ml;
      bal = __ballot_sync(kFull, c);
      if (__popc(bal) > 1) {
        const unsigned me = __reduce_min_sync(kFull, c ? static_cast<unsigned>(he) : 0xFFFFFFFFu);
        c = c && static_cast<unsigned>(he) == me;
      }
    }
    // the one winning lane records rank j and publishes it, tagged with the
    // layer and the rank, in this CTA's rank word j, which the cluster's four
    // producers read (three of them through distributed shared memory) to
    // load its expert while the warp picks the rest
    if (c) {
      ids[j] = he;
      S.topv[j] = static_cast<long long>(hk ^ 0x8000000000000000ull);
      ++head;
      *reinterpret_cast<volatile unsigned*>(&S.rank_word[j]) =
          (seq_base + static_cast<unsigned>(j) + 1u) << 8 | static_cast<unsigned>(he);
    }
  }
  __syncwarp();
  if (lane == 0) stamp(p, l - p.l0, EV_RANKS_OUT);
  float ex = 0.f;
  if (lane < p.k) ex = expf(ll_to_float(S.topv[lane] - S.topv[0]) * 9.094947017729282e-13f);   // 2^-40
  float sum = 0.f;
  for (int j = 0; j < p.k; ++j) sum += __shfl_sync(kFull, ex, j);
  const float gv = ex / sum;
  // lane r < 4 writes the k gates into CTA r (itself included) and then arrives
  // there on the top-k barrier (release, cluster scope: its own stores first)
  for (int jj = 0; jj < p.k; ++jj) {
    const float g = __shfl_sync(kFull, gv, jj);
    if (lane < kCl) st_peer_f32(peer_addr(&gates[jj], static_cast<unsigned>(lane)), g);
  }
  if (lane < kCl) arrive_peer(peer_addr(&S.topk_bar, static_cast<unsigned>(lane)));
  __syncwarp();
  return true;
}

// Host-pool mode, cluster 0's top-k warp: the layer's slot-cache step for
// the token (the same rules as the per-layer kernels: hits refresh their
// slot's last use; misses, in top-k order, take among the slots this step has
// not touched the smallest (last use, slot) under LRU, or (use count of the
// slot's expert, last use, slot) under LFU, an empty slot counting -1), then
// the trace record for the host, the counters, and one plan word per rank
// for every producer of the grid.
__device__ void pool_step(const CParams& p, Smem& S, int rel) {
  const int lane = threadIdx.x & 31, k = p.k, N = p.n_slots, l = p.l0 + rel;
  const CLayer* L = p.layers + l;
  const long long t = S.args.step;
  const bool lfu = p.policy == 1;
  const int32_t* ids = S.ids[rel & 1];
  int eos[8];
  long long lu[8], uc[8];
  unsigned used = 0, hits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int sl = lane + 32 * i;
    eos[i] = sl < N ? __ldcg(&L->expert_of_slot[sl]) : -1;
    lu[i] = sl < N ? __ldcg(&L->last_use[sl]) : LLONG_MAX;
    uc[i] = (!lfu || sl >= N) ? 0 : (eos[i] >= 0 ? __ldcg(&L->use_count[eos[i]]) : -1);
    if (sl >= N) used |= 1u << i;
  }
  for (int j = 0; j < k; ++j) {
    const int sl = __ldcg(&L->slot_of_expert[ids[j]]);
    if (sl >= 0) {
      hits |= 1u << j;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == sl) {
          used |= 1u << i;
          lu[i] = t;
        }
    }
  }
  int32_t* rec = p.host_rec + static_cast<size_t>(rel) * (1 + 6 * k);
  int n_miss = 0;
  for (int j = 0; j < k; ++j) {
    const int ej = ids[j];
    int slot, ev = -1;
    if (hits & (1u << j)) {
      slot = __ldcg(&L->slot_of_expert[ej]);
    } else {
      long long bc = LLONG_MAX, bv = LLONG_MAX;
      int bs = INT_MAX;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sl = lane + 32 * i;
        const bool better = uc[i] < bc || (uc[i] == bc && (lu[i] < bv || (lu[i] == bv && sl < bs)));
        if (!(used & (1u << i)) && better) {
          bc = uc[i];
          bv = lu[i];
          bs = sl;
        }
      }
#pragma unroll
      for (int m = 16; m; m >>= 1) {
        const long long oc = shfl_xor_i64(bc, m);
        const long long ov = shfl_xor_i64(bv, m);
        const int os = __shfl_xor_sync(kFull, bs, m);
        if (oc < bc || (oc == bc && (ov < bv || (ov == bv && os < bs)))) {
          bc = oc;
          bv = ov;
          bs = os;
        }
      }
      slot = bs;
      int my_ev = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == bs) {
          my_ev = eos[i];
          eos[i] = ej;
          lu[i] = t;
          used |= 1u << i;
        }
      ev = __shfl_sync(kFull, my_ev, bs & 31);
      if (lane == 0) {
        if (ev >= 0) L->slot_of_expert[ev] = -1;
        L->slot_of_expert[ej] = bs;
        rec[1 + 2 * n_miss] = ej;
        rec[2 + 2 * n_miss] = bs;
      }
      ++n_miss;
    }
    if (lane == 0) {
      int32_t* tr = rec + 1 + 2 * k + 4 * j;
      tr[0] = ej;
      tr[1] = (hits >> j) & 1u;
      tr[2] = slot;
      tr[3] = ev;
      // every producer of the grid reads where rank j's expert is
      const unsigned long long w = static_cast<unsigned long long>(p.tag) << 32 |
                                   static_cast<unsigned long long>(slot) << 16 |
                                   static_cast<unsigned long long>((hits >> j) & 1u) << 8 |
                                   static_cast<unsigned long long>(ej);
      asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p.plan + static_cast<size_t>(l) * 32 + j), "l"(w)
                   : "memory");
    }
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int sl = lane + 32 * i;
    if (sl < N) {
      L->expert_of_slot[sl] = eos[i];
      L->last_use[sl] = lu[i];
    }
  }
  if (lane == 0) {
    if (lfu)
      for (int j = 0; j < k; ++j) L->use_count[ids[j]] += 1;
    rec[0] = n_miss;
    p.lru_counts[2 * l + 0] += k - n_miss;
    p.lru_counts[2 * l + 1] += n_miss;
  }
  __syncwarp();
}

// Rank 0 of each cluster picks the cluster's top-k for its four CTAs (one
// poller per cluster, and the four see the same ranks at the same time).
// Then, in every CTA, the warp zeroes the CTA's share of the vector layer
// rel + 1 adds into: the layer's logits exist, so every CTA has finished the
// previous layer's input step, the last reader of that vector.  The fence
// that makes the zeros visible before this CTA's next reduction runs here,
// off the layer's critical path; the zero barrier hands it to the reduction.
template <bool kPool>
__device__ void topk_warp(const CParams& p, Smem& S) {
  const int lane = threadIdx.x & 31;
  const int n_rel = p.l1 - p.l0, d = p.d;
  for (int rel = 0; rel < n_rel; ++rel) {
    if (cluster_rank() == 0) {
      // the layer's logits need the previous layer's output, which needs this
      // CTA's stages of it: wait for those (suspended, not spinning) before
      // polling, so the poll does not take issue slots from this scheduler's
      // consumer warps during the stages
      if (rel > 0 && !wait_warp(p, &S.end_bar, static_cast<uint32_t>(rel - 1) & 1u, W_END_STAGES)) {
        raise_abort(p);
        return;
      }
      int32_t* sid = S.ids[rel & 1];
      float* sg = S.gates[rel & 1];
      const unsigned base = 64u * static_cast<unsigned>(rel);
      const bool ok = p.E <= 128 ? topk_layer<4>(p, S, p.l0 + rel, sid, sg, base)
                                 : topk_layer<8>(p, S, p.l0 + rel, sid, sg, base);
      if (!ok) return;
      if (kPool && blockIdx.x == 0) pool_step(p, S, rel);
      if (lane == 0) stamp(p, rel, EV_TOPK_DONE);
      if (blockIdx.x == 0 && lane < p.k && rel < S.args.dbg_layers) {
        const DevCallArgs* A = &S.args;
        const size_t o = (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.k + lane;
        if (A->dbg_ids) A->dbg_ids[o] = sid[lane];
        if (A->dbg_gates) A->dbg_gates[o] = sg[lane];
      }
      __syncwarp();
    }
    if (!mbar_wait_cluster(p, &S.topk_bar, static_cast<uint32_t>(rel) & 1u, W_DN_TOPK)) {
      raise_abort(p);
      return;
    }
    if (rel > 0) {
      long long* yz = p.ybuf + static_cast<size_t>((rel + 1) % 3) * d;
      const int share = (d + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
      for (int zj = lane; zj < share; zj += 32) {
        const int zi = static_cast<int>(blockIdx.x) * share + zj;
        if (zi < d) yz[zi] = 0;
      }
      __threadfence();
      fence_proxy_async_global();
    }
    __syncwarp();
    if (lane == 0) mbarrier_arrive(&S.zero_bar);
  }
}

// ------------------------------------------------------------------ consumers

// Logit of router row blockIdx.x of layer rel: the warps' exact partials
// (formed with x in prep) summed, plus the bias, published with this launch's
// tag in both 64-bit words.  Run by consumer warp 0 in prep, right after the
// barrier that completes the partials (the operands of x come after).
__device__ void router_publish(const CParams& p, Smem& S, int cw, int rel, float bv) {
  if (static_cast<int>(blockIdx.x) >= p.E || cw != 0) return;
  const int lane = threadIdx.x & 31;
  if (lane == 0) stamp(p, rel, EV_ROUTER_B);
  // every lane forms the same logit (the warps' parts in warp order, plus the bias)
  long long acc = 0;
  for (int w = 0; w < kNC; ++w) acc += S.rlog[w];
  const DevCallArgs* A = &S.args;
  if (A->bias) {   // bv: this CTA's bias entry, loaded at the start of the layer
    if (!(fabsf(bv) < 1048576.f)) {
      if (lane == 0) atomicOr(p.err, ERR_ROUTER_DOMAIN);
    } else {
      acc += bias_fix40(bv);
    }
  }
  __syncwarp();
  if (lane == 0) mbarrier_arrive(&S.rrow_empty);   // every warp read the row before the barrier
  const long long logit = acc;
  if (lane == 0 && A->dbg_logits && rel < A->dbg_layers)
    A->dbg_logits[(static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.E + blockIdx.x] = logit;
  const unsigned long long tg = static_cast<unsigned long long>(p.tag) << 32;
  const unsigned long long ua = static_cast<unsigned long long>(logit);
  const unsigned n_cl = cluster_count();
  for (unsigned c = lane; c < n_cl; c += 32)
    st_volatile_u64x2(p.tlog + ((static_cast<size_t>(p.l0 + rel) * n_cl + c) * p.E + blockIdx.x) * 2,
                      (ua & 0xFFFFFFFFull) | tg, (ua >> 32) | tg);
  if (lane == 0) stamp(p, rel, EV_LOGIT_OUT);
  __syncwarp();
}

// Layer input: wait for the previous layer's output vector, add it to this
// CTA's copy of the residual stream, RMS norm in a fixed order (every CTA gets
// the same x), x as plain bf16, as mma B fragments and as per-group sums.
__device__ bool prep(const CParams& p, Smem& S, int cw, int rel, int& round, unsigned rank, float bias_v) {
  const int lane = threadIdx.x & 31;
  const int d = p.d, nGd = d / 64;
  const DevCallArgs* A = &S.args;
  constexpr int kGW = (kMaxG + kNC - 1) / kNC;   // groups per warp at most
  float r = 1.f;
  if (rel == 0) {
    // the call's input: every CTA reads all of h_in; warp cw takes groups cw,
    // cw + kNC, ...; lane holds elements 64G + 2*lane, +1
    uint32_t hv[kGW];
#pragma unroll
    for (int i = 0; i < kGW; ++i) {
      const int G = cw + kNC * i;
      hv[i] = G < nGd ? __ldcg(reinterpret_cast<const unsigned*>(A->h_in + 64 * G) + lane) : 0u;
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kGW; ++i) {
      const int G = cw + kNC * i;
      if (G < nGd) {
        reinterpret_cast<uint32_t*>(S.h)[32 * G + lane] = hv[i];
        const float a = bf16_bits_to_float(static_cast<uint16_t>(hv[i] & 0xFFFFu));
        const float b = bf16_bits_to_float(static_cast<uint16_t>(hv[i] >> 16));
        ss += a * a;
        ss += b * b;
      }
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(kFull, ss, m);
    if (lane == 0) S.red[cw] = ss;
    if (!consumer_barrier(p, S, ++round)) return false;   // red[] and S.h complete
    if (p.prenorm) {
      float tot = 0.f;
      for (int w = 0; w < kNC; ++w) tot += S.red[w];
      r = 1.0f / sqrtf(tot / static_cast<float>(d) + p.eps);
    }
  } else {
    // the previous layer's output: every CTA polls the whole vector (element
    // pairs spread over the warps; all rows complete also means every CTA of
    // the grid has finished the previous layer's input step), adds it to its
    // residual copy in place and sums the squares; one CTA barrier then
    // completes h (the previous layer's reads of h all precede its stages).
    const long long* yin = p.ybuf + static_cast<size_t>((rel - 1) % 3) * d;
    const int npair = d / 2;                          // element pairs of the vector
    float ss = 0.f;
    for (int j0 = cw * 32; j0 < npair; j0 += kNC * 32) {
      const int j = j0 + lane, e = 2 * j;
      const bool valid = j < npair;
      float y0, y1;
      if (!poll_rows(p, yin + e, valid, y0, y1, W_Y_POLL)) return false;
      if (valid) {
        const uint32_t hv = reinterpret_cast<const uint32_t*>(S.h)[j];
        const float a = bf16_bits_to_float(static_cast<uint16_t>(hv & 0xFFFFu)) + y0;
        const float b = bf16_bits_to_float(static_cast<uint16_t>(hv >> 16)) + y1;
        const uint32_t v =
            static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
        reinterpret_cast<uint32_t*>(S.h)[j] = v;   // in place: each word by its own lane
        const float ha = bf16_bits_to_float(static_cast<uint16_t>(v & 0xFFFFu));
        const float hb = bf16_bits_to_float(static_cast<uint16_t>(v >> 16));
        ss += ha * ha + hb * hb;
        if (blockIdx.x == 0 && A->dbg_y && rel - 1 < A->dbg_layers) {
          float* dy = A->dbg_y + (static_cast<size_t>(rel - 1) * A->tok_total + A->tok_off) * d + e;
          dy[0] = y0;
          dy[1] = y1;
        }
      }
    }
    if (cw == 0 && lane == 0) stamp(p, rel, EV_Y_SEEN);
#pragma unroll
    for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(kFull, ss, m);
    if (lane == 0) S.red[cw] = ss;
    if (!consumer_barrier(p, S, ++round)) return false;   // red[] and S.h complete
    if (cw == 0 && lane == 0) stamp(p, rel, EV_PREP_B1);
    if (p.prenorm) {
      float tot = 0.f;
      for (int w = 0; w < kNC; ++w) tot += S.red[w];
      r = 1.0f / sqrtf(tot / static_cast<float>(d) + p.eps);
    }
  }
  if (cw == 0 && lane == 0) stamp(p, rel, EV_PREP_B2);
  // x first, with the router row of this CTA's expert dotted into it (each
  // warp adds its elements' exact products: RNE onto the 2^-40 grid, integer
  // sums, so the split does not change the logit); the warps' partials are
  // complete at the next barrier, after which warp 0 publishes the logit while
  // the others build the matrix operands of x
  const bool routes = static_cast<int>(blockIdx.x) < p.E;
  if (routes && !wait_warp(p, &S.rrow_full, static_cast<uint32_t>(rel) & 1u, W_RROW_FULL)) {
    raise_abort(p);
    return false;
  }
  Fix40 fx;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kGW; ++i) {
    const int G = cw + kNC * i;
    if (G >= nGd || !routes) continue;
    uint32_t xv = reinterpret_cast<const uint32_t*>(S.h)[32 * G + lane];
    if (p.prenorm) {
      const float a = bf16_bits_to_float(static_cast<uint16_t>(xv & 0xFFFFu)) * r;
      const float b = bf16_bits_to_float(static_cast<uint16_t>(xv >> 16)) * r;
      xv = static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
    }
    {
      const uint32_t wv = reinterpret_cast<const uint32_t*>(S.rrow)[32 * G + lane];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float pw = hh ? half_hi(wv) : half_lo(wv);
        const float px = bf16_bits_to_float(static_cast<uint16_t>(hh ? (xv >> 16) : (xv & 0xFFFFu)));
        const float prod = pw * px;   // exact: 11-bit x 8-bit significands
        const bool okp = fabsf(prod) < 2048.f;
        bad |= !okp;
        fix40_add(fx, okp ? prod * 1099511627776.0f : 0.f);
      }
    }
  }
  if (routes) {
    long long acc = fix40_value(fx);
#pragma unroll
    for (int m = 16; m; m >>= 1) acc += shfl_xor_i64(acc, m);
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(p.err, ERR_ROUTER_DOMAIN);
    if (lane == 0) S.rlog[cw] = acc;
  }
  if (!consumer_barrier(p, S, ++round)) return false;   // the router partials complete
  if (cw == 0 && lane == 0) stamp(p, rel, EV_X_READY);
  // warp 0 forms and publishes the logit (it arrives on the operands barrier
  // first: the logit is the longer chain), the other warps build the matrix
  // operands of x: fp16 mma B fragments and per-group sums
  ++round;
  if (cw == 0) {
    __syncwarp();
    if (lane == 0) mbarrier_arrive(&S.cbar);
    router_publish(p, S, cw, rel, bias_v);
  } else {
    for (int G = cw - 1; G < nGd; G += kNC - 1) {
      uint32_t xv = reinterpret_cast<const uint32_t*>(S.h)[32 * G + lane];
      if (p.prenorm) {   // the same rounding as above: the same x
        const float a = bf16_bits_to_float(static_cast<uint16_t>(xv & 0xFFFFu)) * r;
        const float b = bf16_bits_to_float(static_cast<uint16_t>(xv >> 16)) * r;
        xv = static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
      }
      // fp16 B fragments: element e = 2*lane of the group lands in (t4, st, pos)
      const float xa = bf16_bits_to_float(static_cast<uint16_t>(xv & 0xFFFFu));
      const float xb = bf16_bits_to_float(static_cast<uint16_t>(xv >> 16));
      const __half ha = __float2half_rn(xa), hb = __float2half_rn(xb);
      if (__any_sync(kFull, !(fabsf(xa) < 65504.f && fabsf(xb) < 65504.f)) && lane == 0)
        atomicOr(p.err, ERR_PF_RANGE);
      const int e = 2 * lane, st = e >> 4, w = e & 15;
      const int t4 = (w & 7) >> 1, hi = w >> 3;
      reinterpret_cast<uint32_t*>(S.xp)[((G * 4 + t4) * 4 + st) * 2 + hi] =
          static_cast<uint32_t>(__half_as_ushort(ha)) | (static_cast<uint32_t>(__half_as_ushort(hb)) << 16);
      float gs = __half2float(ha) + __half2float(hb);
#pragma unroll
      for (int m = 16; m; m >>= 1) gs += __shfl_xor_sync(kFull, gs, m);
      if (lane == 0) S.xg[G] = gs;
      if (blockIdx.x == 0 && A->dbg_x && rel < A->dbg_layers)
        reinterpret_cast<uint32_t*>(A->dbg_x + (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * d)[32 * G + lane] =
            xv;
    }
    __syncwarp();
    if (lane == 0) mbarrier_arrive(&S.cbar);
  }
  const bool ok = wait_warp(p, &S.cbar, static_cast<uint32_t>(round - 1) & 1u, W_CBAR);   // x's operands complete
  if (!ok) raise_abort(p);
  __syncwarp();
  if (cw == 1 && lane == 0) stamp(p, rel, EV_OPS_READY);
  return ok;
}

// Groups [G0, G1) of a gate/up tile: partial gate and up sums of row g.  With
// P = sum_k x_k (1024 + q_k) (gate rows) and sum_k x_k (1024 + 16 q_k) (up
// rows), sum_k x_k (s q_k + b) = s P + (b - 1024 s) X for the gate rows and
// (s / 16) P + (b - 64 s) X for the up rows, X = the group's sum of x.
__device__ void gu_groups(Smem& S, const uint8_t* tile, int G0, int G1, float& ga, float& ua) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
#pragma unroll 4   // four groups' loads and MMAs in flight per warp (2 and 8 measured slower)
  for (int G = G0; G < G1; ++G) {
    const uint8_t* blk = tile + static_cast<size_t>(G) * kGroupBytes;
    const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
    const uint4* xf = reinterpret_cast<const uint4*>(S.xp) + (G * 4 + t4) * 2;
    const uint4 x01 = xf[0], x23 = xf[1];
    float c0[4], c1[4];
    mma_nib<true>(c0, q.x, x01.x, x01.y);
    mma_nib<true>(c1, q.y, x01.z, x01.w);
    mma_nib<false>(c0, q.z, x23.x, x23.y);
    mma_nib<false>(c1, q.w, x23.z, x23.w);
    const float X = S.xg[G];
    const float sg = half_lo(sbv.x), bg = half_hi(sbv.x), su = half_lo(sbv.y), bu = half_hi(sbv.y);
    ga += sg * (c0[0] + c1[0]) + fmaf(-1024.f, sg, bg) * X;
    ua += (su * 0.0625f) * (c0[2] + c1[2]) + fmaf(-64.f, su, bu) * X;
  }
}

// Epilogue of gate/up tile tt of a unit: a = GELU(gate) * up for its 8 rows,
// split into fp16 hi + lo, written as down B fragments into the unit's a-slot
// of every CTA of the cluster, with the tile's sum of a; then one remote
// arrival on each CTA's a_full barrier.  Tile tt of rank r holds the unit's
// intermediate rows 16r + 8tt + g, i.e. k16 step r, in-step rows 8tt + g.
__device__ void gu_push(const CParams& p, Smem& S, int rel, const CTask& t, unsigned rank, float ga, float ua) {
  const int lane = threadIdx.x & 31;
  const float av = gelu_p(ga, p.gelu) * ua;
  if (__any_sync(kFull, !(fabsf(av) < 65504.f)) && lane == 0) atomicOr(p.err, ERR_PF_RANGE);
  const __half hh = __float2half_rn(av);
  const __half hl = __float2half_rn(av - __half2float(hh));
  const uint32_t hi = __half_as_ushort(hh), lo = __half_as_ushort(hl);
  float sh = __half2float(hh), sl = __half2float(hl);
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    sh += __shfl_xor_sync(kFull, sh, m);
    sl += __shfl_xor_sync(kFull, sl, m);
  }
  // word w = (hi/lo column, t4) = 4 * column + t4 packs rows 2*t4 and 2*t4 + 1
  // of that column (held by lanes 8*t4 and 8*t4 + 4); lane w & 7 forms it
  const int par = (lane >> 2) & 1, t4w = lane & 3;
  const uint32_t h0 = __shfl_sync(kFull, hi, 8 * t4w), h1 = __shfl_sync(kFull, hi, 8 * t4w + 4);
  const uint32_t l0 = __shfl_sync(kFull, lo, 8 * t4w), l1 = __shfl_sync(kFull, lo, 8 * t4w + 4);
  const uint32_t word = par ? (l0 | (l1 << 16)) : (h0 | (h1 << 16));
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __shfl_sync(kFull, word, i);
  // lane r < 4 writes this tile's eight words (one 32-byte block) and its sum
  // into CTA r of the cluster with asynchronous remote stores that count their
  // bytes on that CTA's a_full barrier (no fence, nothing to wait for here);
  // each CTA expects the unit's 8 x 36 bytes on its own barrier, once per use,
  // when it pushes its first tile of the unit
  const int aslot = (rel & 1) * kMaxU + t.ui;
  if (lane < kCl) {
    const unsigned r = static_cast<unsigned>(lane);
    if (t.tt == 0 && r == rank) mbar_arrive_expect_tx(&S.a_full[aslot], kAPushBytes);
    const uint32_t a = peer_addr(&S.abuf[aslot][(2 * rank + t.tt) * 8], r);
    const uint32_t bar = peer_addr(&S.a_full[aslot], r);
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(a),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(bar)
                 : "memory");
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     a + 16),
                 "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(bar)
                 : "memory");
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     peer_addr(&S.tsum[aslot][2 * rank + t.tt], r)),
                 "r"(__float_as_uint(sh + sl)), "r"(bar)
                 : "memory");
  }
  __syncwarp();
  if (lane == 0) stamp(p, rel, EV_PUSH_LAST, true);
}

// Host-pool miss: warp qw copies the part of the stage it will multiply (its
// groups of a gate/up tile, or its row tiles of a down slice) from the mapped
// pool into the ring slot and into the expert's device slot, eight 16-byte
// loads in flight per lane.
__device__ void fill_stage(const CParams& p, Smem& S, int slot, const CTask& t, int qw) {
  const int lane = threadIdx.x & 31;
  const uint8_t* src = S.fill_src[slot];
  uint8_t* dst = S.fill_dst[slot];
  const int fs = S.fill_stride[slot];
  uint8_t* ring = S.ring[slot];
  const int nGd = p.d / 64;
  constexpr int kPer = kGroupBytes / 16;   // 16-byte pieces per 576-byte block
  int n16, g0 = 0;
  if (t.kind == K_GU) {
    const int cgu = (nGd + kQW - 1) / kQW;
    g0 = qw * cgu;
    n16 = max(0, min(nGd, g0 + cgu) - g0) * kPer;
  } else {
    n16 = (qw < nGd ? (nGd - qw + kQW - 1) / kQW : 0) * kPer;
  }
  // byte offset of piece i in the pool / slot, and in the ring
  auto offs = [&](int i, long long& go, int& ro) {
    if (t.kind == K_GU) {
      ro = g0 * kGroupBytes + 16 * i;
      go = ro;
    } else {
      const int T = qw + kQW * (i / kPer), o = 16 * (i % kPer);
      ro = T * kGroupBytes + o;
      go = static_cast<long long>(T) * fs + o;
    }
  };
  for (int i0 = 0; i0 < n16; i0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u + lane;
      if (i < n16) {
        long long go;
        int ro;
        offs(i, go, ro);
        v[u] = *reinterpret_cast<const uint4*>(src + go);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u + lane;
      if (i < n16) {
        long long go;
        int ro;
        offs(i, go, ro);
        *reinterpret_cast<uint4*>(ring + ro) = v[u];
        *reinterpret_cast<uint4*>(dst + go) = v[u];
      }
    }
  }
  __syncwarp();
}

// Gate/up stage: warp qw of the quad takes groups [qw * cgu, (qw + 1) * cgu);
// the last warp of the quad to finish sums the four partials in warp order and
// pushes a.
__device__ void stage_gu(const CParams& p, Smem& S, int qw, int rel, int slot, const CTask& t, unsigned rank) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nGd = p.d / 64, cgu = (nGd + kQW - 1) / kQW;
  const int g0 = qw * cgu, g1 = min(nGd, g0 + cgu);
  float ga = 0.f, ua = 0.f;
  gu_groups(S, S.ring[slot], g0, g1, ga, ua);
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

// RNE(v * 2^32) for |v| < 2^17 with 32-bit conversions only (conversions to
// 64-bit integers run on this part's narrow FP64 path: see grid_to_float):
// for a = |v| * 2^8, floor(a) and a - floor(a) are exact in fp32, so
// RNE(|v| 2^32) = floor(a) 2^24 + RNE((a - floor(a)) 2^24).
__device__ __forceinline__ long long grid_from_float(float v) {
  const float a = fabsf(v) * 256.f;
  const float fa = floorf(a);
  const long long m = static_cast<long long>(static_cast<int>(fa)) * 16777216ll +
                      static_cast<long long>(__float2uint_rn((a - fa) * 16777216.f));
  return v < 0.f ? -m : m;
}

// Down stage: this CTA's d/64 row tiles of the unit's group, warp qw of the
// quad taking tiles qw, qw + 4, ...; every tile uses the same 64 values of a
// (fp16 hi + lo in two B columns).  Rows g and g + 8 of a tile follow the
// gate/up epilogue's two forms (1024 + q and 1024 + 16 q).
__device__ bool stage_dn(const CParams& p, Smem& S, int quad, int qw, int rel, int slot, const CTask& t,
                         unsigned long long* t_ready) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int aslot = (rel & 1) * kMaxU + t.ui;
  if (!mbar_wait_cluster(p, &S.a_full[aslot], (static_cast<uint32_t>(rel) >> 1) & 1u, W_A_FULL)) return false;
  if (lane == 0) {
    stamp(p, rel, EV_DN_A_FIRST);
    stamp(p, rel, EV_A_WAIT_LAST, true);
  }
  if (p.timeline) *t_ready = now_ns();
  float As = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) As += S.tsum[aslot][i];
  // B fragments of lane (g, t4): column g & 1 (hi / lo), k16 step st = sending
  // rank, b0 / b1 = the rank's tiles 0 / 1
  const uint32_t* ab = S.abuf[aslot] + (g & 1) * 4 + t4;
  const uint4 b01 = make_uint4(ab[0], ab[8], ab[16], ab[24]);
  const uint4 b23 = make_uint4(ab[32], ab[40], ab[48], ab[56]);
  const int R = p.d / 64;
  // the unit's weight in the combine: 1 for the shared expert, else its gate
  // (published with the top-k before any routed stage was issued)
  if (t.src >= 0 && !mbar_wait_cluster(p, &S.topk_bar, static_cast<uint32_t>(rel) & 1u, W_DN_TOPK)) return false;
  const float wgt = t.src < 0 ? 1.f : S.gates[rel & 1][t.src];
  float* acc = S.dn_acc[quad];   // this quad's rows; the warp owns row tiles qw, qw + 4, ...
#pragma unroll 2
  for (int T = qw; T < R; T += kQW) {
    const uint8_t* blk = S.ring[slot] + static_cast<size_t>(T) * kGroupBytes;
    const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
    float c0[4], c1[4];
    mma_nib<true>(c0, q.x, b01.x, b01.y);
    mma_nib<true>(c1, q.y, b01.z, b01.w);
    mma_nib<false>(c0, q.z, b23.x, b23.y);
    mma_nib<false>(c1, q.w, b23.z, b23.w);
    const float s0 = half_lo(sbv.x), o0 = half_hi(sbv.x), s1 = half_lo(sbv.y), o1 = half_hi(sbv.y);
    const float y0 = s0 * ((c0[0] + c1[0]) + (c0[1] + c1[1])) + fmaf(-1024.f, s0, o0) * As;
    const float y1 = (s1 * 0.0625f) * ((c0[2] + c1[2]) + (c0[3] + c1[3])) + fmaf(-64.f, s1, o1) * As;
    if (t4 == 0) {
      acc[T * 16 + g] += wgt * y0;
      acc[T * 16 + g + 8] += wgt * y1;
    }
  }
  return true;
}

// End of layer rel: the CTA's rows (the quads' sums of their down stages,
// added in quad order: deterministic) onto the 2^-32 grid with this CTA's
// count in the low byte, and one bulk reduction into the layer's output
// vector (not waited for: readers poll the counts).
__device__ bool layer_end(const CParams& p, Smem& S, int cw, int rel, int& round, unsigned rank) {
  const int lane = threadIdx.x & 31;
  if (!mbar_wait_cluster(p, &S.topk_bar, static_cast<uint32_t>(rel) & 1u, W_END_TOPK)) {   // gates of this layer
    raise_abort(p);
    return false;
  }
  // the previous layer's bulk reduction must have read yq before it is rewritten
  if (cw == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  const unsigned long long te = p.timeline ? now_ns() : 0ull;
  if (!consumer_barrier(p, S, ++round)) return false;   // every down stage of the layer added in
  if (lane == 0 && p.timeline) acc(p, rel, 7, now_ns() - te);
  if (cw == 0 && lane == 0) {
    stamp(p, rel, EV_STAGES_DONE);
    mbarrier_arrive(&S.end_bar);
  }
  const int rows = p.d / kCl;
  bool bad = false;
  for (int i0 = 0; i0 < rows; i0 += kNC * 32) {
    const int i = i0 + cw * 32 + lane;
    if (i < rows) {
      float y = S.dn_acc[0][i];
#pragma unroll
      for (int q = 1; q < kNQ; ++q) y += S.dn_acc[q][i];
#pragma unroll
      for (int q = 0; q < kNQ; ++q) S.dn_acc[q][i] = 0.f;
      // |y| < 2^17 (v < 2^49 on the 2^-32 grid): with at most 64 clusters the
      // int64 sum of (v << 8) stays below 2^63 (the host checks the count)
      const bool ok = fabsf(y) < 131072.f;
      bad |= !ok;
      S.yq[i] = (ok ? (grid_from_float(y) << 8) : 0ll) + 1;   // + 1: this CTA's count
    }
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(p.err, ERR_Y_RANGE);
  fence_proxy_async_smem();   // yq is read by the bulk reduction (async proxy)
  if (!consumer_barrier(p, S, ++round)) return false;
  if (cw != 0) return true;
  // this CTA's zeroing of the next vector (fenced by the top-k warp) before its
  // reduction; the other CTAs zeroed this vector before adding their rows of
  // the previous one, which this CTA has read complete.  The whole warp waits
  // and decides together.
  if (!wait_warp(p, &S.zero_bar, static_cast<uint32_t>(rel) & 1u, W_ZERO)) {
    raise_abort(p);
    return false;
  }
  if (lane == 0) {
    fence_proxy_async_global();
    stamp(p, rel, EV_BULK_ISSUED);
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u64 [%0], [%1], %2;" ::"l"(
                     p.ybuf + static_cast<size_t>(rel % 3) * p.d + static_cast<size_t>(rank) * rows),
                 "r"(smem_u32(S.yq)), "r"(static_cast<uint32_t>(rows) * 8u)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    stamp(p, rel, EV_REDUCED);
  }
  __syncwarp();
  return true;
}

// After the last layer, cluster 0's four CTAs poll their quarters of the
// final vector: h_out = bf16(h + y), y_last, the last layer's debug y, and the
// last two vectors zeroed for the next launch (every CTA has added into the
// last one, so every CTA is done reading the one before it).
__device__ void finish(const CParams& p, Smem& S, int cw, int rel, unsigned rank) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x >= static_cast<unsigned>(kCl)) return;
  const DevCallArgs* A = &S.args;
  const int d = p.d, npair = d / 8;
  if (cw * 32 >= npair) return;
  const int j = cw * 32 + lane, e = static_cast<int>(rank) * (d / 4) + 2 * j;
  const bool valid = j < npair;
  long long* yv = p.ybuf + static_cast<size_t>(rel % 3) * d + e;
  float y0, y1;
  if (!poll_rows(p, yv, valid, y0, y1, W_FINISH) || !valid) return;
  const uint32_t hv = reinterpret_cast<const uint32_t*>(S.h)[e / 2];
  const float a = bf16_bits_to_float(static_cast<uint16_t>(hv & 0xFFFFu)) + y0;
  const float b = bf16_bits_to_float(static_cast<uint16_t>(hv >> 16)) + y1;
  reinterpret_cast<uint32_t*>(A->h_out)[e / 2] =
      static_cast<uint32_t>(float_to_bf16_bits(a)) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
  if (A->y_last) {
    A->y_last[e] = y0;
    A->y_last[e + 1] = y1;
  }
  if (A->dbg_y && rel < A->dbg_layers) {
    float* dy = A->dbg_y + (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * d + e;
    dy[0] = y0;
    dy[1] = y1;
  }
  *reinterpret_cast<longlong2*>(yv) = make_longlong2(0, 0);
  if (rel > 0)
    *reinterpret_cast<longlong2*>(p.ybuf + static_cast<size_t>((rel - 1) % 3) * d + e) = make_longlong2(0, 0);
}

template <bool kPool>
__device__ void consumer(const CParams& p, Smem& S, int cw, unsigned rank) {
  const int lane = threadIdx.x & 31;
  const int quad = cw / kQW, qw = cw % kQW;
  const int n_rel = p.l1 - p.l0;
  int round = 0;
  for (int rel = 0; rel < n_rel; ++rel) {
    // the logit bias of this CTA's expert, loaded now and used once the logit is formed
    float bias_v = 0.f;
    if (cw == 0 && S.args.bias && static_cast<int>(blockIdx.x) < p.E)
      bias_v = S.args.bias[(static_cast<size_t>(rel) * S.args.tok_total + S.args.tok_off) * p.E + blockIdx.x];
    if (!prep(p, S, cw, rel, round, rank, bias_v)) return;
    // stage u of the CTA goes to quad u mod 4
    int s = 0;
    for (int i = 0; i < S.n_tasks; ++i) {
      const CTask t = S.tasks[i];
      if (t.kind == K_TOPK) continue;
      const uint32_t u = static_cast<uint32_t>(rel) * S.n_stages + s++;
      if (static_cast<int>(u % kNQ) != quad) continue;
      const int slot = u % kNS;
      const unsigned long long t0 = p.timeline ? now_ns() : 0ull;
      if (!wait_warp(p, &S.full[slot], (u / kNS) & 1u, W_FULL)) {
        raise_abort(p);
        return;
      }
      const unsigned long long t1 = p.timeline ? now_ns() : 0ull;
      if (lane == 0) {
        stamp(p, rel, t.src < 0 ? EV_SHARED_DATA : EV_ROUTED_DATA);
        stamp(p, rel, EV_DATA_LAST, true);
        acc(p, rel, t.src < 0 ? 6 : 3, t1 - t0);
      }
      unsigned long long ta = t1;
      if (kPool && S.fill_src[slot]) fill_stage(p, S, slot, t, qw);
      if (t.kind == K_GU) {
        stage_gu(p, S, qw, rel, slot, t, rank);
      } else if (!stage_dn(p, S, quad, qw, rel, slot, t, &ta)) {
        raise_abort(p);
        return;
      }
      if (lane == 0 && p.timeline) {
        const unsigned long long t2 = now_ns();
        acc(p, rel, t.kind == K_GU ? 0 : 1, t2 - ta);
        acc(p, rel, t.kind == K_GU ? 4 : 5, 1);
        if (t.kind == K_DN) acc(p, rel, 2, ta - t1);
      }
      __syncwarp();
      if (lane == 0) mbarrier_arrive(&S.empty[slot]);
    }
    if (!layer_end(p, S, cw, rel, round, rank)) return;
  }
  finish(p, S, cw, n_rel - 1, rank);
}

// 18 warps put five on two of the SM's four schedulers; each scheduler has 16 K
// registers, so a thread may hold at most 96 (launch bounds give exactly that).
// The cluster shape is a property of the kernel (not only of the launch), so
// every launch path, a profiler's replay included, runs it in 4-CTA clusters.
template <bool kPool>
__global__ void __cluster_dims__(kCCluster, 1, 1) __launch_bounds__(kCThreads, 1) k_decode_cluster(CParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const unsigned rank = cluster_rank();
  // every distributed-shared-memory address below assumes clusters of kCl
  // CTAs covering the grid: anything else returns before touching a peer
  // (and the bulk and TMA copies into the ring need its 128-byte alignment,
  // the same in every CTA of the launch)
  if (cluster_size() != static_cast<unsigned>(kCl) || cluster_count() * kCl != gridDim.x ||
      (smem_u32(smem_raw) & 127u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, ERR_LAUNCH_SHAPE);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kQW);
    }
    for (int i = 0; i < 2 * kMaxU; ++i) mbar_init(&S.a_full[i], 1);
    mbar_init(&S.rrow_full, 1);
    mbar_init(&S.rrow_empty, 1);
    mbar_init(&S.topk_bar, 1);
    mbar_init(&S.zero_bar, 1);
    mbar_init(&S.end_bar, 1);
    for (int j = 0; j < 32; ++j) S.rank_word[j] = 0;
    mbar_init(&S.cbar, kNC);
    fence_mbar_init();
    S.args = *p.args;
    if (build_tasks(p, S, static_cast<int>(cluster_idx()), static_cast<int>(cluster_count())) > kMaxU)
      raise_abort(p);
  }
  if (threadIdx.x < kNS) S.gu_cnt[threadIdx.x] = 0;
  for (int i = threadIdx.x; i < kNQ * kMaxRows; i += blockDim.x) (&S.dn_acc[0][0])[i] = 0.f;
  __syncthreads();
  cluster_sync_all();   // every CTA's barriers exist before any remote arrival
  if (!aborted(p)) {
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) producer<kPool>(p, S, rank);
    } else if (warp <= kNC) {
      consumer<kPool>(p, S, warp - 1, rank);
    } else {
      topk_warp<kPool>(p, S);
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // this thread's bulk reductions are done
  __syncthreads();
  cluster_sync_all();   // no CTA leaves while a peer may still write into its shared memory
  // the last CTA out resets the exit counter and the abort flag (and, after an
  // abort, zeroes the output vectors, whose counts would otherwise be stale)
  if (threadIdx.x == 0) {
    __threadfence();
    S.last_out = atomicAdd(p.exit_cnt, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (S.last_out) {
    __threadfence();
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
  const cudaError_t e = cudaFuncSetAttribute((const void*)k_decode_cluster<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(Smem)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute((const void*)k_decode_cluster<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(Smem)));
}

// Clusters of kCCluster CTAs (one per SM) that can be resident at once.
cudaError_t cluster_max_active(int* n_clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCCluster);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  return cudaOccupancyMaxActiveClusters(n_clusters, (const void*)k_decode_cluster<false>, &cfg);
}

cudaError_t launch_cluster(CParams& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // two instances: the resident one carries none of the host-pool code
  return p.pool ? cudaLaunchKernelEx(&cfg, k_decode_cluster<true>, p)
                : cudaLaunchKernelEx(&cfg, k_decode_cluster<false>, p);
}

}  // namespace moe
