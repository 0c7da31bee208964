// Persistent decode kernel: one cooperative launch runs a B = 1 token through
// every layer of a resident context.
//
// The TurboFieldfare write-up's routed-MoE lesson (section "MoE needed
// parallel work, reuse, and coarse overlap": workgroups that stay resident and
// take rows until the dispatch is done) is taken to the whole decode step: one CTA
// per SM lives for the whole step, and the only things that serialise it are
// the data dependencies of the method itself (h_l -> router -> top-k ->
// routed gate/up -> down -> h_{l+1}).
//
// Per CTA:
//   warp 0, lane 0 (producer) walks the CTA's stage list and streams every
//     stage's weight bytes into a ring of five 25 KB shared-memory slots with
//     1-D bulk copies (TMA engine).  A stage is one gate/up tile (8 gate + 8 up
//     rows, all of d), four consecutive 16-row down tiles of one routed expert,
//     the 16-row down tile of the shared expert, or one router row; copies this
//     large keep the copy engine near the HBM rate, where 6 KB copies do not.
//     The producer needs the routing only for the routed experts' addresses;
//     while a layer routes it asks L2 to prefetch the next layer's router rows
//     and shared-expert tiles, which do not depend on routing.
//   warps 1..16 (consumers) split each stage into up to four 11-group chunks
//     taken round-robin: router rows (exact fixed-point logits, all consumer
//     warps together), gate/up chunks (int4 on mma.sync, GELU(gate)*up once a
//     tile's chunks are summed), and down chunks whose last finisher per row
//     tile does the fixed-order combine and the residual.
//   warp 17 (top-k) waits for a layer's logits, takes the top-k and the gates
//     and hands the experts to the producer through an mbarrier.  It is a warp
//     of its own because warp-wide shuffles measured several times slower in
//     the warp whose lane 0 issues the copies.
// Cross-CTA dependencies are monotone counters in global memory polled by one
// lane; every wait is bounded and gives up through an abort flag, and the last
// CTA to leave zeroes the counters for the next launch.  Each CTA computes the
// RMS norm and the top-k itself, so nothing is broadcast.
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

#include <climits>
#include <cstddef>

namespace moe {

namespace {

constexpr int kNC = kPConsumers;                  // consumer warps
constexpr int kNS = kPStages;                     // ring slots
constexpr int kSG = kPStageGroups;                // int4 groups per chunk
constexpr int kSub = 4;                           // chunks per slot
constexpr int kChunkBytes = kSG * kGroupBytes;    // 6336
constexpr int kSlotBytes = kSub * kChunkBytes;    // 25344
constexpr int kGuSlots = 16;                      // gate/up tiles in flight per CTA
constexpr int kMaxTasks = 64;                     // stages per CTA per layer

enum : int { T_PREP, T_R, T_GUS, T_TOPK, T_GUR, T_DNS, T_DNR };

// One entry of a CTA's stage pattern.  The pattern is the same for every layer
// and is built once per launch, so walking it costs a few shared loads per stage.
struct PTask {
  int16_t kind;
  int16_t a, b;          // R: expert; GUS: tile; GUR: j*(f/8)+tile; DNS: row tile; DNR: j, first row tile
  int16_t n_sub;         // chunks in the stage (0 for markers)
  int16_t owner0;        // consumer warp of chunk 0; chunk s goes to (owner0 + s) % kNC
  int16_t seq;           // gate/up tile number in the layer (from 1), or router row number (from 0)
  int32_t u;             // ring use of the stage within its layer
};

struct Smem {
  alignas(128) uint8_t ring[kNS][kSlotBytes];   // bulk-copy targets, read with 16-byte loads
  alignas(16) uint64_t full[kNS];
  alignas(16) uint64_t empty[kNS];
  alignas(16) uint16_t xs[kPMaxD];               // FFN input x of the current layer
  alignas(16) uint16_t xp[kPMaxD];               // x as mma B fragments
  alignas(16) float xg[kPMaxD / 64];             // per-group sums of x
  alignas(16) uint8_t abuf[kNC][kSG * 256];      // per-warp down B fragments (hi/lo), cp.async targets
  alignas(16) float asb[kNC][kSG * 16];          // per-warp tile sums for the bias term, cp.async targets
  alignas(16) float asg[kNC][kSG];
  alignas(16) float gu_part[kGuSlots][kSub][8][2];  // gate/up chunk partials [slot][chunk][row][gate/up]
  alignas(16) long long rlog[2][kNC];            // router-row partials per consumer warp (two rows in flight)
  alignas(16) DevCallArgs args;                  // per-call pointers, copied once per launch
  PTask tasks[kMaxTasks];
  int n_tasks, stages_per_layer, tiles_per_layer, rows_per_layer;
  float red[kNC];
  int gu_cnt[kGuSlots];
  int32_t ids[2][32];
  float gates[2][32];
  alignas(8) uint64_t cbar;                     // consumer-warp barrier (one arrival per consumer warp)
  alignas(8) uint64_t topk_bar;                 // one phase per layer: the top-k warp has published ids
};

static_assert(offsetof(Smem, ring) % 128 == 0, "ring must be 128-byte aligned");
static_assert(kSlotBytes % 128 == 0 && kChunkBytes % 16 == 0, "slots keep 16-byte alignment");
static_assert(offsetof(Smem, full) % 8 == 0 && offsetof(Smem, empty) % 8 == 0, "mbarriers need 8 bytes");
static_assert(offsetof(Smem, xs) % 16 == 0 && offsetof(Smem, xp) % 16 == 0, "x read as uint4");
static_assert(offsetof(Smem, abuf) % 16 == 0 && (kSG * 256) % 16 == 0, "abuf: cp.async 16-byte targets");
static_assert(offsetof(Smem, asb) % 16 == 0 && (kSG * 16 * 4) % 16 == 0, "asb: cp.async 16-byte targets");
static_assert(offsetof(Smem, rlog) % 8 == 0, "int64 partials");

// ------------------------------------------------------------------ timeline (optional)

// Event times (%globaltimer, ns) of the step, min or max over CTAs, row l of
// the caller's timeline buffer; CTA 0's accumulated wait/compute times at row
// (n_layers + l): [0] gate/up slot wait, [1] gate/up compute, [2] gate/up
// chunks, [3] down dependency + operand wait, [5] down slot wait, [6] down
// compute, [7] down chunks.
enum : int { EV_PREP_IN, EV_H_READY, EV_PREP_DONE, EV_LOGIT, EV_LOGITS_ALL, EV_TOPK, EV_GUR_ISSUE0,
             EV_DNR_ISSUED, EV_GUR_START, EV_GUR_DONE, EV_DNR_READY, EV_DNR_DONE, EV_COMBINE, EV_GUS_DONE,
             EV_DNS_DONE, EV_START };

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tl_max(const PParams& p, int l, int ev) {
  if (p.timeline) atomicMax(p.timeline + l * 16 + ev, gtimer());
}
__device__ __forceinline__ void tl_min(const PParams& p, int l, int ev) {
  if (p.timeline) atomicMin(p.timeline + l * 16 + ev, gtimer());
}
__device__ __forceinline__ void acc_add(const PParams& p, int l, int slot, unsigned long long v) {
  if (p.timeline && blockIdx.x == 0) atomicAdd(p.timeline + (p.n_layers_tl + l) * 16 + slot, v);
}
// Per-CTA stamps of the step's third layer (the last one if fewer) at row
// 2 * n_layers + blockIdx.x: cta_stamp keeps the first time, cta_stamp_max the last.
__device__ __forceinline__ bool stamped_layer(const PParams& p, int rel) {
  const int n_rel = p.l1 - p.l0;
  return p.timeline && rel == (n_rel > 2 ? 2 : n_rel - 1);
}
__device__ __forceinline__ void cta_stamp(const PParams& p, int rel, int k) {
  if (!stamped_layer(p, rel)) return;
  atomicCAS(p.timeline + (2 * p.n_layers_tl + blockIdx.x) * 16 + k, 0ull, gtimer());
}
__device__ __forceinline__ void cta_stamp_max(const PParams& p, int rel, int k) {
  if (!stamped_layer(p, rel)) return;
  atomicMax(p.timeline + (2 * p.n_layers_tl + blockIdx.x) * 16 + k, gtimer());
}

// ------------------------------------------------------------------ sync helpers

__device__ __forceinline__ int pos_mod(int a, int m) {
  const int r = a % m;
  return r < 0 ? r + m : r;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ bool aborted(const PParams& p) {
  return *reinterpret_cast<volatile unsigned*>(p.abort_flag) != 0;
}

__device__ __forceinline__ void raise_abort(const PParams& p) {
  atomicOr(p.err, ERR_WAIT_TIMEOUT);
  atomicExch(p.abort_flag, 1u);
}

// Bounded wait on a phase of a local mbarrier (this CTA's threads or copies)
// by a whole warp: the lanes decide together (a vote per poll), so a warp never
// splits between going on and giving up.  False after p.spin_limit cycles or
// once another CTA has aborted.
__device__ bool wait_warp(const PParams& p, uint64_t* bar, uint32_t parity) {
  if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(0xFFFFFFFFu, clock64() - t0 > p.spin_limit || ((it & 15) == 0 && aborted(p)))) {
      if ((threadIdx.x & 31) == 0) atomicOr(p.err, ERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// The same wait by a single thread (the producer).
__device__ bool wait_one(const PParams& p, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > p.spin_limit || ((it & 15) == 0 && aborted(p))) {
      atomicOr(p.err, ERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// The whole warp waits until *ctr >= target (acquire).  False on abort or
// timeout.  Every lane polls (the loads of one instruction hit one address, so
// this costs one request): a loop run by one lane while the others wait leaves
// the warp diverged, and every later warp-wide instruction (shuffle, vote,
// mma.sync) then measured about six times slower until the warp reconverged.
__device__ bool warp_wait_counter(const PParams& p, const unsigned* ctr, unsigned target) {
  if (__all_sync(0xFFFFFFFFu, ld_acquire(ctr) >= target)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    __nanosleep(64);
    if (__all_sync(0xFFFFFFFFu, ld_acquire(ctr) >= target)) return true;
    if ((it & 255) == 0) {
      if (__any_sync(0xFFFFFFFFu, aborted(p))) return false;
      if (__any_sync(0xFFFFFFFFu, clock64() - t0 > p.spin_limit)) {
        if ((threadIdx.x & 31) == 0) raise_abort(p);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Consumer-warp barrier: an mbarrier with one arrival per consumer warp per
// round; waiting warps sleep in try_wait.  Round r (from 1) completes phase
// r - 1.  False on timeout or abort (bounded wait).
__device__ bool consumer_barrier(const PParams& p, Smem& S, int round) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbarrier_arrive(&S.cbar);
  const bool ok = wait_warp(p, &S.cbar, static_cast<uint32_t>(round - 1) & 1u);
  if (!ok) raise_abort(p);
  __syncwarp();
  return ok;
}

// ------------------------------------------------------------------ stage list

__device__ __forceinline__ int gu_chunks(const PParams& p) { return (p.d / 64 + kSG - 1) / kSG; }

// The CTA's stages for one layer (identical for the producer and the consumers).
template <class F>
__device__ void for_each_stage(const PParams& p, int c, int G, F&& visit) {
  const int nT = p.d / 16, nT4 = (nT + kSub - 1) / kSub;
  const int gu_st = gu_chunks(p);
  const int n_gus = p.fs / 8, n_gur = p.k * (p.f / 8), n_dns = nT, n_dnr = p.k * nT4;
  int base = 0;
  visit(T_PREP, 0, 0, 0);
  for (int i = pos_mod(c - base, G); i < p.E; i += G) visit(T_R, i, 0, 1);
  base = (base + p.E) % G;
  for (int i = pos_mod(c - base, G); i < n_gus; i += G) visit(T_GUS, i, 0, gu_st);
  base = (base + n_gus) % G;
  visit(T_TOPK, 0, 0, 0);
  for (int i = pos_mod(c - base, G); i < n_gur; i += G) visit(T_GUR, i, 0, gu_st);
  base = (base + n_gur) % G;
  for (int i = pos_mod(c - base, G); i < n_dns; i += G) visit(T_DNS, i, 0, p.n_sc);
  base = (base + n_dns) % G;
  for (int i = pos_mod(c - base, G); i < n_dnr; i += G) {
    const int j = i / nT4, T0 = (i % nT4) * kSub;
    visit(T_DNR, j, T0, min(kSub, nT - T0));
  }
}

struct StageSrc {
  const uint8_t* src;
  uint32_t bytes;
};

// Global source of a stage (producer side); L = the stage's layer.
__device__ StageSrc stage_src(const PParams& p, const PLayer& L, const PTask& e, const int32_t* ids) {
  const int nGd = p.d / 64, nGf = p.f / 64, nGs = p.fs / 64;
  const size_t gu_tile = static_cast<size_t>(nGd) * kGroupBytes;
  StageSrc r;
  switch (e.kind) {
    case T_R:
      r.src = reinterpret_cast<const uint8_t*>(L.router_w + static_cast<size_t>(e.a) * p.d);
      r.bytes = p.d * 2;
      break;
    case T_GUS:
      r.src = L.shared + e.a * gu_tile;
      r.bytes = static_cast<uint32_t>(gu_tile);
      break;
    case T_GUR: {
      const int j = e.a / (p.f / 8), tile = e.a % (p.f / 8);
      r.src = L.experts + static_cast<long long>(ids[j]) * p.expert_stride + tile * gu_tile;
      r.bytes = static_cast<uint32_t>(gu_tile);
      break;
    }
    case T_DNS: {
      const size_t gu_s = static_cast<size_t>(p.fs / 8) * gu_tile;
      r.src = L.shared + gu_s + static_cast<size_t>(e.a) * nGs * kGroupBytes;
      r.bytes = nGs * kGroupBytes;
      break;
    }
    default: {  // T_DNR
      const size_t gu_r = static_cast<size_t>(p.f / 8) * gu_tile;
      r.src = L.experts + static_cast<long long>(ids[e.a]) * p.expert_stride + gu_r +
              static_cast<size_t>(e.b) * nGf * kGroupBytes;
      r.bytes = e.n_sub * nGf * kGroupBytes;
      break;
    }
  }
  return r;
}

// ------------------------------------------------------------------ top-k

// Top-k (ties to the lower index) and softmax gates over layer l's logits, one
// warp.  Each lane holds up to 8 logits sorted by (value desc, index asc); a
// round picks the warp-wide best head with three warp reductions on the
// order-preserving unsigned image of the int64 logit and on the index.
__device__ void warp_topk(const PParams& p, int l, int32_t* ids, float* gates) {
  const int lane = threadIdx.x & 31;
  const long long* lg = p.logits + static_cast<size_t>(l) * p.E;
  unsigned long long key[8];
  int idx[8];
  int n = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0ull;
    idx[i] = 0x7fffffff;
    if (e < p.E) {
      key[i] = static_cast<unsigned long long>(__ldcg(&lg[e])) ^ 0x8000000000000000ull;
      idx[i] = e;
      ++n;
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
  int head = 0;
  int my_id = 0;
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
    const unsigned mh = __reduce_max_sync(0xFFFFFFFFu, hi);
    const bool c1 = has && hi == mh;
    const unsigned ml = __reduce_max_sync(0xFFFFFFFFu, c1 ? lo : 0u);
    const bool c2 = c1 && lo == ml;
    const unsigned me = __reduce_min_sync(0xFFFFFFFFu, c2 ? static_cast<unsigned>(he) : 0xFFFFFFFFu);
    if (c2 && static_cast<unsigned>(he) == me) ++head;
    if (lane == j) {
      my_id = static_cast<int>(me);
      my_v = static_cast<long long>((static_cast<unsigned long long>(mh) << 32 | ml) ^ 0x8000000000000000ull);
    }
  }
  const long long top = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  float ex = 0.f;
  if (lane < p.k) ex = expf(__ll2float_rn(my_v - top) * 9.094947017729282e-13f);
  float sum = 0.f;
  for (int j = 0; j < p.k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
  if (lane < p.k) {
    ids[lane] = my_id;
    gates[lane] = ex / sum;
  }
  __syncwarp();
}

__device__ __forceinline__ float gelu_p(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

__device__ __forceinline__ int afrag_index(int r, int par) {
  const int G = r >> 6, st = (r >> 4) & 3, w = r & 15;
  const int t4 = (w & 7) >> 1, pos = ((w >> 3) << 1) | (w & 1);
  return ((((G * 2 + par) * 4 + t4) * 4 + st) << 2) + pos;
}

// ------------------------------------------------------------------ producer

// One thread (lane 0 of warp 0) issues every stage.  At a layer's top-k marker
// it asks L2 for the next layer's routing-independent bytes, then waits for the
// top-k warp to publish the layer's experts.
__device__ void producer(const PParams& p, Smem& S) {
  const int n_rel = p.l1 - p.l0;
  const int n_tasks = S.n_tasks, spl = S.stages_per_layer;
  uint32_t u_issued = 0;   // ring uses issued so far
  for (int rel = 0; rel < n_rel; ++rel) {
    const int l = p.l0 + rel;
    const PLayer Lc = p.layers[l];
    for (int i = 0; i < n_tasks; ++i) {
      const PTask e = S.tasks[i];
      if (e.kind == T_PREP) continue;
      if (e.kind == T_TOPK) {
        cta_stamp(p, rel, 0);
        if (rel + 1 < n_rel) {
          const PLayer Ln = p.layers[l + 1];
          for (int i2 = 0; i2 < n_tasks; ++i2) {
            const PTask e2 = S.tasks[i2];
            if (e2.kind == T_R || e2.kind == T_GUS || e2.kind == T_DNS) {
              const StageSrc ss = stage_src(p, Ln, e2, nullptr);
              prefetch_l2(ss.src, ss.bytes);
            }
          }
        }
        if (!wait_one(p, &S.topk_bar, static_cast<uint32_t>(rel) & 1u)) {
          raise_abort(p);
          break;
        }
        continue;
      }
      const uint32_t u = static_cast<uint32_t>(rel) * spl + e.u;
      const int slot = u % kNS;
      if (!wait_one(p, &S.empty[slot], ((u / kNS) & 1) ^ 1)) {
        raise_abort(p);
        break;
      }
      const StageSrc ss = stage_src(p, Lc, e, S.ids[rel & 1]);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&S.full[slot], ss.bytes);
      bulk_g2s(S.ring[slot], ss.src, ss.bytes, &S.full[slot]);
      u_issued = u + 1;
      if (p.timeline) {
        if (e.kind == T_GUR) tl_max(p, l, EV_GUR_ISSUE0);
        if (e.kind == T_DNR) tl_max(p, l, EV_DNR_ISSUED);
        if (e.kind == T_GUR) cta_stamp(p, rel, 4);
        if (e.kind == T_DNR) cta_stamp(p, rel, 5);
      }
    }
    if (aborted(p)) break;
  }
  // on abort, the last min(u_issued, kNS) stages may still be in flight: wait for each, bounded
  if (aborted(p))
    for (uint32_t v = (u_issued > static_cast<uint32_t>(kNS) ? u_issued - kNS : 0); v < u_issued; ++v)
      mbar_wait_bounded(&S.full[v % kNS], (v / kNS) & 1, p.err);
}

// The top-k warp: per layer, waits for every router row, takes the top-k and
// the gates, publishes them (shared memory for the producer, global memory for
// the combine) and releases the producer.
__device__ void topk_warp(const PParams& p, Smem& S) {
  const int lane = threadIdx.x & 31;
  const int n_rel = p.l1 - p.l0;
  for (int rel = 0; rel < n_rel; ++rel) {
    const int l = p.l0 + rel;
    if (!warp_wait_counter(p, p.logit_cnt + l, static_cast<unsigned>(p.E))) return;
    if (lane == 0) {
      tl_max(p, l, EV_LOGITS_ALL);
      cta_stamp(p, rel, 2);
    }
    int32_t* sid = S.ids[rel & 1];
    float* sg = S.gates[rel & 1];
    warp_topk(p, l, sid, sg);
    if (lane < p.k) p.gates_g[static_cast<size_t>(l) * p.k + lane] = sg[lane];
    if (blockIdx.x == 0 && lane < p.k && rel < S.args.dbg_layers) {
      const DevCallArgs* A = &S.args;
      const size_t o = (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.k + lane;
      if (A->dbg_ids) A->dbg_ids[o] = sid[lane];
      if (A->dbg_gates) A->dbg_gates[o] = sg[lane];
    }
    __syncwarp();
    if (lane == 0) {
      tl_max(p, l, EV_TOPK);
      cta_stamp(p, rel, 3);
      mbarrier_arrive(&S.topk_bar);
    }
  }
}

// ------------------------------------------------------------------ consumers

// Layer input: wait for the previous layer's output (one thread per CTA), RMS
// norm in a fixed order (every CTA gets the same x), x as plain bf16, as mma B
// fragments and as per-group sums.
__device__ bool prep(const PParams& p, Smem& S, int cw, int rel, int& round) {
  const int lane = threadIdx.x & 31;
  const int d = p.d, nGd = d / 64;
  const DevCallArgs* A = &S.args;
  const int l = p.l0 + rel;
  if (lane == 0) tl_min(p, l, EV_PREP_IN);
  if (lane == 0 && cw == 0) cta_stamp(p, rel, 8);
  if (rel > 0) {
    if (cw == 0 && !warp_wait_counter(p, p.rows_done + (l - 1), static_cast<unsigned>(d / 16))) return false;
    if (!consumer_barrier(p, S, ++round)) return false;
  }
  if (lane == 0) tl_max(p, l, EV_H_READY);
  if (lane == 0 && cw == 0) cta_stamp(p, rel, 9);
  const uint16_t* h = rel == 0 ? A->h_in : ((rel - 1) & 1 ? p.hbuf1 : p.hbuf0);
  // this warp's groups G = cw, cw + kNC, ...; lane holds elements 64G + 2*lane, +1
  uint32_t hv[(kPMaxD / 64 + kNC - 1) / kNC];
  float ss = 0.f;
  int ng = 0;
  for (int G = cw; G < nGd; G += kNC, ++ng) {
    hv[ng] = __ldcg(reinterpret_cast<const unsigned*>(h + 64 * G) + lane);
    const float a = bf16_bits_to_float(static_cast<uint16_t>(hv[ng] & 0xFFFFu));
    const float b = bf16_bits_to_float(static_cast<uint16_t>(hv[ng] >> 16));
    ss += a * a;
    ss += b * b;
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
  if (lane == 0) S.red[cw] = ss;
  if (!consumer_barrier(p, S, ++round)) return false;  // all earlier work done, red[] complete
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
    for (int m = 16; m; m >>= 1) gs += __shfl_xor_sync(0xFFFFFFFFu, gs, m);
    if (lane == 0) S.xg[G] = gs;
    if (blockIdx.x == 0 && A->dbg_x && rel < A->dbg_layers)
      reinterpret_cast<uint32_t*>(A->dbg_x + (static_cast<size_t>(rel) * A->tok_total + A->tok_off) * d)[32 * G + lane] = xv;
  }
  const bool okb = consumer_barrier(p, S, ++round);  // x complete
  if (lane == 0) tl_max(p, l, EV_PREP_DONE);
  if (lane == 0 && cw == 0) cta_stamp(p, rel, 10);
  return okb;
}

// Router row e of layer l, computed by all consumer warps together (the row is
// a short dot product on the critical path): warp cw takes 8-element chunks
// cw*32 + lane, cw*32 + lane + 512, ...; the int64 partials are summed in warp
// order (the sum is exact, so the order does not change it).
__device__ bool task_router(const PParams& p, Smem& S, int rel, int l, int e_row, const uint8_t* stage, int cw,
                            int& round, int buf) {
  const int lane = threadIdx.x & 31;
  const uint4* wr = reinterpret_cast<const uint4*>(stage);
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
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(p.err, ERR_ROUTER_DOMAIN);
  if (lane == 0) S.rlog[buf][cw] = acc;
  if (!consumer_barrier(p, S, ++round)) return false;
  if (cw != 0) return true;
  acc = 0;
  for (int w = 0; w < kNC; ++w) acc += S.rlog[buf][w];
  if (lane == 0) {
    const DevCallArgs* A = &S.args;
    if (A->bias) {
      const float bv = A->bias[(static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.E + e_row];
      if (!(fabsf(bv) < 1048576.f)) atomicOr(p.err, ERR_ROUTER_DOMAIN);
      else acc += __float2ll_rn(bv * 1099511627776.0f);
    }
    p.logits[static_cast<size_t>(l) * p.E + e_row] = acc;
    if (A->dbg_logits && rel < A->dbg_layers)
      A->dbg_logits[(static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.E + e_row] = acc;
    red_add_release(p.logit_cnt + l, 1u);
    tl_max(p, l, EV_LOGIT);
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

// Epilogue of a gate/up tile: a = GELU(gate) * up for its 8 rows, as bf16 hi + lo
// B fragments of the down projection, plus the tile's hi / lo sums.
__device__ void gu_epilogue(const PParams& p, int src, int tile, float ga, float ua, int l) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const bool routed = src >= 0;
  uint16_t* ab = routed ? p.a_r + static_cast<size_t>(src) * 2 * p.f : p.a_s;
  float* sb = routed ? p.asum_r + static_cast<size_t>(src) * (p.f / 8) * 2 : p.asum_s;
  const float av = gelu_p(ga, p.gelu) * ua;
  const uint16_t hi = float_to_bf16_bits(av);
  const uint16_t lo = float_to_bf16_bits(av - bf16_bits_to_float(hi));
  const int r = tile * 8 + g;
  if (t4 == 0) {
    ab[afrag_index(r, 0)] = hi;
    ab[afrag_index(r, 1)] = lo;
  }
  float sh = bf16_bits_to_float(hi), sl = bf16_bits_to_float(lo);
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    sh += __shfl_xor_sync(0xFFFFFFFFu, sh, m);
    sl += __shfl_xor_sync(0xFFFFFFFFu, sl, m);
  }
  if (lane == 0) {
    sb[tile * 2] = sh;
    sb[tile * 2 + 1] = sl;
  }
  fence_acq_rel_gpu();
  __syncwarp();
  if (lane == 0) {
    const int ctr = routed ? p.n_sc + src : (tile * 8 / 64) / kSG;
    red_add_release(p.gu_cnt + static_cast<size_t>(l) * (p.n_sc + p.k) + ctr, 1u);
    tl_max(p, l, routed ? EV_GUR_DONE : EV_GUS_DONE);
  }
}

// Gate/up chunk s of tile (src, tile).  The last chunk of a tile to finish sums
// the chunk partials in chunk order and runs the epilogue.
__device__ void task_gu(const PParams& p, Smem& S, int l, const uint8_t* slot, int s, int src, int tile, int gslot) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nGd = p.d / 64, n_ch = gu_chunks(p);
  const int g0 = s * kSG, ng = min(kSG, nGd - g0);
  float ga = 0.f, ua = 0.f;
  gu_chunk(S, slot + s * kChunkBytes, g0, ng, ga, ua);
  if (n_ch == 1) {
    gu_epilogue(p, src, tile, ga, ua, l);
    return;
  }
  if (t4 == 0) {
    S.gu_part[gslot][s][g][0] = ga;
    S.gu_part[gslot][s][g][1] = ua;
  }
  __threadfence_block();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&S.gu_cnt[gslot], 1) == n_ch - 1;
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;
  __threadfence_block();
  ga = 0.f;
  ua = 0.f;
  for (int ch = 0; ch < n_ch; ++ch) {
    ga += reinterpret_cast<volatile float*>(S.gu_part[gslot][ch][g])[0];
    ua += reinterpret_cast<volatile float*>(S.gu_part[gslot][ch][g])[1];
  }
  if (lane == 0) S.gu_cnt[gslot] = 0;
  gu_epilogue(p, src, tile, ga, ua, l);
}

// Waits for the source's gate/up results and stages their B fragments and
// group sums in this warp's buffers.  ctr: gate/up counter; target: tiles.
__device__ bool dn_operands(const PParams& p, Smem& S, int cw, int l, bool routed, int src, int g0, int ng,
                            int ctr, unsigned target) {
  const int lane = threadIdx.x & 31;
  if (!warp_wait_counter(p, p.gu_cnt + static_cast<size_t>(l) * (p.n_sc + p.k) + ctr, target)) return false;
  const uint16_t* abase = routed ? p.a_r + static_cast<size_t>(src) * 2 * p.f : p.a_s;
  const float* sbase = routed ? p.asum_r + static_cast<size_t>(src) * (p.f / 8) * 2 : p.asum_s;
  const uint8_t* asrc = reinterpret_cast<const uint8_t*>(abase) + static_cast<size_t>(g0) * 256;
  // uniform loops with predicated bodies keep the warp converged (see warp_wait_counter)
  for (int i0 = 0; i0 < ng * 16; i0 += 32)
    if (i0 + lane < ng * 16) cp_async16(S.abuf[cw] + (i0 + lane) * 16, asrc + (i0 + lane) * 16);
  const uint8_t* ssrc = reinterpret_cast<const uint8_t*>(sbase + static_cast<size_t>(g0) * 16);
  for (int i0 = 0; i0 < ng * 4; i0 += 32)
    if (i0 + lane < ng * 4)
      cp_async16(reinterpret_cast<uint8_t*>(S.asb[cw]) + (i0 + lane) * 16, ssrc + (i0 + lane) * 16);
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  __syncwarp();
  {
    const int gl = min(lane, ng - 1);
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a += S.asb[cw][gl * 16 + 2 * i] + S.asb[cw][gl * 16 + 2 * i + 1];
    if (lane < ng) S.asg[cw][lane] = a;
  }
  __syncwarp();
  return true;
}

// Down chunk: rows 16T..16T+15, ng groups of the source, weights at `w`.
// Writes the partial into part slot ctr; the last part of the row tile combines.
__device__ void dn_chunk(const PParams& p, Smem& S, int cw, int rel, int l, int T, int ctr, const uint8_t* w,
                         int ng) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  float y0 = 0.f, y1 = 0.f;
  for (int i = 0; i < ng; ++i) {
    const uint8_t* blk = w + i * kGroupBytes;
    const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
    const uint4* bf = reinterpret_cast<const uint4*>(S.abuf[cw] + i * 256 + ((g & 1) * 4 + t4) * 32);
    const uint4 b01 = bf[0], b23 = bf[1];
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
    const float As = S.asg[cw][i];
    const float s0 = half_lo(sbv.x), b0 = half_hi(sbv.x), s1 = half_lo(sbv.y), b1 = half_hi(sbv.y);
    y0 += s0 * ((c0[0] + c1[0]) + (c0[1] + c1[1])) + fmaf(-128.f, s0, b0) * As;
    y1 += s1 * ((c0[2] + c1[2]) + (c0[3] + c1[3])) + fmaf(-128.f, s1, b1) * As;
  }
  const int n_parts = p.n_sc + p.k;
  float* part = p.part + (static_cast<size_t>(rel & 1) * n_parts + ctr) * p.d;
  if (t4 == 0) {
    part[T * 16 + g] = y0;
    part[T * 16 + g + 8] = y1;
  }
  fence_acq_rel_gpu();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    tl_max(p, l, ctr >= p.n_sc ? EV_DNR_DONE : EV_DNS_DONE);
    last = atom_add_acq_rel(p.row_cnt + static_cast<size_t>(l) * (p.d / 16) + T, 1u) ==
           static_cast<unsigned>(n_parts - 1);
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;
  fence_acq_rel_gpu();
  // combine row tile T in fixed order: shared chunks, then top-k positions 0..k-1.
  // The gates were published by the CTAs that issued routed work, before it existed.
  const float* gates = p.gates_g + static_cast<size_t>(l) * p.k;
  const DevCallArgs* A = &S.args;
  const int n_rel = p.l1 - p.l0;
  const bool last_layer = rel == n_rel - 1;
  const uint16_t* hin = rel == 0 ? A->h_in : ((rel - 1) & 1 ? p.hbuf1 : p.hbuf0);
  uint16_t* hout = last_layer ? A->h_out : (rel & 1 ? p.hbuf1 : p.hbuf0);
  const float* pp = p.part + static_cast<size_t>(rel & 1) * n_parts * p.d;
  {
    // all 32 lanes run the sums (lanes 16..31 repeat rows 0..15) so the warp stays converged
    const int row = T * 16 + (lane & 15);
    float y = 0.f;
    for (int c2 = 0; c2 < p.n_sc; ++c2) y += __ldcg(&pp[static_cast<size_t>(c2) * p.d + row]);
    for (int j = 0; j < p.k; ++j) y += __ldcg(&gates[j]) * __ldcg(&pp[static_cast<size_t>(p.n_sc + j) * p.d + row]);
    const float hv = bf16_bits_to_float(__ldcg(&hin[row]));
    if (lane < 16) {
      hout[row] = float_to_bf16_bits(hv + y);
      if (last_layer && A->y_last) A->y_last[row] = y;
      if (A->dbg_y && rel < A->dbg_layers) A->dbg_y[(static_cast<size_t>(rel) * A->tok_total + A->tok_off) * p.d + row] = y;
    }
  }
  fence_acq_rel_gpu();
  __syncwarp();
  if (lane == 0) {
    red_add_release(p.rows_done + l, 1u);
    tl_max(p, l, EV_COMBINE);
  }
}

__device__ void consumer(const PParams& p, Smem& S, int cw) {
  const int lane = threadIdx.x & 31;
  const int n_rel = p.l1 - p.l0;
  const int n_tasks = S.n_tasks, spl = S.stages_per_layer;
  const int tpl = S.tiles_per_layer, rpl = S.rows_per_layer;
  const int nGf = p.f / 64, nGs = p.fs / 64;
  int round = 0;
  for (int rel = 0; rel < n_rel; ++rel) {
    const int l = p.l0 + rel;
    for (int i = 0; i < n_tasks; ++i) {
      const PTask e = S.tasks[i];
      if (e.kind == T_TOPK) continue;
      if (e.kind == T_PREP) {
        if (!prep(p, S, cw, rel, round)) return;
        continue;
      }
      const uint32_t u = static_cast<uint32_t>(rel) * spl + e.u;
      const int slot = u % kNS;
      const uint32_t par = (u / kNS) & 1;
      if (e.kind == T_R) {
        if (!wait_warp(p, &S.full[slot], par)) {
          raise_abort(p);
          return;
        }
        if (!task_router(p, S, rel, l, e.a, S.ring[slot], cw, round, (rel * rpl + e.seq) & 1)) return;
        if (lane == 0 && cw == 0) cta_stamp(p, rel, 11);
        // every warp has read the row once the reduction barrier passed; warp 0 frees the slot
        if (cw == 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive_n(&S.empty[slot], kSub);
        }
        continue;
      }
      int s = cw - e.owner0;
      if (s < 0) s += kNC;
      if (s >= e.n_sub) continue;  // not this warp's chunk
      const unsigned long long t0 = p.timeline ? gtimer() : 0ull;
      bool ok = true;
      if (e.kind == T_GUS || e.kind == T_GUR) {
        if (!wait_warp(p, &S.full[slot], par)) {
          raise_abort(p);
          return;
        }
        const unsigned long long t1 = p.timeline ? gtimer() : 0ull;
        if (e.kind == T_GUR && lane == 0) tl_min(p, l, EV_GUR_START);
        if (e.kind == T_GUR && lane == 0) cta_stamp(p, rel, 12);
        if (e.kind == T_GUR && lane == 0) cta_stamp_max(p, rel, 1);
        if (e.kind == T_GUS && lane == 0) cta_stamp(p, rel, 6);
        const int gslot = (rel * tpl + e.seq) % kGuSlots;
        if (e.kind == T_GUS) task_gu(p, S, l, S.ring[slot], s, -1, e.a, gslot);
        else task_gu(p, S, l, S.ring[slot], s, e.a / (p.f / 8), e.a % (p.f / 8), gslot);
        if (lane == 0) cta_stamp_max(p, rel, e.kind == T_GUR ? 7 : 13);
        if (lane == 0 && e.kind == T_GUR && p.timeline) {
          acc_add(p, l, 0, t1 - t0);
          acc_add(p, l, 1, gtimer() - t1);
          acc_add(p, l, 2, 1);
        }
      } else if (e.kind == T_DNS) {
        // chunk s of the shared down row tile e.a: groups [11 s, 11 s + ng)
        const int g0 = s * kSG, ng = min(kSG, nGs - g0);
        const unsigned target = min(kSG * 8, p.fs / 8 - s * kSG * 8);
        ok = dn_operands(p, S, cw, l, false, -1, g0, ng, s, target);
        if (ok) ok = wait_warp(p, &S.full[slot], par);
        if (ok) dn_chunk(p, S, cw, rel, l, e.a, s, S.ring[slot] + s * kChunkBytes, ng);
      } else {  // T_DNR: row tile e.b + s of routed position j = e.a
        ok = dn_operands(p, S, cw, l, true, e.a, 0, nGf, p.n_sc + e.a, p.f / 8);
        if (lane == 0 && ok) tl_max(p, l, EV_DNR_READY);
        const unsigned long long t2 = p.timeline ? gtimer() : 0ull;
        if (ok) ok = wait_warp(p, &S.full[slot], par);
        const unsigned long long t3 = p.timeline ? gtimer() : 0ull;
        if (lane == 0 && ok) cta_stamp(p, rel, 14);
        if (ok) dn_chunk(p, S, cw, rel, l, e.b + s, p.n_sc + e.a, S.ring[slot] + s * nGf * kGroupBytes, nGf);
        if (lane == 0 && p.timeline) {
          acc_add(p, l, 3, t2 - t0);
          acc_add(p, l, 5, t3 - t2);
          acc_add(p, l, 6, gtimer() - t3);
          acc_add(p, l, 7, 1);
        }
      }
      if (!ok) {
        raise_abort(p);
        return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&S.empty[slot], s == 0 ? 1 + kSub - e.n_sub : 1);
    }
    if (lane == 0) cta_stamp_max(p, rel, 15);
  }
}

// 18 warps put five on two of the SM's four schedulers; each scheduler has 16 K
// registers, so a thread may hold at most 96 (launch bounds give exactly that).
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(PParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kSub);
    }
    mbar_init(&S.cbar, kNC);
    mbar_init(&S.topk_bar, 1);
    fence_mbar_init();
    S.args = *p.args;
    // this CTA's stage pattern for one layer
    int n = 0, u = 0, seq = 0, tiles = 0, rows = 0;
    for_each_stage(p, blockIdx.x, gridDim.x, [&](int kind, int a, int b, int n_sub) {
      PTask e;
      e.kind = static_cast<int16_t>(kind);
      e.a = static_cast<int16_t>(a);
      e.b = static_cast<int16_t>(b);
      e.n_sub = static_cast<int16_t>(n_sub);
      e.owner0 = static_cast<int16_t>(seq % kNC);
      e.seq = 0;
      e.u = u;
      if (kind == T_GUS || kind == T_GUR) e.seq = static_cast<int16_t>(++tiles);
      if (kind == T_R) e.seq = static_cast<int16_t>(rows++);
      if (kind != T_PREP && kind != T_TOPK) ++u;
      if (kind == T_GUS || kind == T_GUR || kind == T_DNS || kind == T_DNR) seq += n_sub;
      if (n < kMaxTasks) S.tasks[n] = e;
      ++n;
    });
    S.n_tasks = n < kMaxTasks ? n : kMaxTasks;
    S.stages_per_layer = u;
    S.tiles_per_layer = tiles;
    S.rows_per_layer = rows;
    if (n > kMaxTasks) raise_abort(p);
  }
  if (threadIdx.x < kGuSlots) S.gu_cnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) tl_min(p, p.l0, EV_START);
  __syncthreads();
  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) producer(p, S);
  } else if (warp <= kNC) {
    consumer(p, S, warp - 1);
  } else {
    topk_warp(p, S);
  }
  __syncthreads();
  // the last CTA out zeroes the dependency counters for the next launch
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(p.exit_cnt, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.counters[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      *p.abort_flag = 0;
      *p.exit_cnt = 0;
      __threadfence();
    }
  }
}

}  // namespace

size_t persistent_smem() { return sizeof(Smem); }

int persistent_max_tiles_per_cta() { return kGuSlots; }

int persistent_max_tasks() { return kMaxTasks; }

cudaError_t persistent_attrs() {
  return cudaFuncSetAttribute((const void*)k_decode_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(Smem)));
}

cudaError_t persistent_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_decode_persistent, kPThreads,
                                                       sizeof(Smem));
}

cudaError_t launch_persistent(PParams& p, int grid, cudaStream_t s) {
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel((const void*)k_decode_persistent, dim3(grid), dim3(kPThreads), args,
                                     sizeof(Smem), s);
}

}  // namespace moe
