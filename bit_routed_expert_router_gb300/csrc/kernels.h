// Launchers of the libmoe kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

constexpr int kGuWarps = 4;     // warps per gate/up CTA, one row tile each
constexpr int kDnWarps = 8;     // warps per down CTA
constexpr int kMaxDecodeB = 32; // tokens per decode launch

// Persistent decode kernel (B = 1, resident, every layer in one launch).
constexpr int kPConsumers = 16;        // consumer warps per CTA
constexpr int kPStages = 5;            // shared-memory ring slots of four 11-group chunks
constexpr int kPStageGroups = 11;      // int4 groups (576 B each) per stage
constexpr int kPMaxD = 3072;
constexpr int kPThreads = 32 * (kPConsumers + 2);  // producer, consumers, top-k warp

struct PLayer {                        // device addresses of one layer's weights
  const uint16_t* router_w;
  const uint8_t* shared;
  const uint8_t* experts;
};

struct PParams {
  int d, f, fs, E, k, prenorm, gelu;
  float eps;
  int l0, l1;                          // layers of this call
  int n_sc;                            // shared down chunks of <= kPStageGroups groups
  long long expert_stride;
  const PLayer* layers;                // [n_layers]
  const DevCallArgs* args;
  uint16_t* hbuf0;
  uint16_t* hbuf1;
  long long* logits;                   // [n_layers][E]
  unsigned* counters;                  // all dependency counters, zeroed by the last CTA out
  int n_counters;
  unsigned* logit_cnt;                 // [n_layers]
  unsigned* gu_cnt;                    // [n_layers][n_sc + k]
  unsigned* row_cnt;                   // [n_layers][d / 16]
  unsigned* rows_done;                 // [n_layers]
  unsigned* exit_cnt;
  unsigned* abort_flag;
  uint16_t* a_s;                       // [2 * f_shared] hi/lo fragments
  uint16_t* a_r;                       // [k][2 * f]
  float* asum_s;                       // [f_shared / 8][2]
  float* asum_r;                       // [k][f / 8][2]
  float* part;                         // [2][n_sc + k][d]
  uint32_t* err;
  unsigned long long* timeline;        // optional [n_layers][16] event times (ns), null = off
  float* gates_g;                      // [n_layers][k] gates published before any routed work
  int n_layers_tl;                     // rows of the timeline's all-CTA part (= n_layers)
  long long spin_limit;                // bounded waits give up after this many cycles
};

size_t persistent_smem();
int persistent_max_tiles_per_cta();
int persistent_max_tasks();
cudaError_t persistent_attrs();
cudaError_t persistent_occupancy(int* blocks_per_sm);
cudaError_t launch_persistent(PParams& p, int grid, cudaStream_t s);

// Clustered persistent decode kernel (B = 1, resident, every layer in one
// launch on clusters of kCCluster CTAs, one CTA per SM).
constexpr int kCCluster = 4;           // CTAs per cluster
constexpr int kCStages = 7;            // shared-memory ring slots (one gate/up tile or down slice each)
constexpr int kCMaxUnits = 6;          // (source, group) units per cluster and layer
constexpr int kCMaxD = 2816;           // largest d of the clustered kernel (its ring slots are sized for it)
constexpr int kCThreads = 32 * 18;     // producer warp, 16 consumer warps, top-k warp

struct CLayer {                        // one layer, device memory (the tensor maps keep it 64-byte aligned)
  CUtensorMap dn_shared;               // shared expert's down region as u32 [1][d/16][f_s/64 * 144], box 144 x d/64
  CUtensorMap dn_routed;               // resident: the experts' down regions as u32 [E][d/16][f/64 * 144], same
                                       // box; host pool: the slots' down regions, [N][d/16][f/64 * 144]
  const uint16_t* router_w;            // fp16 [E][d]
  const uint8_t* shared;               // shared expert, device layout (gate/up region first)
  const uint8_t* experts;              // resident: expert 0, device layout; host pool: slot 0
  // host pool only (null otherwise): the layer's slot cache and its pinned pool
  const uint8_t* pool;                 // expert 0 of the layer in the mapped host pool, device layout
  int32_t* slot_of_expert;             // [E], -1 = not held
  int32_t* expert_of_slot;             // [N], -1 = empty
  long long* last_use;                 // [N], step of the slot's last use (-1: empty)
  long long* use_count;                // [E], picks over the run (LFU)
};

struct CParams {
  int d, f, fs, E, k, prenorm, gelu;
  float eps;
  int l0, l1;                          // layers of this call
  long long expert_stride;
  const CLayer* layers;                // [n_layers]
  const DevCallArgs* args;
  unsigned long long* tlog;            // [n_layers][n_cl][E][2]: per cluster, logit low / high word, each | tag << 32
  unsigned tag;                        // this launch's tag (never 0)
  long long spin_limit;                // bounded waits give up after this many cycles
  unsigned* diag;                      // first wait that ran out: site << 16 | CTA (0: none)
  // host-pool mode (pool != 0): cluster 0 runs the slot-cache step and publishes
  // each rank's (slot, hit) in plan; misses are read from the mapped pool
  int pool, n_slots, policy;
  unsigned long long* plan;            // [n_layers][32]: tag << 32 | slot << 16 | hit << 8 | expert
  int32_t* host_rec;                   // mapped [n_rel][1 + 6k]: misses (expert, slot), then per rank
                                       // (expert, hit, slot, evicted)
  long long* lru_counts;               // [n_layers][2]: hits, misses
  long long* ybuf;                     // [3][d] layer outputs: sum over CTAs of (v << 8) + 1, v on the 2^-32 grid;
                                       // zero between launches
  unsigned* exit_cnt;
  unsigned* abort_flag;
  uint32_t* err;
  unsigned long long* timeline;        // optional [grid][16] event times (ns) of one layer, null = off
};

// Cluster of shared unit G (of the shared expert's f_s/64 groups) when the
// Ur routed units are dealt round-robin over n_cl clusters (clusters below
// Ur mod n_cl get one more).  Shared units run while the routing is not yet
// known, so every cluster takes one before any takes two; the clusters with
// fewer routed units come first in that round-robin.
__host__ __device__ inline int cluster_unit_owner_shared(int G, int Ur, int n_cl) {
  const int extra = Ur % n_cl, i = G % n_cl;
  return i < n_cl - extra ? extra + i : i - (n_cl - extra);
}

size_t cluster_smem();
int cluster_max_units();
cudaError_t cluster_attrs();
cudaError_t cluster_max_active(int* n_clusters);
cudaError_t launch_cluster(CParams& p, int grid, cudaStream_t s);

// Prefill (tcgen05 grouped GEMM over int4 weights).
constexpr int kPfTileNBig = 256;       // token rows per GEMM tile (groups of about 200 rows and more)
constexpr int kPfTileN = 128;          // token rows per GEMM tile (mid-sized groups)
constexpr int kPfTileNSmall = 32;      // token rows per GEMM tile when every expert has only a few rows
constexpr int kPfMinDecodeB = 16;     // resident decode steps of at least this many tokens take the tcgen05 path
constexpr int kClusterLoopMaxB = 4;   // resident decode steps of 2 to this many tokens: one clustered launch per token
constexpr int kPfGraphMaxT = 512;     // tcgen05-path calls of at most this many tokens replay a CUDA graph
enum : int { PF_GU = 0, PF_DN_ROUTED = 1, PF_DN_SHARED = 2 };

struct PfGemm {
  const uint8_t* w;                    // weight region (gate/up or down) of expert 0, device layout
  long long w_stride;                  // bytes between experts (0: one matrix)
  int nG;                              // K / 64
  const int32_t* items;                // [n][3] expert, first row, rows; null: 128-row tiles of rows_total
  const int32_t* n_items_dev;          // item count on the device (null: n_items)
  int n_items, rows_total;
  int mode;                            // PF_*
  int d, k, gelu;
  uint16_t* out16;                     // PF_GU: fp16 [rows][f_out]
  int f_out;
  float* out32;                        // PF_DN_ROUTED: fp32 [T*k][d] by pair; PF_DN_SHARED: fp32 [T][d]
  const int32_t* pair_of_row;          // PF_DN_ROUTED: pair of each expert-ordered row
  uint32_t* err;
  unsigned long long* tl;              // optional: 16 event times (ns) of CTA (0, 0), null = off
};

size_t pf_gemm_smem(int n);
cudaError_t pf_set_attrs();
cudaError_t launch_pf_gemm(int n, const CUtensorMap& tmap_b, const PfGemm& p, int m_tiles, int max_items,
                           cudaStream_t s);
// xv / xg (or null): the tokens' x rows for the small-batch GEMVs (fp16 in
// their fragment order) and their 64-element group sums, [T][d] and [T][d / 64].
cudaError_t launch_pf_prep(const uint16_t* h, int T, int d, int prenorm, float eps, uint16_t* x_bf, uint16_t* x16,
                           uint16_t* dbg_x, float* xn2, float* xmax, uint16_t* xv, float* xg, uint32_t* err,
                           cudaStream_t s);
cudaError_t launch_pf_row_stats(const uint16_t* rows, int n, int d, float* n2, float* mx, cudaStream_t s);
cudaError_t launch_pf_router(const uint16_t* x_bf, const uint16_t* router_w, const float* bias, int T, int d, int E,
                             int k, float* approx, float* xn2, float* wn2, float* xmax, float* wmax, int32_t* ids,
                             float* gates, int32_t* dbg_ids, float* dbg_gates, int64_t* dbg_logits, uint32_t* err, int n_sm,
                             cudaStream_t s);
cudaError_t launch_pf_plan(const int32_t* ids, int P, int E, int tile, int32_t* cnt, int32_t* row_pair,
                           int32_t* items, int32_t* n_items, cudaStream_t s);
cudaError_t launch_pf_combine(const float* ys, const float* ytok, const float* gates, const uint16_t* hin,
                              uint16_t* hout, float* y_last, float* dbg_y, int T, int d, int k, cudaStream_t s);
cudaError_t launch_pf_gather(const uint16_t* x16, const int32_t* row_pair, int P, int d, int k, uint16_t* xp,
                             cudaStream_t s);

// Launches of the grouped path (routing, grouping, GEMMs or GEMVs, combine):
// with g_chain_pdl set, each may start while the previous kernel of the stream
// finishes (programmatic dependent launch); every such kernel waits for it
// (griddepcontrol.wait) before touching memory, so the setting changes timing
// only.  Set by the host for each call from its context.
extern bool g_chain_pdl;

template <typename... Params, typename... Args>
inline cudaError_t launch_chain(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_chain_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// Small-batch grouped GEMVs (mma.sync from a TMA ring) for calls of at most
// kSgMaxT tokens, after the prefill path's routing and expert grouping.
constexpr int kSgMaxT = 32;            // tokens of a small-batch call
constexpr int kSgMaxG = 44;            // int4 groups one ring slot holds (d, f, f_s <= 2816)
enum : int { SG_GU = 0, SG_DN = 1 };

struct SgParams {
  int mode;                            // SG_GU or SG_DN
  int d, f, fs, T, P, gelu;            // P = T * top_k expert-ordered rows
  const uint8_t* experts;              // expert 0's device record (gate/up tiles, then down)
  long long stride;                    // bytes between experts
  const uint8_t* shared;               // the shared expert's device record
  const int32_t* items;                // [n][3]: active expert, its first expert-ordered row, its rows (<= kSgMaxT)
  const int32_t* n_items;              // n, on the device
  const int32_t* row_pair;             // [P]: pair (t * k + j) of each expert-ordered row
  const uint16_t* xv;                  // [T][d]: fp16 x of each token in fragment order (an expert's row c
                                       // is token row_pair[row0 + c] / k)
  const float* xg;                     // [T][d / 64]: group sums of those rows
  uint16_t* av_r;                      // [P][f]: fp16 a of the routed rows, fragment order
  uint16_t* av_s;                      // [T][fs]: fp16 a of the shared expert, fragment order
  float* y_r;                          // [T * k][d]: routed down outputs by pair
  float* y_s;                          // [T][d]: shared down output
  uint32_t* err;
};

bool sg_shape_ok(int d, int f, int fs);
size_t sg_smem();
cudaError_t sg_set_attrs();
cudaError_t launch_sg(const SgParams& p, int n_sm, cudaStream_t s);

size_t gateup_smem(int d);
size_t down_smem(int cg, int nb4);
int pick_nb(int B);
int pick_nb4(int B);
cudaError_t set_kernel_attrs(int max_smem);
cudaError_t launch_router(KParams& p, int B, cudaStream_t s, bool pdl);
cudaError_t launch_gateup(KParams& p, int B, int max_items, int n_sm, cudaStream_t s, bool pdl);
cudaError_t launch_down(KParams& p, int B, int max_items, int n_sm, cudaStream_t s, bool pdl);
cudaError_t launch_repack(const uint8_t* gq, const uint16_t* gsb, const uint8_t* uq, const uint16_t* usb,
                          const uint8_t* dq, const uint16_t* dsb, int d, int f, uint8_t* dst, cudaStream_t s);

}  // namespace moe
