// Host side of libmoe: the C ABI declared in include/moe.h.
//
// Owns the device weights (repacked), the pinned host expert pool and the
// per-layer device slots of host-pool contexts, the per-call scratch, a side
// stream for staging copies, and the CUDA graphs that replay a resident
// decode step (router, gate/up, down per layer) with one launch.
#include "moe.h"

#include <chrono>
#include <cerrno>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <thread>
#include <tuple>
#include <new>
#include <vector>

#ifndef _GNU_SOURCE
#define _GNU_SOURCE
#endif
#include <fcntl.h>
#include <unistd.h>

#include "expert_file.h"

#include <cudaTypedefs.h>

#include "internal.h"
#include "kernels.h"
#include "staging.h"

using namespace moe;

namespace {

constexpr int kArgRing = 32;

struct LayerStore {
  bool ready = false;
  uint16_t* router_w = nullptr;       // device fp16 [E][d]
  float* router_stats = nullptr;      // device [2][E]: |row|^2 and max |row_i| (prefill router bound)
  uint8_t* shared = nullptr;          // device layout
  uint8_t* experts = nullptr;         // resident: E * stride
  uint8_t* slots = nullptr;           // host pool: N * stride
  int32_t* slot_of_expert = nullptr;  // [E]
  int32_t* expert_of_slot = nullptr;  // [N]
  long long* last_use = nullptr;      // [N]
  long long* use_count = nullptr;     // [E] whole-run picks per expert (LFU)
};

template <class T>
T* dalloc(size_t n, std::vector<void*>& owned, size_t& bytes) {
  void* p = nullptr;
  if (cudaMalloc(&p, n * sizeof(T) > 0 ? n * sizeof(T) : 16) != cudaSuccess) return nullptr;
  owned.push_back(p);
  bytes += n * sizeof(T);
  return static_cast<T*>(p);
}

}  // namespace

struct moe_ctx {
  moe_config cfg{};
  int device = 0;
  int n_sm = 148;
  bool poisoned = false;
  std::string err;
  int residency = -1;
  int n_slots = 0;
  long long expert_bytes = 0, shared_bytes = 0, stride = 0;
  int n_sc = 1, cg = 1, Bd = 1;
  std::vector<LayerStore> L;
  uint8_t* pool = nullptr;
  const uint8_t* pool_dev = nullptr;     // the pool's device address (mapped), or null
  bool stage_device = false;             // moe_set_staging(MOE_STAGING_DEVICE)
  bool stage_fused = false;              // moe_set_staging(MOE_STAGING_FUSED): the clustered kernel does it all
  size_t pool_bytes = 0;
  // expert file tier (MOE_FILE_POOL contexts)
  int file_fd = -1;
  int file_rfd = -1;                     // O_DIRECT read descriptor (MOE_FILE_DIRECT), else -1
  FilePool* fpool = nullptr;
  uint64_t file_chunk = 512u << 10;
  size_t file_stride = 0;                // bytes between records (expert device bytes rounded up to 4096)
  uint8_t* fstage = nullptr;             // pinned [2][top_k][file_stride] staging records
  cudaEvent_t fev[2] = {nullptr, nullptr};   // copies out of each staging half done
  int fhalf = 0;
  long long file_read_bytes = 0, file_read_us = 0;
  // host tier in front of the expert file (moe_set_file_cache): per layer n_host
  // pinned records with an LRU table; a miss of the slot cache that the host
  // tier holds is copied from it, any other is read from the file into it
  int n_host = 0;
  uint8_t* hcache = nullptr;             // pinned [n_layers][n_host][file_stride]
  std::vector<int32_t> h_expert_of_slot; // [n_layers][n_host], -1 = empty
  std::vector<long long> h_last_use;     // [n_layers][n_host], -1 = empty
  std::vector<int32_t> h_slot_of_expert; // [n_layers][n_experts], -1 = not held
  std::vector<char> h_touched;           // [n_host] scratch of one step
  const uint8_t* h_src[32] = {};         // source record of each miss of the current layer
  cudaEvent_t hev = nullptr;             // every copy out of the host tier issued so far is done
  long long host_hits = 0;
  std::vector<void*> owned;           // scratch allocations
  size_t device_bytes = 0;
  // scratch
  uint16_t* hbuf[2] = {nullptr, nullptr};
  uint16_t* x_perm = nullptr;
  float* xg = nullptr;
  long long* logits = nullptr;
  int32_t* ids = nullptr;
  float* gates = nullptr;
  int32_t* tok_cnt = nullptr;
  int32_t* all_cnt = nullptr;
  PlanHdr* plan = nullptr;
  int32_t *act_expert = nullptr, *act_off = nullptr, *act_cnt = nullptr, *act_pass = nullptr;
  int32_t* pair_tok = nullptr;
  float* pair_gate = nullptr;
  int32_t* pos_of = nullptr;
  uint16_t *a_s = nullptr, *a_r = nullptr;
  float *asum_s = nullptr, *asum_r = nullptr, *part_s = nullptr, *y_r = nullptr;
  int32_t* row_cnt = nullptr;
  uint32_t* err_word = nullptr;
  long long* lru_counts = nullptr;
  int policy = MOE_CACHE_LRU;         // slot cache eviction policy (host-pool contexts)
  DevCallArgs* dargs = nullptr;
  DevCallArgs* args_ring = nullptr;   // pinned host ring of argument blocks
  cudaEvent_t ring_ev[kArgRing] = {};
  bool ring_used[kArgRing] = {};
  int ring_pos = 0;
  int32_t* host_rec = nullptr;        // pinned, mapped
  int32_t* host_rec_dev = nullptr;
  cudaStream_t side = nullptr;
  cudaStream_t cap = nullptr;
  cudaEvent_t ev_route = nullptr, ev_copy = nullptr;
  // debug capture
  uint16_t* dbg_x = nullptr;
  int32_t* dbg_ids = nullptr;
  float* dbg_gates = nullptr;
  float* dbg_y = nullptr;
  int64_t* dbg_logits = nullptr;
  int dbg_layers = 0;
  // counters
  long long step = 0, steps = 0, staged = 0;
  // hooks
  bool hook_fail_copy = false;
  bool hook_force_timeout = false;     // the next host wait reports a timeout
  long long hook_free_bytes = -1;      // >= 0: budget checks use this as free device memory
  long long wait_limit_us = 20000000;
  bool pdl = true;
  std::map<std::tuple<int, int, int>, cudaGraphExec_t> graphs;
  // tcgen05-path graphs for small batches: key (T, l0, l1, with bias, with y_last)
  std::map<std::tuple<int, int, int, int, int>, cudaGraphExec_t> pf_graphs;
  uint16_t *pf_gin = nullptr, *pf_gout = nullptr;   // graph-owned copies of h in / h out [max_tokens][d]
  float* pf_gbias = nullptr;                        // [n_layers][max_tokens][E], made on first use
  float* pf_gy = nullptr;                           // [max_tokens][d]
  // persistent decode kernel (resident, B = 1)
  bool use_persistent = true;
  bool p_ok = false;                   // one CTA per SM fits
  PLayer* p_layers = nullptr;          // device [n_layers]
  long long* p_logits = nullptr;
  unsigned* p_counters = nullptr;
  int p_n_counters = 0;
  unsigned* p_exit = nullptr;          // exit counter, abort flag
  uint16_t *p_a_s = nullptr, *p_a_r = nullptr;
  float *p_asum_s = nullptr, *p_asum_r = nullptr, *p_part = nullptr;
  int p_n_sc = 1;
  float* p_gates = nullptr;            // [n_layers][k]
  // clustered persistent decode kernel (resident, B = 1; preferred when available)
  bool c_ok = false;                   // shapes and device allow it
  bool use_cluster = true;             // test hook 9
  int c_grid = 0;                      // CTAs: resident clusters x kCCluster
  CLayer* c_layers = nullptr;          // device [n_layers]
  unsigned long long* c_plan = nullptr;  // device [n_layers][32]: host-pool plan words of the clustered kernel
  unsigned long long* c_tlog = nullptr;  // [n_layers][n_cl][E][2] tagged logits, one replica per cluster
  bool c_loop = true;                    // 2 to kClusterLoopMaxB tokens: one clustered launch per token
  long long spin_limit = 4000000000LL; // test hook 10: wait limit (cycles) of the clustered kernel's bounded waits
  long long* c_ybuf = nullptr;         // [3][d] fixed-point layer outputs
  unsigned* c_counters = nullptr;      // exit counter, abort flag
  unsigned c_tag = 0;                  // tag of the last launch
  // batched prefill on tcgen05 (resident contexts): scratch for max_tokens tokens, made on first use
  bool pf_ok = false;                  // shapes and device allow it
  bool use_pf = true;                  // test hook 7
  bool pf_ready = false;
  std::vector<void*> pf_owned;
  uint16_t *pf_xbf = nullptr, *pf_x16 = nullptr, *pf_xp = nullptr, *pf_ar = nullptr, *pf_as = nullptr;
  uint16_t* pf_h[2] = {nullptr, nullptr};
  int32_t *pf_ids = nullptr, *pf_cnt = nullptr, *pf_rowpair = nullptr, *pf_items = nullptr, *pf_nitems = nullptr;
  float *pf_gates = nullptr, *pf_ytok = nullptr;
  float *pf_approx = nullptr, *pf_xn2 = nullptr, *pf_xmax = nullptr;
  float* pf_ys = nullptr;
  // small-batch grouped GEMVs (calls of at most kSgMaxT tokens on the tcgen05 path's routing)
  bool sg_ok = false;                  // shapes and device allow it
  bool use_sg = true;                  // test hook 13
  uint16_t* sg_xv = nullptr;           // [kSgMaxT][d] fp16 x of each token in fragment order
  float* sg_xg = nullptr;              // [kSgMaxT][d / 64] their group sums
  unsigned long long* pf_timeline = nullptr;   // test hook 8: [4][16] GEMM event times of the first layer
  // chunked prefill of host-pool / expert-file contexts: the union of a chunk's
  // experts of one layer, staged into an arena (expert e at e * stride)
  uint8_t* pf_arena = nullptr;
  int32_t* pf_cnt_host = nullptr;              // pinned [n_experts]: pairs per expert of the layer
  cudaEvent_t pf_ev_cnt = nullptr;             // pf_cnt_host filled
  cudaEvent_t pf_ev_read = nullptr;            // the GEMMs that read the arena last are done
  CUtensorMap pf_map_xp[3]{}, pf_map_x16[3]{}, pf_map_ar[3]{}, pf_map_as[3]{};   // [0]: 128-row boxes, [1]: 32, [2]: 256
  unsigned long long* p_timeline = nullptr;   // caller device buffer [n_layers][16], test hook 5
  // per-kernel timing
  bool profiling = false;
  std::vector<cudaEvent_t> prof_ev;
  std::vector<int> prof_kind;
  int prof_n = 0;
  moe_kernel_time prof[MOE_N_KERNEL_KINDS] = {};
};

namespace {

thread_local std::string g_create_error;  // why the last moe_create failed

moe_status fail(moe_ctx* c, moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) {
    c->err = buf;
    if (s == MOE_ECUDA || s == MOE_ETIMEOUT || s == MOE_EIO) c->poisoned = true;
  }
  return s;
}

#define CK(call)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail(ctx, MOE_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

bool cfg_valid(const moe_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("config is NULL");
  if (c->group != 64) return bad("group must be 64");
  if (c->d <= 0 || c->d % 64 || c->d > 3072) return bad("d must be a positive multiple of 64, at most 3072");
  if (c->f <= 0 || c->f % 64) return bad("f must be a positive multiple of 64");
  if (c->f_shared <= 0 || c->f_shared % 64) return bad("f_shared must be a positive multiple of 64");
  if (c->n_experts < 1 || c->n_experts > 256) return bad("n_experts must be in [1, 256]");
  if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > 32) return bad("top_k must be in [1, min(n_experts, 32)]");
  if (c->n_layers < 1 || c->n_layers > 4096) return bad("n_layers must be in [1, 4096]");
  if (c->gelu_variant != 0 && c->gelu_variant != 1) return bad("gelu_variant must be 0 or 1");
  if (c->prenorm != 0 && c->prenorm != 1) return bad("prenorm must be 0 or 1");
  if (c->max_tokens < 1 || c->max_tokens > 65536) return bad("max_tokens must be in [1, 65536]");
  if (!(c->norm_eps >= 0.f) || c->norm_eps > 1.f) return bad("norm_eps must be in [0, 1]");
  return true;
}

long long expert_bytes_of(int d, int f) { return static_cast<long long>(f) * d * 27 / 16; }

long long now_us() {
  return std::chrono::duration_cast<std::chrono::microseconds>(
             std::chrono::steady_clock::now().time_since_epoch())
      .count();
}

// Bounded host wait on an event.
moe_status wait_event(moe_ctx* ctx, cudaEvent_t ev, const char* what) {
  if (ctx->hook_force_timeout) {
    ctx->hook_force_timeout = false;
    cudaEventSynchronize(ev);  // leave no work of ours in flight
    return fail(ctx, MOE_ETIMEOUT, "waiting for %s: time limit (forced by test hook)", what);
  }
  const long long t0 = now_us();
  int spins = 0;
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotReady) return fail(ctx, MOE_ECUDA, "waiting for %s: %s", what, cudaGetErrorString(e));
    if (now_us() - t0 > ctx->wait_limit_us) return fail(ctx, MOE_ETIMEOUT, "waiting for %s: time limit", what);
    if (++spins > 64) std::this_thread::yield();
  }
}

cudaError_t free_device_bytes(moe_ctx* ctx, size_t* free_b) {
  size_t total_b = 0;
  cudaError_t e = cudaMemGetInfo(free_b, &total_b);
  if (e == cudaSuccess && ctx->hook_free_bytes >= 0) *free_b = static_cast<size_t>(ctx->hook_free_bytes);
  return e;
}

KParams base_params(moe_ctx* ctx, int layer, int rel, int first, int last, int B) {
  KParams p{};
  const moe_config& c = ctx->cfg;
  p.d = c.d;
  p.f = c.f;
  p.fs = c.f_shared;
  p.E = c.n_experts;
  p.k = c.top_k;
  p.B = B;
  p.prenorm = c.prenorm;
  p.gelu = c.gelu_variant;
  p.eps = c.norm_eps;
  p.n_sc = ctx->n_sc;
  p.cg = ctx->cg;
  p.layer = layer;
  p.rel_layer = rel;
  p.first = first;
  p.last = last;
  p.pool = ctx->residency == MOE_HOST_POOL || ctx->residency == MOE_FILE_POOL;
  p.pass = -1;
  p.n_slots = ctx->n_slots;
  const LayerStore& Ls = ctx->L[layer];
  p.router_w = Ls.router_w;
  p.shared = Ls.shared;
  p.experts = p.pool ? Ls.slots : Ls.experts;
  p.expert_stride = ctx->stride;
  p.slot_of_expert = Ls.slot_of_expert;
  p.expert_of_slot = Ls.expert_of_slot;
  p.last_use = Ls.last_use;
  p.lru_counts = ctx->lru_counts;
  p.policy = ctx->policy;
  p.use_count = Ls.use_count;
  p.host_rec = ctx->host_rec_dev;
  p.args = ctx->dargs;
  p.x_perm = ctx->x_perm;
  p.xg = ctx->xg;
  p.logits = ctx->logits;
  p.ids = ctx->ids;
  p.gates = ctx->gates;
  p.tok_cnt = ctx->tok_cnt;
  p.all_cnt = ctx->all_cnt;
  p.plan = ctx->plan;
  p.act_expert = ctx->act_expert;
  p.act_off = ctx->act_off;
  p.act_cnt = ctx->act_cnt;
  p.act_pass = ctx->act_pass;
  p.pair_tok = ctx->pair_tok;
  p.pair_gate = ctx->pair_gate;
  p.pos_of = ctx->pos_of;
  p.a_s = ctx->a_s;
  p.a_r = ctx->a_r;
  p.asum_s = ctx->asum_s;
  p.asum_r = ctx->asum_r;
  p.part_s = ctx->part_s;
  p.y_r = ctx->y_r;
  p.row_cnt = ctx->row_cnt;
  p.err = ctx->err_word;
  return p;
}

int gu_max_items(const moe_ctx* ctx, int B) {
  const moe_config& c = ctx->cfg;
  const int maxU = std::min(c.n_experts, B * c.top_k);
  return c.f_shared / 8 + maxU * (c.f / 8);
}

int dn_max_items(const moe_ctx* ctx, int B) {
  const moe_config& c = ctx->cfg;
  const int maxU = std::min(c.n_experts, B * c.top_k);
  return (c.d / 16) * (ctx->n_sc + maxU);
}

// Event pair around one launch while profiling.
moe_status prof_mark(moe_ctx* ctx, int kind, cudaStream_t s) {
  if (!ctx->profiling) return MOE_OK;
  if (ctx->prof_n + 1 >= static_cast<int>(ctx->prof_ev.size())) {
    for (int i = 0; i < 256; ++i) {
      cudaEvent_t e;
      CK(cudaEventCreate(&e));
      ctx->prof_ev.push_back(e);
    }
    ctx->prof_kind.resize(ctx->prof_ev.size() / 2 + 1);
  }
  if (kind >= 0) ctx->prof_kind[ctx->prof_n / 2] = kind;
  CK(cudaEventRecord(ctx->prof_ev[ctx->prof_n++], s));
  return MOE_OK;
}

#define PROF(kind, s)                              \
  do {                                             \
    moe_status ps_ = prof_mark(ctx, (kind), (s));  \
    if (ps_ != MOE_OK) return ps_;                 \
  } while (0)

moe_status prof_collect(moe_ctx* ctx, cudaStream_t s) {
  if (!ctx->profiling || ctx->prof_n == 0) return MOE_OK;
  CK(cudaStreamSynchronize(s));
  for (int i = 0; i + 1 < ctx->prof_n; i += 2) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, ctx->prof_ev[i], ctx->prof_ev[i + 1]));
    moe_kernel_time& t = ctx->prof[ctx->prof_kind[i / 2]];
    t.launches += 1;
    t.total_ms += ms;
  }
  ctx->prof_n = 0;
  return MOE_OK;
}

// Enqueue the three kernels of one resident layer on stream s.
moe_status enqueue_layer(moe_ctx* ctx, int layer, int rel, int n_rel, int B, cudaStream_t s) {
  KParams p = base_params(ctx, layer, rel, rel == 0, rel == n_rel - 1, B);
  p.h_src = rel == 0 ? nullptr : ctx->hbuf[(rel - 1) & 1];
  p.h_dst = rel == n_rel - 1 ? nullptr : ctx->hbuf[rel & 1];
  const bool pdl = ctx->pdl && !ctx->profiling;
  PROF(0, s);
  CK(launch_router(p, B, s, pdl));
  PROF(-1, s);
  PROF(1, s);
  CK(launch_gateup(p, B, gu_max_items(ctx, B), ctx->n_sm, s, pdl));
  PROF(-1, s);
  PROF(2, s);
  CK(launch_down(p, B, dn_max_items(ctx, B), ctx->n_sm, s, pdl));
  PROF(-1, s);
  return MOE_OK;
}

// Write the per-call argument block through a pinned ring slot.
moe_status put_args(moe_ctx* ctx, const DevCallArgs& a, cudaStream_t s) {
  const int i = ctx->ring_pos;
  ctx->ring_pos = (ctx->ring_pos + 1) % kArgRing;
  if (ctx->ring_used[i]) {
    moe_status st = wait_event(ctx, ctx->ring_ev[i], "argument ring slot");
    if (st != MOE_OK) return st;
  }
  ctx->args_ring[i] = a;
  CK(cudaMemcpyAsync(ctx->dargs, &ctx->args_ring[i], sizeof(DevCallArgs), cudaMemcpyHostToDevice, s));
  CK(cudaEventRecord(ctx->ring_ev[i], s));
  ctx->ring_used[i] = true;
  return MOE_OK;
}

bool dbg_on(const moe_ctx* ctx) {
  return ctx->dbg_x || ctx->dbg_ids || ctx->dbg_gates || ctx->dbg_y || ctx->dbg_logits;
}

DevCallArgs make_args(moe_ctx* ctx, const void* h_in, void* h_out, float* y_last, const float* bias, int B,
                      int tok_total, int tok_off) {
  DevCallArgs a{};
  a.h_in = static_cast<const uint16_t*>(h_in);
  a.h_out = static_cast<uint16_t*>(h_out);
  a.y_last = y_last;
  a.bias = bias;
  a.dbg_x = ctx->dbg_x;
  a.dbg_ids = ctx->dbg_ids;
  a.dbg_gates = ctx->dbg_gates;
  a.dbg_y = ctx->dbg_y;
  a.dbg_logits = ctx->dbg_logits;
  a.dbg_layers = dbg_on(ctx) ? ctx->dbg_layers : 0;
  a.B = B;
  a.tok_total = tok_total;
  a.tok_off = tok_off;
  a.step = ctx->step;
  return a;
}

moe_status check_ready(moe_ctx* ctx, int l0, int l1) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (l0 < 0 || l1 > ctx->cfg.n_layers || l0 >= l1) return fail(ctx, MOE_EINVAL, "bad layer range [%d, %d)", l0, l1);
  for (int l = l0; l < l1; ++l)
    if (!ctx->L[l].ready) return fail(ctx, MOE_ESTATE, "layer %d is not initialised", l);
  return MOE_OK;
}

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// does not link libcuda itself (it loads on machines without a driver).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

// 3-D tensor map over the down regions of n_mat matrices seen as 32-bit words:
// x = the nG * 144 words of one 16-row tile (nG groups of 576 bytes), y = the
// nT tiles, z = the matrices (mat_stride bytes apart).  A box is one group of
// nT / 4 consecutive tiles: the down slice of one cluster rank for one unit.
bool encode_down(CUtensorMap* m, const void* base, int nG, int nT, int n_mat, long long mat_stride) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(nG) * kGroupBytes;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(nG) * (kGroupBytes / 4), static_cast<cuuint64_t>(nT),
                        static_cast<cuuint64_t>(n_mat)};
  cuuint64_t gstride[2] = {row, n_mat > 1 ? static_cast<cuuint64_t>(mat_stride) : row * nT};
  cuuint32_t box[3] = {kGroupBytes / 4, static_cast<cuuint32_t>(nT / kCCluster), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest number of (source, group) units any cluster gets per layer (the
// kernel's dealing rule: routed unit i -> cluster i mod n_cl, shared units by
// cluster_unit_owner_shared).
int cluster_units_max(const moe_config& c, int n_cl) {
  const int Ur = c.top_k * (c.f / 64);
  std::vector<int> n(static_cast<size_t>(n_cl), 0);
  for (int i = 0; i < Ur; ++i) ++n[static_cast<size_t>(i % n_cl)];
  for (int G = 0; G < c.f_shared / 64; ++G) ++n[static_cast<size_t>(cluster_unit_owner_shared(G, Ur, n_cl))];
  int m = 0;
  for (int v : n) m = v > m ? v : m;
  return m;
}

// The clustered kernel's view of a host-pool layer: its slots in place of
// the resident experts (down tensor map over the N slots), the mapped pool and
// the slot-cache state.  Built once the layer and its slots both exist.
moe_status cluster_pool_layer(moe_ctx* ctx, int l) {
  const moe_config& c = ctx->cfg;
  LayerStore& Ls = ctx->L[static_cast<size_t>(l)];
  if (!ctx->c_ok || !ctx->pool_dev || ctx->residency != MOE_HOST_POOL || !Ls.ready || !Ls.slots || ctx->n_slots < 1)
    return MOE_OK;
  CLayer cl{};
  const size_t gu_s = static_cast<size_t>(c.f_shared / 8) * (c.d / 64) * kGroupBytes;
  const size_t gu_r = static_cast<size_t>(c.f / 8) * (c.d / 64) * kGroupBytes;
  if (!encode_down(&cl.dn_shared, Ls.shared + gu_s, c.f_shared / 64, c.d / 16, 1, 0) ||
      !encode_down(&cl.dn_routed, Ls.slots + gu_r, c.f / 64, c.d / 16, ctx->n_slots, ctx->stride))
    return fail(ctx, MOE_ECUDA, "layer %d: cuTensorMapEncodeTiled failed for the slots' down regions", l);
  cl.router_w = Ls.router_w;
  cl.shared = Ls.shared;
  cl.experts = Ls.slots;
  cl.pool = ctx->pool_dev + static_cast<size_t>(l) * c.n_experts * ctx->stride;
  cl.slot_of_expert = Ls.slot_of_expert;
  cl.expert_of_slot = Ls.expert_of_slot;
  cl.last_use = Ls.last_use;
  cl.use_count = Ls.use_count;
  CK(cudaMemcpy(ctx->c_layers + l, &cl, sizeof(CLayer), cudaMemcpyHostToDevice));
  return MOE_OK;
}

// Resident decode of one token through [l0, l1) with the clustered kernel.
moe_status cluster_run(moe_ctx* ctx, int l0, int l1, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  CParams p{};
  p.d = c.d;
  p.f = c.f;
  p.fs = c.f_shared;
  p.E = c.n_experts;
  p.k = c.top_k;
  p.prenorm = c.prenorm;
  p.gelu = c.gelu_variant;
  p.eps = c.norm_eps;
  p.l0 = l0;
  p.l1 = l1;
  p.expert_stride = ctx->stride;
  p.layers = ctx->c_layers;
  p.args = ctx->dargs;
  if (++ctx->c_tag == 0) {   // tags wrapped: no stale entry may carry the new one
    CK(cudaMemsetAsync(ctx->c_tlog, 0, static_cast<size_t>(c.n_layers) * (ctx->c_grid / kCCluster) * c.n_experts * 16,
                       s));
    CK(cudaMemsetAsync(ctx->c_plan, 0, static_cast<size_t>(c.n_layers) * 32 * 8, s));
    ctx->c_tag = 1;
  }
  if (ctx->residency == MOE_HOST_POOL && ctx->stage_fused) {
    p.pool = 1;
    p.n_slots = ctx->n_slots;
    p.policy = ctx->policy;
    p.plan = ctx->c_plan;
    p.host_rec = ctx->host_rec_dev;
    p.lru_counts = ctx->lru_counts;
  }
  p.tlog = ctx->c_tlog;
  p.tag = ctx->c_tag;
  p.ybuf = ctx->c_ybuf;
  p.exit_cnt = ctx->c_counters;
  p.abort_flag = ctx->c_counters + 1;
  p.diag = ctx->c_counters + 2;
  p.err = ctx->err_word;
  p.timeline = ctx->p_timeline;
  p.spin_limit = ctx->spin_limit;
  PROF(3, s);
  CK(launch_cluster(p, ctx->c_grid, s));
  PROF(-1, s);
  return prof_collect(ctx, s);
}

// Resident decode of one token through [l0, l1) with the persistent kernel.
moe_status persistent_run(moe_ctx* ctx, int l0, int l1, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  PParams p{};
  p.d = c.d;
  p.f = c.f;
  p.fs = c.f_shared;
  p.E = c.n_experts;
  p.k = c.top_k;
  p.prenorm = c.prenorm;
  p.gelu = c.gelu_variant;
  p.eps = c.norm_eps;
  p.l0 = l0;
  p.l1 = l1;
  p.n_sc = ctx->p_n_sc;
  p.expert_stride = ctx->stride;
  p.layers = ctx->p_layers;
  p.args = ctx->dargs;
  p.hbuf0 = ctx->hbuf[0];
  p.hbuf1 = ctx->hbuf[1];
  p.logits = ctx->p_logits;
  p.counters = ctx->p_counters;
  p.n_counters = ctx->p_n_counters;
  const int pparts = ctx->p_n_sc + c.top_k;
  p.logit_cnt = ctx->p_counters;
  p.gu_cnt = p.logit_cnt + c.n_layers;
  p.row_cnt = p.gu_cnt + static_cast<size_t>(c.n_layers) * pparts;
  p.rows_done = p.row_cnt + static_cast<size_t>(c.n_layers) * (c.d / 16);
  p.exit_cnt = ctx->p_exit;
  p.abort_flag = ctx->p_exit + 1;
  p.a_s = ctx->p_a_s;
  p.a_r = ctx->p_a_r;
  p.asum_s = ctx->p_asum_s;
  p.asum_r = ctx->p_asum_r;
  p.part = ctx->p_part;
  p.err = ctx->err_word;
  p.timeline = ctx->p_timeline;
  p.gates_g = ctx->p_gates;
  p.n_layers_tl = c.n_layers;
  p.spin_limit = ctx->spin_limit;
  PROF(3, s);
  CK(launch_persistent(p, ctx->n_sm, s));
  PROF(-1, s);
  return prof_collect(ctx, s);
}

// Resident decode of B tokens through [l0, l1): one graph launch (or, while
// profiling, direct launches with event pairs).
moe_status resident_run(moe_ctx* ctx, int B, int l0, int l1, cudaStream_t s) {
  if (ctx->profiling) {
    for (int l = l0; l < l1; ++l) {
      moe_status st = enqueue_layer(ctx, l, l - l0, l1 - l0, B, s);
      if (st != MOE_OK) return st;
    }
    return prof_collect(ctx, s);
  }
  const auto key = std::make_tuple(B, l0, l1);
  auto it = ctx->graphs.find(key);
  if (it == ctx->graphs.end()) {
    cudaGraph_t g = nullptr;
    CK(cudaStreamBeginCapture(ctx->cap, cudaStreamCaptureModeThreadLocal));
    moe_status st = MOE_OK;
    for (int l = l0; l < l1 && st == MOE_OK; ++l) st = enqueue_layer(ctx, l, l - l0, l1 - l0, B, ctx->cap);
    cudaError_t e = cudaStreamEndCapture(ctx->cap, &g);
    if (st != MOE_OK) {
      if (g) cudaGraphDestroy(g);
      return st;
    }
    CK(e);
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    CK(e);
    it = ctx->graphs.emplace(key, ex).first;
  }
  CK(cudaGraphLaunch(it->second, s));
  return MOE_OK;
}

// One read of expert `ex` of layer `l` from the expert file into `dst` (pinned,
// 4096-byte aligned, file_stride bytes).
moe_status file_read_record(moe_ctx* ctx, int l, int ex, uint8_t* dst) {
  const uint64_t off = (static_cast<uint64_t>(l) * ctx->cfg.n_experts + ex) * ctx->file_stride;
  const long long t0 = now_us();
  // O_DIRECT reads whole 4096-byte-aligned records
  const bool direct = ctx->file_rfd >= 0;
  const int e = file_pool_transfer(ctx->fpool, direct ? ctx->file_rfd : ctx->file_fd, false, off, dst,
                                   direct ? ctx->file_stride : ctx->expert_bytes, ctx->file_chunk);
  ctx->file_read_us += now_us() - t0;
  if (e != 0) return fail(ctx, MOE_EIO, "expert file read (layer %d, expert %d): %s", l, ex, strerror(e));
  ctx->file_read_bytes += ctx->expert_bytes;
  return MOE_OK;
}

// The host tier's step for the slot-cache misses of layer `l` (rec: the miss
// record, n_miss >= 1), with the slot cache's LRU rules one level down: the
// misses it holds refresh their record (last use = the step counter); the
// others, in top-k order, each take the record with the smallest (last use,
// index) among those this step has not touched (empty ones first) and are read
// from the file into it.  Sets h_src[m] to each miss's source record.
moe_status host_tier_step(moe_ctx* ctx, int l, const volatile int32_t* rec, int n_miss) {
  const int H = ctx->n_host;
  uint8_t* base = ctx->hcache + static_cast<size_t>(l) * H * ctx->file_stride;
  int32_t ids[32], where[32], hit[32], evicted[32];
  for (int m = 0; m < n_miss; ++m) ids[m] = rec[1 + 2 * m];
  const int n_read = host_tier_lru_step(H, ctx->h_expert_of_slot.data() + static_cast<size_t>(l) * H,
                                        ctx->h_last_use.data() + static_cast<size_t>(l) * H,
                                        ctx->h_slot_of_expert.data() + static_cast<size_t>(l) * ctx->cfg.n_experts,
                                        ids, n_miss, ctx->step, where, hit, evicted, ctx->h_touched.data());
  if (n_read < 0) return fail(ctx, MOE_ECUDA, "host tier has no free record (%d records, %d misses)", H, n_miss);
  // a record is rewritten only once the copies issued out of it earlier are done
  if (n_read > 0) CK(cudaEventSynchronize(ctx->hev));
  for (int m = 0; m < n_miss; ++m) {
    uint8_t* dst = base + static_cast<size_t>(where[m]) * ctx->file_stride;
    if (hit[m]) {
      ++ctx->host_hits;
    } else {
      moe_status st = file_read_record(ctx, l, ids[m], dst);
      if (st != MOE_OK) return st;
    }
    ctx->h_src[m] = dst;
  }
  return MOE_OK;
}

void host_tier_clear(moe_ctx* ctx) {
  std::fill(ctx->h_expert_of_slot.begin(), ctx->h_expert_of_slot.end(), -1);
  std::fill(ctx->h_last_use.begin(), ctx->h_last_use.end(), -1);
  std::fill(ctx->h_slot_of_expert.begin(), ctx->h_slot_of_expert.end(), -1);
  ctx->host_hits = 0;
  ctx->file_read_bytes = 0;
  ctx->file_read_us = 0;
}

// Host-pool decode of one token through [l0, l1): per layer, route + LRU,
// shared and hit experts while the misses are staged, then the misses, then down.
moe_status pool_run(moe_ctx* ctx, int l0, int l1, cudaStream_t s, moe_trace_rec* trace, int trace_cap,
                    int* trace_len) {
  const int k = ctx->cfg.top_k;
  int n_rec = 0;
  for (int l = l0; l < l1; ++l) {
    const int rel = l - l0, n_rel = l1 - l0;
    KParams p = base_params(ctx, l, rel, rel == 0, rel == n_rel - 1, 1);
    p.h_src = rel == 0 ? nullptr : ctx->hbuf[(rel - 1) & 1];
    p.h_dst = rel == n_rel - 1 ? nullptr : ctx->hbuf[rel & 1];
    CK(launch_router(p, 1, s, false));
    CK(cudaEventRecord(ctx->ev_route, s));
    p.pass = 0;
    CK(launch_gateup(p, 1, gu_max_items(ctx, 1), ctx->n_sm, s, false));
    moe_status st = wait_event(ctx, ctx->ev_route, "router / LRU step");
    if (st != MOE_OK) return st;
    const volatile int32_t* rec = ctx->host_rec + static_cast<size_t>(rel) * (1 + 6 * k);
    const int n_miss = rec[0];
    if (n_miss < 0 || n_miss > k) return fail(ctx, MOE_ECUDA, "corrupt miss record (%d)", n_miss);
    const LayerStore& Ls = ctx->L[l];
    const bool from_file = ctx->file_fd >= 0;
    const bool tiered = from_file && ctx->n_host > 0;
    const int half = ctx->fhalf;
    for (int m = 0; m < n_miss; ++m) {
      const int ex = rec[1 + 2 * m], slot = rec[2 + 2 * m];
      if (ex < 0 || ex >= ctx->cfg.n_experts || slot < 0 || slot >= ctx->n_slots)
        return fail(ctx, MOE_ECUDA, "corrupt miss record (expert %d, slot %d)", ex, slot);
    }
    if (tiered && n_miss > 0) {
      st = host_tier_step(ctx, l, rec, n_miss);
      if (st != MOE_OK) return st;
    } else if (from_file && n_miss > 0) {
      // the copies out of this staging half two layers ago must be done before it is refilled
      CK(cudaEventSynchronize(ctx->fev[half]));
    }
    for (int m = 0; m < n_miss; ++m) {
      const int ex = rec[1 + 2 * m], slot = rec[2 + 2 * m];
      if (ctx->hook_fail_copy) {
        ctx->hook_fail_copy = false;
        return fail(ctx, MOE_ECUDA, "staging copy failed (injected by test hook)");
      }
      const uint8_t* src;
      if (tiered) {
        src = ctx->h_src[m];
      } else if (from_file) {
        uint8_t* dst = ctx->fstage + (static_cast<size_t>(half) * k + m) * ctx->file_stride;
        st = file_read_record(ctx, l, ex, dst);
        if (st != MOE_OK) return st;
        src = dst;
      } else {
        src = ctx->pool + (static_cast<size_t>(l) * ctx->cfg.n_experts + ex) * ctx->stride;
      }
      CK(cudaMemcpyAsync(Ls.slots + static_cast<size_t>(slot) * ctx->stride, src, ctx->expert_bytes,
                         cudaMemcpyHostToDevice, ctx->side));
      ctx->staged += ctx->expert_bytes;
    }
    if (tiered && n_miss > 0) {
      CK(cudaEventRecord(ctx->hev, ctx->side));
    } else if (from_file && n_miss > 0) {
      CK(cudaEventRecord(ctx->fev[half], ctx->side));
      ctx->fhalf ^= 1;
    }
    CK(cudaEventRecord(ctx->ev_copy, ctx->side));
    CK(cudaStreamWaitEvent(s, ctx->ev_copy, 0));
    if (n_miss > 0) {
      p.pass = 1;
      CK(launch_gateup(p, 1, gu_max_items(ctx, 1), ctx->n_sm, s, false));
    }
    p.pass = -1;
    CK(launch_down(p, 1, dn_max_items(ctx, 1), ctx->n_sm, s, false));
    if (trace) {
      for (int j = 0; j < k && n_rec < trace_cap; ++j) {
        const volatile int32_t* tr = rec + 1 + 2 * k + 4 * j;
        moe_trace_rec r;
        r.token = static_cast<int32_t>(ctx->step);
        r.layer = l;
        r.k_pos = j;
        r.expert = tr[0];
        r.hit = tr[1];
        r.slot = tr[2];
        r.evicted = tr[3];
        trace[n_rec++] = r;
      }
    }
  }
  if (trace_len) *trace_len = n_rec;
  return MOE_OK;
}

// Device-driven variant of pool_run (moe_set_staging MOE_STAGING_DEVICE): per
// layer, a staging kernel on the side stream, ordered after the router kernel,
// reads the router's miss record and copies the missed experts from the
// mapped host pool into their slots; the host enqueues every layer without
// waiting and fills the trace, if asked for, once the step is done.
// The trace records the device wrote into the mapped host record (device
// staging and the fused step), once the step has finished.
moe_status device_trace(moe_ctx* ctx, int l0, int l1, cudaStream_t s, moe_trace_rec* trace, int trace_cap,
                        int* trace_len) {
  const int k = ctx->cfg.top_k, n_rel = l1 - l0;
  int n_rec = 0;
  if (trace) {
    CK(cudaEventRecord(ctx->ev_route, s));
    moe_status st = wait_event(ctx, ctx->ev_route, "decode step (trace)");
    if (st != MOE_OK) return st;
    for (int rel = 0; rel < n_rel; ++rel) {
      const volatile int32_t* rec = ctx->host_rec + static_cast<size_t>(rel) * (1 + 6 * k);
      for (int j = 0; j < k && n_rec < trace_cap; ++j) {
        const volatile int32_t* tr = rec + 1 + 2 * k + 4 * j;
        moe_trace_rec r;
        r.token = static_cast<int32_t>(ctx->step);
        r.layer = l0 + rel;
        r.k_pos = j;
        r.expert = tr[0];
        r.hit = tr[1];
        r.slot = tr[2];
        r.evicted = tr[3];
        trace[n_rec++] = r;
      }
    }
  }
  if (trace_len) *trace_len = n_rec;
  return MOE_OK;
}

moe_status pool_run_device(moe_ctx* ctx, int l0, int l1, cudaStream_t s, moe_trace_rec* trace, int trace_cap,
                           int* trace_len) {
  const int k = ctx->cfg.top_k, E = ctx->cfg.n_experts;
  const int n_rel = l1 - l0;
  for (int l = l0; l < l1; ++l) {
    const int rel = l - l0;
    KParams p = base_params(ctx, l, rel, rel == 0, rel == n_rel - 1, 1);
    p.h_src = rel == 0 ? nullptr : ctx->hbuf[(rel - 1) & 1];
    p.h_dst = rel == n_rel - 1 ? nullptr : ctx->hbuf[rel & 1];
    CK(launch_router(p, 1, s, false));
    CK(cudaEventRecord(ctx->ev_route, s));
    CK(cudaStreamWaitEvent(ctx->side, ctx->ev_route, 0));
    CK(launch_stage_misses(ctx->host_rec_dev + static_cast<size_t>(rel) * (1 + 6 * k),
                           ctx->pool_dev + static_cast<size_t>(l) * E * ctx->stride, ctx->L[l].slots, ctx->stride,
                           ctx->expert_bytes, E, ctx->n_slots, k, ctx->err_word, ctx->n_sm, ctx->side));
    CK(cudaEventRecord(ctx->ev_copy, ctx->side));
    p.pass = 0;
    CK(launch_gateup(p, 1, gu_max_items(ctx, 1), ctx->n_sm, s, false));
    CK(cudaStreamWaitEvent(s, ctx->ev_copy, 0));
    p.pass = 1;
    CK(launch_gateup(p, 1, gu_max_items(ctx, 1), ctx->n_sm, s, false));
    p.pass = -1;
    CK(launch_down(p, 1, dn_max_items(ctx, 1), ctx->n_sm, s, false));
  }
  return device_trace(ctx, l0, l1, s, trace, trace_cap, trace_len);
}

// Host-pool step in one launch of the clustered kernel: router, slot-cache
// step (in cluster 0), hits from the slots and misses read from the mapped
// pool by the consumers, which also fill the slots.
moe_status pool_run_fused(moe_ctx* ctx, int l0, int l1, cudaStream_t s, moe_trace_rec* trace, int trace_cap,
                          int* trace_len) {
  const moe_status st = cluster_run(ctx, l0, l1, s);
  if (st != MOE_OK) return st;
  return device_trace(ctx, l0, l1, s, trace, trace_cap, trace_len);
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_EINVAL: return "MOE_EINVAL";
    case MOE_ENOMEM: return "MOE_ENOMEM";
    case MOE_ECUDA: return "MOE_ECUDA";
    case MOE_ESTATE: return "MOE_ESTATE";
    case MOE_ETIMEOUT: return "MOE_ETIMEOUT";
    case MOE_EDOMAIN: return "MOE_EDOMAIN";
    case MOE_EIO: return "MOE_EIO";
  }
  return "unknown";
}

const char* moe_last_error(const moe_ctx* ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

int64_t moe_expert_bytes(const moe_config* cfg) {
  if (!cfg_valid(cfg, nullptr)) return 0;
  return expert_bytes_of(cfg->d, cfg->f);
}

int64_t moe_shared_bytes(const moe_config* cfg) {
  if (!cfg_valid(cfg, nullptr)) return 0;
  return expert_bytes_of(cfg->d, cfg->f_shared);
}

moe_status moe_create(const moe_config* cfg, int device, moe_ctx** out) {
  g_create_error.clear();
  if (!out) {
    g_create_error = "out is NULL";
    return MOE_EINVAL;
  }
  *out = nullptr;
  std::string why;
  if (!cfg_valid(cfg, &why)) {
    g_create_error = why;
    return MOE_EINVAL;
  }
  int n_dev = 0;
  if (cudaGetDeviceCount(&n_dev) != cudaSuccess || device < 0 || device >= n_dev) {
    cudaGetLastError();
    g_create_error = "no such CUDA device";
    return MOE_EINVAL;
  }
  moe_ctx* ctx = new moe_ctx();
  ctx->cfg = *cfg;
  ctx->device = device;
  int bail_line = 0;
  auto bail_at = [&](moe_status s, int line) {
    cudaError_t ce = cudaGetLastError();
    char buf[256];
    snprintf(buf, sizeof(buf), "moe_create failed (%s) at moe_api.cu:%d, last CUDA error: %s", moe_status_string(s),
             line, cudaGetErrorString(ce));
    moe_destroy(ctx);
    g_create_error = buf;
    return s;
  };
#define bail(s) bail_at((s), __LINE__)
  (void)bail_line;
  if (cudaSetDevice(device) != cudaSuccess) return bail(MOE_ECUDA);
  cudaDeviceGetAttribute(&ctx->n_sm, cudaDevAttrMultiProcessorCount, device);
  const moe_config& c = ctx->cfg;
  ctx->expert_bytes = expert_bytes_of(c.d, c.f);
  ctx->shared_bytes = expert_bytes_of(c.d, c.f_shared);
  ctx->stride = (ctx->expert_bytes + 255) / 256 * 256;
  ctx->cg = c.f / 64;
  ctx->n_sc = (c.f_shared / 64 + ctx->cg - 1) / ctx->cg;
  ctx->Bd = std::min(c.max_tokens, kMaxDecodeB);
  ctx->L.resize(c.n_layers);
  const size_t Bd = ctx->Bd, P = Bd * c.top_k;
  size_t& nb = ctx->device_bytes;
  auto& o = ctx->owned;
  ctx->hbuf[0] = dalloc<uint16_t>(Bd * c.d, o, nb);
  ctx->hbuf[1] = dalloc<uint16_t>(Bd * c.d, o, nb);
  ctx->x_perm = dalloc<uint16_t>(Bd * c.d, o, nb);
  ctx->xg = dalloc<float>(Bd * (c.d / 64), o, nb);
  ctx->logits = dalloc<long long>(Bd * c.n_experts, o, nb);
  ctx->ids = dalloc<int32_t>(P, o, nb);
  ctx->gates = dalloc<float>(P, o, nb);
  ctx->tok_cnt = dalloc<int32_t>(Bd, o, nb);
  ctx->all_cnt = dalloc<int32_t>(1, o, nb);
  ctx->plan = dalloc<PlanHdr>(1, o, nb);
  ctx->act_expert = dalloc<int32_t>(P, o, nb);
  ctx->act_off = dalloc<int32_t>(P, o, nb);
  ctx->act_cnt = dalloc<int32_t>(P, o, nb);
  ctx->act_pass = dalloc<int32_t>(P, o, nb);
  ctx->pair_tok = dalloc<int32_t>(P, o, nb);
  ctx->pair_gate = dalloc<float>(P, o, nb);
  ctx->pos_of = dalloc<int32_t>(P, o, nb);
  ctx->a_s = dalloc<uint16_t>(Bd * c.f_shared * 2, o, nb);
  ctx->a_r = dalloc<uint16_t>(P * c.f * 2, o, nb);
  ctx->asum_s = dalloc<float>(Bd * (c.f_shared / 8) * 2, o, nb);
  ctx->asum_r = dalloc<float>(P * (c.f / 8) * 2, o, nb);
  ctx->part_s = dalloc<float>(static_cast<size_t>(ctx->n_sc) * Bd * c.d, o, nb);
  ctx->y_r = dalloc<float>(P * c.d, o, nb);
  ctx->row_cnt = dalloc<int32_t>(c.d / 16, o, nb);
  ctx->err_word = dalloc<uint32_t>(1, o, nb);
  ctx->lru_counts = dalloc<long long>(static_cast<size_t>(c.n_layers) * 2, o, nb);
  ctx->dargs = dalloc<DevCallArgs>(1, o, nb);
  ctx->p_n_sc = (c.f_shared / 64 + kPStageGroups - 1) / kPStageGroups;
  const int pparts = ctx->p_n_sc + c.top_k;
  ctx->p_n_counters = c.n_layers * (1 + pparts + c.d / 16 + 1);
  ctx->p_layers = dalloc<PLayer>(c.n_layers, o, nb);
  ctx->p_logits = dalloc<long long>(static_cast<size_t>(c.n_layers) * c.n_experts, o, nb);
  ctx->p_counters = dalloc<unsigned>(ctx->p_n_counters, o, nb);
  ctx->p_exit = dalloc<unsigned>(2, o, nb);
  ctx->p_a_s = dalloc<uint16_t>(static_cast<size_t>(c.f_shared) * 2, o, nb);
  ctx->p_a_r = dalloc<uint16_t>(static_cast<size_t>(c.top_k) * c.f * 2, o, nb);
  ctx->p_asum_s = dalloc<float>(static_cast<size_t>(c.f_shared / 8) * 2, o, nb);
  ctx->p_asum_r = dalloc<float>(static_cast<size_t>(c.top_k) * (c.f / 8) * 2, o, nb);
  ctx->p_part = dalloc<float>(static_cast<size_t>(2) * pparts * c.d, o, nb);
  ctx->p_gates = dalloc<float>(static_cast<size_t>(c.n_layers) * c.top_k, o, nb);
  ctx->c_layers = dalloc<CLayer>(c.n_layers, o, nb);
  ctx->c_ybuf = dalloc<long long>(static_cast<size_t>(3) * c.d, o, nb);
  ctx->c_counters = dalloc<unsigned>(4, o, nb);   // exit counter, abort flag, wait diagnostic, spare
  for (void* ptr : o)
    if (!ptr) return bail(MOE_ENOMEM);
  if (!ctx->hbuf[0] || !ctx->hbuf[1] || !ctx->x_perm || !ctx->dargs || !ctx->y_r || !ctx->part_s || !ctx->a_r)
    return bail(MOE_ENOMEM);
  // zero counters and tables
  if (cudaMemset(ctx->tok_cnt, 0, Bd * 4) != cudaSuccess || cudaMemset(ctx->all_cnt, 0, 4) != cudaSuccess ||
      cudaMemset(ctx->row_cnt, 0, (c.d / 16) * 4) != cudaSuccess || cudaMemset(ctx->err_word, 0, 4) != cudaSuccess ||
      cudaMemset(ctx->plan, 0, sizeof(PlanHdr)) != cudaSuccess ||
      cudaMemset(ctx->lru_counts, 0, static_cast<size_t>(c.n_layers) * 16) != cudaSuccess ||
      cudaMemset(ctx->p_counters, 0, static_cast<size_t>(ctx->p_n_counters) * 4) != cudaSuccess ||
      cudaMemset(ctx->p_exit, 0, 8) != cudaSuccess ||
      cudaMemset(ctx->p_layers, 0, sizeof(PLayer) * c.n_layers) != cudaSuccess ||
      cudaMemset(ctx->c_layers, 0, sizeof(CLayer) * c.n_layers) != cudaSuccess ||
      cudaMemset(ctx->c_ybuf, 0, static_cast<size_t>(3) * c.d * 8) != cudaSuccess ||
      cudaMemset(ctx->c_counters, 0, 16) != cudaSuccess)
    return bail(MOE_ECUDA);
  if (cudaHostAlloc(reinterpret_cast<void**>(&ctx->args_ring), sizeof(DevCallArgs) * kArgRing, cudaHostAllocDefault) !=
      cudaSuccess)
    return bail(MOE_ENOMEM);
  const size_t rec_bytes = static_cast<size_t>(c.n_layers) * (1 + 6 * c.top_k) * sizeof(int32_t);
  if (cudaHostAlloc(reinterpret_cast<void**>(&ctx->host_rec), rec_bytes, cudaHostAllocMapped) != cudaSuccess)
    return bail(MOE_ENOMEM);
  memset(ctx->host_rec, 0, rec_bytes);
  if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&ctx->host_rec_dev), ctx->host_rec, 0) != cudaSuccess)
    return bail(MOE_ECUDA);
  for (int i = 0; i < kArgRing; ++i)
    if (cudaEventCreateWithFlags(&ctx->ring_ev[i], cudaEventDisableTiming) != cudaSuccess) return bail(MOE_ECUDA);
  if (cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->cap, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->ev_route, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->ev_copy, cudaEventDisableTiming) != cudaSuccess)
    return bail(MOE_ECUDA);
  int max_smem = 0;
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (gateup_smem(c.d) > static_cast<size_t>(max_smem) || down_smem(ctx->cg, 8) > static_cast<size_t>(max_smem))
    return bail(MOE_EINVAL);
  if (set_kernel_attrs(max_smem) != cudaSuccess) return bail(MOE_ECUDA);
  // the persistent kernel's shape limits: gate/up tiles of at most 4 chunks of
  // 11 groups, routed down tiles of one chunk, shared down tiles of at most 4
  const int n_cta = ctx->n_sm;
  const int nT = c.d / 16;
  const int tiles_per_cta = (c.f_shared / 8 + n_cta - 1) / n_cta + (c.top_k * (c.f / 8) + n_cta - 1) / n_cta;
  const int stages_per_cta = 2 + (c.n_experts + n_cta - 1) / n_cta + tiles_per_cta + (nT + n_cta - 1) / n_cta +
                             (c.top_k * ((nT + 3) / 4) + n_cta - 1) / n_cta;
  if (n_cta >= 2 && c.d <= 44 * 64 && c.f_shared <= 44 * 64 && c.f <= 11 * 64 &&
      tiles_per_cta <= persistent_max_tiles_per_cta() && stages_per_cta <= persistent_max_tasks() &&
      persistent_smem() + 2048 <= static_cast<size_t>(max_smem)) {   // + the kernel's static shared memory
    int per_sm = 0;
    if (persistent_attrs() == cudaSuccess && persistent_occupancy(&per_sm) == cudaSuccess && per_sm >= 1)
      ctx->p_ok = true;
    cudaGetLastError();
  }
  // the clustered decode kernel: one router row per CTA, at most kCMaxUnits
  // (source, group) units per cluster and layer, its shared memory, a
  // cooperative launch of every resident cluster, and at most 64 clusters (the
  // range of its int64 layer-output sums)
  {
    int n_cl = 0;
    if (c.top_k <= 32 && c.d <= kCMaxD && cluster_smem() <= static_cast<size_t>(max_smem) &&
        cluster_attrs() == cudaSuccess &&
        cluster_max_active(&n_cl) == cudaSuccess && n_cl >= 1 && n_cl <= 64 && c.n_experts <= n_cl * kCCluster &&
        cluster_units_max(c, n_cl) <= cluster_max_units()) {
      // the tagged logits, one replica per cluster of every layer
      ctx->c_tlog = dalloc<unsigned long long>(static_cast<size_t>(c.n_layers) * n_cl * c.n_experts * 2, o, nb);
      if (!ctx->c_tlog) return bail(MOE_ENOMEM);
      ctx->c_plan = dalloc<unsigned long long>(static_cast<size_t>(c.n_layers) * 32, o, nb);
      if (!ctx->c_plan) return bail(MOE_ENOMEM);
      if (cudaMemset(ctx->c_plan, 0, static_cast<size_t>(c.n_layers) * 32 * 8) != cudaSuccess) return bail(MOE_ECUDA);
      if (cudaMemset(ctx->c_tlog, 0, static_cast<size_t>(c.n_layers) * n_cl * c.n_experts * 16) != cudaSuccess)
        return bail(MOE_ECUDA);
      ctx->c_ok = true;
      ctx->c_grid = n_cl * kCCluster;
    }
    cudaGetLastError();
  }
  // the tcgen05 prefill: 128-row weight tiles of the down projection, one router
  // CTA column of 128 experts, and its shared memory
  if (c.d % 128 == 0 && c.n_experts <= 128 && pf_gemm_smem(kPfTileN) <= static_cast<size_t>(max_smem) &&
      pf_gemm_smem(kPfTileNSmall) <= static_cast<size_t>(max_smem) &&
      pf_gemm_smem(kPfTileNBig) <= static_cast<size_t>(max_smem)) {
    if (pf_set_attrs() == cudaSuccess) ctx->pf_ok = true;
    cudaGetLastError();
  }
  // the small-batch GEMVs run on the tcgen05 path's routing and grouping
  if (ctx->pf_ok && sg_shape_ok(c.d, c.f, c.f_shared) && sg_smem() <= static_cast<size_t>(max_smem)) {
    if (sg_set_attrs() == cudaSuccess) ctx->sg_ok = true;
    cudaGetLastError();
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(MOE_ECUDA);
  *out = ctx;
  return MOE_OK;
#undef bail
}

void moe_destroy(moe_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  for (auto& kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& kv : ctx->pf_graphs) cudaGraphExecDestroy(kv.second);
  for (auto& Ls : ctx->L) {
    cudaFree(Ls.router_w);
    cudaFree(Ls.router_stats);
    cudaFree(Ls.shared);
    cudaFree(Ls.experts);
    cudaFree(Ls.slots);
    cudaFree(Ls.slot_of_expert);
    cudaFree(Ls.expert_of_slot);
    cudaFree(Ls.last_use);
    cudaFree(Ls.use_count);
  }
  for (void* p : ctx->owned) cudaFree(p);
  for (void* p : ctx->pf_owned) cudaFree(p);
  if (ctx->pool) cudaFreeHost(ctx->pool);
  if (ctx->fpool) file_pool_destroy(ctx->fpool);
  if (ctx->file_fd >= 0) ::close(ctx->file_fd);
  if (ctx->file_rfd >= 0) ::close(ctx->file_rfd);
  if (ctx->fstage) cudaFreeHost(ctx->fstage);
  if (ctx->hcache) cudaFreeHost(ctx->hcache);
  if (ctx->hev) cudaEventDestroy(ctx->hev);
  if (ctx->pf_cnt_host) cudaFreeHost(ctx->pf_cnt_host);
  if (ctx->pf_ev_cnt) cudaEventDestroy(ctx->pf_ev_cnt);
  if (ctx->pf_ev_read) cudaEventDestroy(ctx->pf_ev_read);
  for (auto& e : ctx->fev)
    if (e) cudaEventDestroy(e);
  if (ctx->args_ring) cudaFreeHost(ctx->args_ring);
  if (ctx->host_rec) cudaFreeHost(ctx->host_rec);
  for (auto& e : ctx->ring_ev)
    if (e) cudaEventDestroy(e);
  for (auto& e : ctx->prof_ev) cudaEventDestroy(e);
  if (ctx->ev_route) cudaEventDestroy(ctx->ev_route);
  if (ctx->ev_copy) cudaEventDestroy(ctx->ev_copy);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  if (ctx->cap) cudaStreamDestroy(ctx->cap);
  delete ctx;
}

moe_status moe_init_layer(moe_ctx* ctx, int layer, const uint16_t* router_w, const moe_expert_weights* experts,
                          const moe_expert_weights* shared, int residency) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  const moe_config& c = ctx->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(ctx, MOE_EINVAL, "layer %d out of range", layer);
  if (residency != MOE_RESIDENT_HBM && residency != MOE_HOST_POOL && residency != MOE_FILE_POOL)
    return fail(ctx, MOE_EINVAL, "unknown residency %d", residency);
  if (residency == MOE_FILE_POOL && ctx->file_fd < 0)
    return fail(ctx, MOE_ESTATE, "MOE_FILE_POOL needs moe_set_expert_file first");
  if (ctx->residency >= 0 && residency != ctx->residency)
    return fail(ctx, MOE_EINVAL, "all layers of a context must use the same residency");
  if (!router_w || !experts || !shared) return fail(ctx, MOE_EINVAL, "NULL weights");
  for (int e = 0; e <= c.n_experts; ++e) {
    const moe_expert_weights& w = e < c.n_experts ? experts[e] : *shared;
    if (!w.gate_q || !w.gate_sb || !w.up_q || !w.up_sb || !w.down_q || !w.down_sb)
      return fail(ctx, MOE_EINVAL, "NULL projection pointer (expert %d)", e);
  }
  CK(cudaSetDevice(ctx->device));
  LayerStore& Ls = ctx->L[layer];
  const bool pool = residency == MOE_HOST_POOL || residency == MOE_FILE_POOL;
  const bool file = residency == MOE_FILE_POOL;
  // memory budget before allocating
  size_t free_b = 0;
  CK(free_device_bytes(ctx, &free_b));
  const size_t fs_can = static_cast<size_t>(c.f_shared) * c.d * 27 / 16 + 64;
  size_t need = static_cast<size_t>(c.n_experts) * c.d * 2 + ctx->shared_bytes + 3 * fs_can;
  need += static_cast<size_t>(c.n_experts) * ctx->stride;  // resident experts or the staging buffer
  if (!Ls.ready && need + (256u << 20) > free_b)
    return fail(ctx, MOE_ENOMEM, "layer needs %zu bytes, %zu free", need, free_b);
  if (pool && !file && !ctx->pool) {
    const size_t pb = static_cast<size_t>(c.n_layers) * c.n_experts * ctx->stride;
    if (cudaHostAlloc(reinterpret_cast<void**>(&ctx->pool), pb, cudaHostAllocMapped) != cudaSuccess) {
      ctx->pool = nullptr;
      cudaGetLastError();
      return fail(ctx, MOE_ENOMEM, "pinned host pool of %zu bytes", pb);
    }
    ctx->pool_bytes = pb;
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, ctx->pool, 0) == cudaSuccess) ctx->pool_dev = static_cast<const uint8_t*>(dp);
    cudaGetLastError();
  }
  ctx->residency = residency;
  if (!Ls.router_w) CK(cudaMalloc(&Ls.router_w, static_cast<size_t>(c.n_experts) * c.d * 2));
  if (!Ls.shared) CK(cudaMalloc(&Ls.shared, ctx->shared_bytes));
  if (!pool && !Ls.experts) CK(cudaMalloc(&Ls.experts, static_cast<size_t>(c.n_experts) * ctx->stride));
  if (pool && !Ls.slot_of_expert) CK(cudaMalloc(&Ls.slot_of_expert, static_cast<size_t>(c.n_experts) * 4));
  CK(cudaMemcpy(Ls.router_w, router_w, static_cast<size_t>(c.n_experts) * c.d * 2, cudaMemcpyDefault));
  if (!Ls.router_stats) CK(cudaMalloc(&Ls.router_stats, static_cast<size_t>(c.n_experts) * 2 * sizeof(float)));
  CK(launch_pf_row_stats(Ls.router_w, c.n_experts, c.d, Ls.router_stats, Ls.router_stats + c.n_experts, nullptr));

  // canonical staging buffers (largest f), then repack on the device
  const int fmax = std::max(c.f, c.f_shared);
  const size_t q_b = static_cast<size_t>(fmax) * c.d / 2;
  const size_t sb_b = static_cast<size_t>(fmax) * (c.d / 64) * 4;
  uint8_t* can = nullptr;
  CK(cudaMalloc(&can, 3 * q_b + 3 * sb_b));
  uint8_t* tmp = nullptr;
  if (pool) {
    cudaError_t e = cudaMalloc(&tmp, static_cast<size_t>(c.n_experts) * ctx->stride);
    if (e != cudaSuccess) {
      cudaFree(can);
      return fail(ctx, MOE_ECUDA, "staging buffer: %s", cudaGetErrorString(e));
    }
  }
  auto stage = [&](const moe_expert_weights& w, int f, uint8_t* dst) -> cudaError_t {
    const size_t gq = static_cast<size_t>(f) * c.d / 2, gsb = static_cast<size_t>(f) * (c.d / 64) * 4;
    const size_t dsb = static_cast<size_t>(c.d) * (f / 64) * 4;
    uint8_t* p_gq = can;
    uint8_t* p_uq = can + q_b;
    uint8_t* p_dq = can + 2 * q_b;
    uint8_t* p_gs = can + 3 * q_b;
    uint8_t* p_us = p_gs + sb_b;
    uint8_t* p_ds = p_us + sb_b;
    cudaError_t e;
    if ((e = cudaMemcpy(p_gq, w.gate_q, gq, cudaMemcpyDefault)) != cudaSuccess) return e;
    if ((e = cudaMemcpy(p_uq, w.up_q, gq, cudaMemcpyDefault)) != cudaSuccess) return e;
    if ((e = cudaMemcpy(p_dq, w.down_q, gq, cudaMemcpyDefault)) != cudaSuccess) return e;
    if ((e = cudaMemcpy(p_gs, w.gate_sb, gsb, cudaMemcpyDefault)) != cudaSuccess) return e;
    if ((e = cudaMemcpy(p_us, w.up_sb, gsb, cudaMemcpyDefault)) != cudaSuccess) return e;
    if ((e = cudaMemcpy(p_ds, w.down_sb, dsb, cudaMemcpyDefault)) != cudaSuccess) return e;
    return launch_repack(p_gq, reinterpret_cast<uint16_t*>(p_gs), p_uq, reinterpret_cast<uint16_t*>(p_us), p_dq,
                         reinterpret_cast<uint16_t*>(p_ds), c.d, f, dst, nullptr);
  };
  cudaError_t e = stage(*shared, c.f_shared, Ls.shared);
  for (int ex = 0; ex < c.n_experts && e == cudaSuccess; ++ex) {
    uint8_t* dst = (pool ? tmp : Ls.experts) + static_cast<size_t>(ex) * ctx->stride;
    e = stage(experts[ex], c.f, dst);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess && pool && !file)
    e = cudaMemcpy(ctx->pool + static_cast<size_t>(layer) * c.n_experts * ctx->stride, tmp,
                   static_cast<size_t>(c.n_experts) * ctx->stride, cudaMemcpyDeviceToHost);
  int io_err = 0;
  if (e == cudaSuccess && file) {
    // the layer's records, through a host bounce buffer, written in parallel chunks
    std::vector<uint8_t> host;
    try {
      host.resize(static_cast<size_t>(c.n_experts) * ctx->stride);
    } catch (const std::bad_alloc&) {
      cudaFree(can);
      cudaFree(tmp);
      return fail(ctx, MOE_ENOMEM, "init_layer %d: host bounce buffer", layer);
    }
    e = cudaMemcpy(host.data(), tmp, host.size(), cudaMemcpyDeviceToHost);
    for (int ex = 0; ex < c.n_experts && e == cudaSuccess && io_err == 0; ++ex)
      io_err = file_pool_transfer(ctx->fpool, ctx->file_fd, true,
                                  (static_cast<uint64_t>(layer) * c.n_experts + ex) * ctx->file_stride,
                                  host.data() + static_cast<size_t>(ex) * ctx->stride, ctx->expert_bytes,
                                  ctx->file_chunk);
  }
  cudaFree(can);
  if (tmp) cudaFree(tmp);
  if (e != cudaSuccess) return fail(ctx, MOE_ECUDA, "init_layer %d: %s", layer, cudaGetErrorString(e));
  if (io_err != 0) return fail(ctx, MOE_EIO, "init_layer %d: expert file write: %s", layer, strerror(io_err));
  if (pool && ctx->n_slots > 0 && Ls.slot_of_expert) CK(cudaMemset(Ls.slot_of_expert, 0xFF, c.n_experts * 4));
  PLayer pl{Ls.router_w, Ls.shared, Ls.experts};
  CK(cudaMemcpy(ctx->p_layers + layer, &pl, sizeof(PLayer), cudaMemcpyHostToDevice));
  if (ctx->c_ok && !pool) {
    CLayer cl{};
    const size_t gu_s = static_cast<size_t>(c.f_shared / 8) * (c.d / 64) * kGroupBytes;
    const size_t gu_r = static_cast<size_t>(c.f / 8) * (c.d / 64) * kGroupBytes;
    if (!encode_down(&cl.dn_shared, Ls.shared + gu_s, c.f_shared / 64, c.d / 16, 1, 0) ||
        !encode_down(&cl.dn_routed, Ls.experts + gu_r, c.f / 64, c.d / 16, c.n_experts, ctx->stride))
      return fail(ctx, MOE_ECUDA, "init_layer %d: cuTensorMapEncodeTiled failed for the down regions", layer);
    cl.router_w = Ls.router_w;
    cl.shared = Ls.shared;
    cl.experts = Ls.experts;
    CK(cudaMemcpy(ctx->c_layers + layer, &cl, sizeof(CLayer), cudaMemcpyHostToDevice));
  }
  Ls.ready = true;
  if (pool) return cluster_pool_layer(ctx, layer);
  return MOE_OK;
}

moe_status moe_set_slots(moe_ctx* ctx, int n_slots) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  const moe_config& c = ctx->cfg;
  if (ctx->residency != MOE_HOST_POOL && ctx->residency != MOE_FILE_POOL)
    return fail(ctx, MOE_ESTATE, "slots need a host-pool or file-pool context");
  if (n_slots < c.top_k || n_slots > c.n_experts)
    return fail(ctx, MOE_EINVAL, "n_slots %d outside [top_k=%d, n_experts=%d]", n_slots, c.top_k, c.n_experts);
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());
  const size_t per_layer = static_cast<size_t>(n_slots) * ctx->stride + static_cast<size_t>(n_slots) * 12;
  const size_t need = per_layer * c.n_layers;
  size_t have = 0;
  for (auto& Ls : ctx->L)
    if (Ls.slots) have += static_cast<size_t>(ctx->n_slots) * ctx->stride + static_cast<size_t>(ctx->n_slots) * 12;
  size_t free_b = 0;
  CK(free_device_bytes(ctx, &free_b));
  if (need > free_b + have || need + (256u << 20) > free_b + have)
    return fail(ctx, MOE_ENOMEM, "%d slots x %d layers need %zu bytes, %zu available", n_slots, c.n_layers, need,
                free_b + have);
  for (auto& Ls : ctx->L) {
    cudaFree(Ls.slots);
    cudaFree(Ls.expert_of_slot);
    cudaFree(Ls.last_use);
    Ls.slots = nullptr;
    Ls.expert_of_slot = nullptr;
    Ls.last_use = nullptr;
  }
  ctx->n_slots = 0;
  for (auto& Ls : ctx->L) {
    CK(cudaMalloc(&Ls.slots, static_cast<size_t>(n_slots) * ctx->stride));
    CK(cudaMalloc(&Ls.expert_of_slot, static_cast<size_t>(n_slots) * 4));
    CK(cudaMalloc(&Ls.last_use, static_cast<size_t>(n_slots) * 8));
    if (!Ls.slot_of_expert) CK(cudaMalloc(&Ls.slot_of_expert, static_cast<size_t>(c.n_experts) * 4));
    if (!Ls.use_count) CK(cudaMalloc(&Ls.use_count, static_cast<size_t>(c.n_experts) * 8));
  }
  ctx->n_slots = n_slots;
  for (int l = 0; l < c.n_layers; ++l) {
    const moe_status st = cluster_pool_layer(ctx, l);
    if (st != MOE_OK) return st;
  }
  return moe_reset_cache(ctx);
}

moe_status moe_set_cache_policy(moe_ctx* ctx, int policy) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (policy != MOE_CACHE_LRU && policy != MOE_CACHE_LFU) return fail(ctx, MOE_EINVAL, "unknown policy %d", policy);
  if (ctx->residency != MOE_HOST_POOL && ctx->residency != MOE_FILE_POOL)
    return fail(ctx, MOE_ESTATE, "cache policy needs a host-pool or file-pool context");
  ctx->policy = policy;
  return moe_reset_cache(ctx);
}

moe_status moe_set_expert_file(moe_ctx* ctx, const char* path, int n_threads, uint64_t chunk_bytes, int flags) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (!path || n_threads < 1 || n_threads > 64 || chunk_bytes % 4096 != 0 || (flags & ~MOE_FILE_DIRECT))
    return fail(ctx, MOE_EINVAL, "bad expert file arguments");
  if (ctx->residency >= 0 || ctx->file_fd >= 0)
    return fail(ctx, MOE_EINVAL, "the expert file must be set before any layer is initialised, once");
  const int fd = ::open(path, O_RDWR | O_CREAT | O_TRUNC, 0644);
  if (fd < 0) return fail(ctx, MOE_EINVAL, "cannot create expert file %s: %s", path, strerror(errno));
  int rfd = -1;
  const size_t fstride = (ctx->expert_bytes + 4095) / 4096 * 4096;
  if (flags & MOE_FILE_DIRECT) {
    // whole records are read: the file spans every record in full (sparse tails)
    rfd = ::open(path, O_RDONLY | O_DIRECT);
    const off_t full = static_cast<off_t>(ctx->cfg.n_layers) * ctx->cfg.n_experts * static_cast<off_t>(fstride);
    if (rfd < 0 || ::ftruncate(fd, full) != 0) {
      const int e = errno;
      if (rfd >= 0) ::close(rfd);
      ::close(fd);
      return fail(ctx, MOE_EINVAL, "O_DIRECT reads of %s refused: %s", path, strerror(e));
    }
  }
  uint8_t* stage = nullptr;
  if (cudaHostAlloc(reinterpret_cast<void**>(&stage), 2 * static_cast<size_t>(ctx->cfg.top_k) * fstride,
                    cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    ::close(fd);
    if (rfd >= 0) ::close(rfd);
    return fail(ctx, MOE_ENOMEM, "pinned staging for the expert file");
  }
  for (auto& ev : ctx->fev)
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaFreeHost(stage);
      ::close(fd);
      if (rfd >= 0) ::close(rfd);
      return fail(ctx, MOE_ECUDA, "events for the expert file");
    }
  ctx->file_fd = fd;
  ctx->file_rfd = rfd;
  ctx->file_stride = fstride;
  ctx->fstage = stage;
  ctx->file_chunk = chunk_bytes == 0 ? (512u << 10) : chunk_bytes;
  ctx->fpool = file_pool_create(n_threads);
  if (!ctx->fpool) {
    ::close(ctx->file_fd);
    if (ctx->file_rfd >= 0) ::close(ctx->file_rfd);
    ctx->file_fd = ctx->file_rfd = -1;
    cudaFreeHost(ctx->fstage);
    ctx->fstage = nullptr;
    return fail(ctx, MOE_ENOMEM, "expert file reader threads");
  }
  return MOE_OK;
}

moe_status moe_set_staging(moe_ctx* ctx, int mode) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (mode != MOE_STAGING_HOST && mode != MOE_STAGING_DEVICE && mode != MOE_STAGING_FUSED)
    return fail(ctx, MOE_EINVAL, "unknown staging mode %d", mode);
  if (ctx->residency != MOE_HOST_POOL) return fail(ctx, MOE_ESTATE, "staging modes apply to host-pool contexts");
  if (mode != MOE_STAGING_HOST && !ctx->pool_dev)
    return fail(ctx, MOE_ESTATE, "the host pool is not mapped into the device address space");
  if (mode == MOE_STAGING_FUSED && !ctx->c_ok)
    return fail(ctx, MOE_ESTATE, "the clustered decode kernel is unavailable for this configuration or device");
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());
  ctx->stage_device = mode == MOE_STAGING_DEVICE;
  ctx->stage_fused = mode == MOE_STAGING_FUSED;
  return moe_reset_cache(ctx);
}

moe_status moe_set_file_cache(moe_ctx* ctx, int n_host) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (ctx->file_fd < 0) return fail(ctx, MOE_ESTATE, "the host tier needs an expert file (moe_set_expert_file)");
  const moe_config& c = ctx->cfg;
  if (n_host != 0 && (n_host < c.top_k || n_host > c.n_experts))
    return fail(ctx, MOE_EINVAL, "host records per layer %d outside {0} + [top_k=%d, n_experts=%d]", n_host, c.top_k,
                c.n_experts);
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());   // no copy out of the old records is in flight
  if (ctx->hcache) cudaFreeHost(ctx->hcache);
  ctx->hcache = nullptr;
  ctx->n_host = 0;
  if (n_host > 0) {
    const size_t bytes = static_cast<size_t>(c.n_layers) * n_host * ctx->file_stride;
    if (cudaHostAlloc(reinterpret_cast<void**>(&ctx->hcache), bytes, cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      ctx->hcache = nullptr;
      return fail(ctx, MOE_ENOMEM, "pinned host tier (%zu bytes)", bytes);
    }
    if (!ctx->hev) CK(cudaEventCreateWithFlags(&ctx->hev, cudaEventDisableTiming));
    ctx->n_host = n_host;
  }
  ctx->h_expert_of_slot.assign(static_cast<size_t>(c.n_layers) * n_host, -1);
  ctx->h_last_use.assign(static_cast<size_t>(c.n_layers) * n_host, -1);
  ctx->h_slot_of_expert.assign(static_cast<size_t>(c.n_layers) * c.n_experts, -1);
  ctx->h_touched.assign(static_cast<size_t>(n_host), 0);
  host_tier_clear(ctx);
  return MOE_OK;
}

moe_status moe_reset_cache(moe_ctx* ctx) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());
  const moe_config& c = ctx->cfg;
  for (auto& Ls : ctx->L) {
    if (Ls.slot_of_expert) CK(cudaMemset(Ls.slot_of_expert, 0xFF, static_cast<size_t>(c.n_experts) * 4));
    if (Ls.expert_of_slot) CK(cudaMemset(Ls.expert_of_slot, 0xFF, static_cast<size_t>(ctx->n_slots) * 4));
    if (Ls.last_use) CK(cudaMemset(Ls.last_use, 0xFF, static_cast<size_t>(ctx->n_slots) * 8));
    if (Ls.use_count) CK(cudaMemset(Ls.use_count, 0, static_cast<size_t>(c.n_experts) * 8));
  }
  CK(cudaMemset(ctx->lru_counts, 0, static_cast<size_t>(c.n_layers) * 16));
  ctx->step = 0;
  ctx->steps = 0;
  ctx->staged = 0;
  host_tier_clear(ctx);
  return MOE_OK;
}

namespace {
moe_status pf_run(moe_ctx* ctx, const void* h, int T, int l0, int l1, const float* logit_bias, void* h_out,
                  float* y_last, cudaStream_t s);
}  // namespace

moe_status moe_decode_step(moe_ctx* ctx, const void* h_in, int B, int layer_begin, int layer_end,
                           const float* logit_bias, void* h_out, float* y_last, moe_trace_rec* trace, int trace_cap,
                           int* trace_len, void* stream) {
  moe_status st = check_ready(ctx, layer_begin, layer_end);
  if (st != MOE_OK) return st;
  if (!h_in || !h_out) return fail(ctx, MOE_EINVAL, "NULL h_in / h_out");
  const bool pool = ctx->residency == MOE_HOST_POOL || ctx->residency == MOE_FILE_POOL;
  if (B < 1 || B > ctx->Bd) return fail(ctx, MOE_EINVAL, "B=%d outside [1, %d]", B, ctx->Bd);
  if (pool && B != 1) return fail(ctx, MOE_EINVAL, "host-pool decode takes one token per call");
  if (pool && ctx->n_slots < ctx->cfg.top_k) return fail(ctx, MOE_ESTATE, "slots are not set");
  if (trace && trace_cap < 0) return fail(ctx, MOE_EINVAL, "negative trace_cap");
  if (trace_len) *trace_len = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(cudaSetDevice(ctx->device));
  st = put_args(ctx, make_args(ctx, h_in, h_out, y_last, logit_bias, B, B, 0), s);
  if (st != MOE_OK) return st;
  if (pool) {
    st = ctx->stage_fused    ? pool_run_fused(ctx, layer_begin, layer_end, s, trace, trace_cap, trace_len)
         : ctx->stage_device ? pool_run_device(ctx, layer_begin, layer_end, s, trace, trace_cap, trace_len)
                             : pool_run(ctx, layer_begin, layer_end, s, trace, trace_cap, trace_len);
    ++ctx->step;
    ++ctx->steps;
    return st;
  }
  if (B == 1 && ctx->use_persistent) {
    if (ctx->c_ok && ctx->use_cluster) return cluster_run(ctx, layer_begin, layer_end, s);
    if (ctx->p_ok) return persistent_run(ctx, layer_begin, layer_end, s);
  }
  // a few tokens: one clustered-kernel launch per token beats the grouped
  // path's per-layer launches (measured: 2 and 4 tokens at 1,150 and 1,787
  // tok/s grouped against about 1,960 one at a time; 5 tokens grouped 2,090)
  if (B <= kClusterLoopMaxB && ctx->use_persistent && ctx->c_ok && ctx->use_cluster && ctx->c_loop) {
    const int d = ctx->cfg.d;
    for (int t = 0; t < B; ++t) {
      st = put_args(ctx,
                    make_args(ctx, static_cast<const uint16_t*>(h_in) + static_cast<size_t>(t) * d,
                              static_cast<uint16_t*>(h_out) + static_cast<size_t>(t) * d,
                              y_last ? y_last + static_cast<size_t>(t) * d : nullptr, logit_bias, 1, B, t),
                    s);
      if (st != MOE_OK) return st;
      st = cluster_run(ctx, layer_begin, layer_end, s);
      if (st != MOE_OK) return st;
    }
    return MOE_OK;
  }
  // the grouped path: with the small-batch GEMVs for every batch of two tokens or more, else
  // (tcgen05 GEMMs) from about 16 tokens on (measured crossover with the per-layer GEMVs)
  const bool grouped = ctx->pf_ok && ctx->use_pf && B >= 2 && ((ctx->sg_ok && ctx->use_sg) || B >= kPfMinDecodeB);
  if (grouped) return pf_run(ctx, h_in, B, layer_begin, layer_end, logit_bias, h_out, y_last, s);
  return resident_run(ctx, B, layer_begin, layer_end, s);
}

namespace {

// 2-D tensor map over a row-major fp16 matrix [rows][K]: boxes of 64 columns x
// box_rows rows with the 128-byte swizzle the GEMM's operand tiles use.
bool encode_rows(CUtensorMap* m, void* base, int K, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scratch of the tcgen05 prefill for max_tokens tokens (made once).
moe_status pf_alloc(moe_ctx* ctx) {
  if (ctx->pf_ready) return MOE_OK;
  const moe_config& c = ctx->cfg;
  const size_t T = c.max_tokens, P = T * c.top_k;
  size_t nb = 0;
  auto& o = ctx->pf_owned;
  ctx->pf_xbf = dalloc<uint16_t>(T * c.d, o, nb);
  ctx->pf_x16 = dalloc<uint16_t>(T * c.d, o, nb);
  ctx->pf_xp = dalloc<uint16_t>(P * c.d, o, nb);
  ctx->pf_ar = dalloc<uint16_t>(P * c.f, o, nb);
  ctx->pf_as = dalloc<uint16_t>(T * c.f_shared, o, nb);
  ctx->pf_h[0] = dalloc<uint16_t>(T * c.d, o, nb);
  ctx->pf_h[1] = dalloc<uint16_t>(T * c.d, o, nb);
  ctx->pf_ids = dalloc<int32_t>(P, o, nb);
  ctx->pf_gates = dalloc<float>(P, o, nb);
  ctx->pf_cnt = dalloc<int32_t>(c.n_experts, o, nb);
  ctx->pf_rowpair = dalloc<int32_t>(P, o, nb);
  ctx->pf_items = dalloc<int32_t>(3 * (P / kPfTileNSmall + c.n_experts + 1), o, nb);
  ctx->pf_nitems = dalloc<int32_t>(1, o, nb);
  ctx->pf_ytok = dalloc<float>(P * c.d, o, nb);
  ctx->pf_approx = dalloc<float>(T * c.n_experts, o, nb);
  ctx->pf_xn2 = dalloc<float>(T, o, nb);
  ctx->pf_xmax = dalloc<float>(T, o, nb);
  ctx->pf_ys = dalloc<float>(T * c.d, o, nb);
  if (ctx->sg_ok) {
    const size_t rows = std::min<size_t>(T, kSgMaxT);
    ctx->sg_xv = dalloc<uint16_t>(rows * c.d, o, nb);
    ctx->sg_xg = dalloc<float>(rows * (c.d / 64), o, nb);
    if (!ctx->sg_xv || !ctx->sg_xg) return fail(ctx, MOE_ENOMEM, "small-batch scratch does not fit");
  }
  if (!ctx->pf_xbf || !ctx->pf_x16 || !ctx->pf_xp || !ctx->pf_ar || !ctx->pf_as || !ctx->pf_h[0] || !ctx->pf_h[1] ||
      !ctx->pf_ids || !ctx->pf_gates || !ctx->pf_cnt || !ctx->pf_rowpair || !ctx->pf_items || !ctx->pf_nitems ||
      !ctx->pf_ytok || !ctx->pf_approx || !ctx->pf_xn2 || !ctx->pf_xmax || !ctx->pf_ys)
    return fail(ctx, MOE_ENOMEM, "prefill scratch (%zu bytes for %zu tokens) does not fit", nb, T);
  for (int i = 0; i < 3; ++i) {
    const int br = i == 0 ? kPfTileN : i == 1 ? kPfTileNSmall : kPfTileNBig;
    if (!encode_rows(&ctx->pf_map_xp[i], ctx->pf_xp, c.d, static_cast<long long>(P), br) ||
        !encode_rows(&ctx->pf_map_x16[i], ctx->pf_x16, c.d, static_cast<long long>(T), br) ||
        !encode_rows(&ctx->pf_map_ar[i], ctx->pf_ar, c.f, static_cast<long long>(P), br) ||
        !encode_rows(&ctx->pf_map_as[i], ctx->pf_as, c.f_shared, static_cast<long long>(T), br))
      return fail(ctx, MOE_ECUDA, "cuTensorMapEncodeTiled failed for the prefill operands");
  }
  // the router's approximate logits accumulate into zeros (each pass zeroes what it reads)
  CK(cudaMemset(ctx->pf_approx, 0, T * c.n_experts * sizeof(float)));
  ctx->device_bytes += nb;
  ctx->pf_ready = true;
  return MOE_OK;
}

// One layer of the batched prefill: route, group by expert, four grouped GEMMs.
// Token tiles of 32 rows when the experts' groups are small (a few rows each),
// else 128 for the routed experts.  The shared expert (every token) takes
// 256-row tiles from 256 tokens on: each dequantised weight tile then serves
// twice the tokens.  (256-row tiles for the routed experts measured 4.5 %
// slower at T = 4096: one CTA per SM leaves no second CTA to overlap the
// epilogue, and the groups are uneven.)
int pf_tile_routed(const moe_config& c, int T) {
  return static_cast<long long>(T) * c.top_k <= 16ll * c.n_experts ? kPfTileNSmall : kPfTileN;
}
int pf_tile_shared(int T) { return T <= 48 ? kPfTileNSmall : T >= kPfTileNBig ? kPfTileNBig : kPfTileN; }
int pf_map_index(int tile) { return tile == kPfTileN ? 0 : tile == kPfTileNSmall ? 1 : 2; }

// One prefill layer, first part: RMS norm, router, the expert-ordered pair list
// and the gathered token rows (pf_cnt then holds the pairs per expert).
moe_status pf_layer_route(moe_ctx* ctx, int l, int rel, const uint16_t* hin, int T, const float* bias,
                          cudaStream_t s, bool small = false) {
  const moe_config& c = ctx->cfg;
  const LayerStore& L = ctx->L[l];
  const int d = c.d, E = c.n_experts, k = c.top_k, P = T * k;
  const bool dbg = rel < ctx->dbg_layers;
  const size_t xo = static_cast<size_t>(rel) * T;
  PROF(4, s);
  CK(launch_pf_prep(hin, T, d, c.prenorm, c.norm_eps, ctx->pf_xbf, ctx->pf_x16,
                    dbg && ctx->dbg_x ? ctx->dbg_x + xo * d : nullptr, ctx->pf_xn2, ctx->pf_xmax,
                    small ? ctx->sg_xv : nullptr, small ? ctx->sg_xg : nullptr, ctx->err_word, s));
  CK(launch_pf_router(ctx->pf_xbf, L.router_w, bias ? bias + xo * E : nullptr, T, d, E, k, ctx->pf_approx,
                      ctx->pf_xn2, L.router_stats, ctx->pf_xmax, L.router_stats + E, ctx->pf_ids, ctx->pf_gates, dbg && ctx->dbg_ids ? ctx->dbg_ids + xo * k : nullptr,
                      dbg && ctx->dbg_gates ? ctx->dbg_gates + xo * k : nullptr,
                      dbg && ctx->dbg_logits ? ctx->dbg_logits + xo * E : nullptr, ctx->err_word, ctx->n_sm, s));
  CK(launch_pf_plan(ctx->pf_ids, P, E, small ? kSgMaxT : pf_tile_routed(c, T), ctx->pf_cnt, ctx->pf_rowpair,
                    ctx->pf_items, ctx->pf_nitems, s));
  if (!small) CK(launch_pf_gather(ctx->pf_x16, ctx->pf_rowpair, P, d, k, ctx->pf_xp, s));
  PROF(-1, s);
  return MOE_OK;
}

PfGemm pf_gemm_base(moe_ctx* ctx) {
  PfGemm g{};
  g.tl = nullptr;
  g.d = ctx->cfg.d;
  g.k = ctx->cfg.top_k;
  g.gelu = ctx->cfg.gelu_variant;
  g.err = ctx->err_word;
  return g;
}

// Shared expert gate/up over every token (needs no routed expert).
moe_status pf_layer_shared_gu(moe_ctx* ctx, int l, int rel, int T, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  const int ns = pf_tile_shared(T), ms = pf_map_index(ns);
  const int t_items = (T + ns - 1) / ns;
  PfGemm b = pf_gemm_base(ctx);
  b.w = ctx->L[l].shared;
  b.nG = c.d / 64;
  b.n_items = t_items;
  b.rows_total = T;
  b.mode = PF_GU;
  b.out16 = ctx->pf_as;
  b.f_out = c.f_shared;
  if (ctx->pf_timeline && rel == 0) b.tl = ctx->pf_timeline + 16;
  CK(launch_pf_gemm(ns, ctx->pf_map_x16[ms], b, c.f_shared / 64, t_items, s));
  return MOE_OK;
}

// The rest of the layer: routed gate/up and down over `experts` (expert e's
// device record at e * stride), shared down, combine (+ residual).
moe_status pf_layer_rest(moe_ctx* ctx, int l, int rel, int n_rel, const uint16_t* hin, uint16_t* hout, int T,
                         float* y_last, const uint8_t* experts, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  const LayerStore& L = ctx->L[l];
  const int d = c.d, E = c.n_experts, k = c.top_k, P = T * k;
  const bool dbg = rel < ctx->dbg_layers;
  const size_t xo = static_cast<size_t>(rel) * T;
  const int nr = pf_tile_routed(c, T), ns = pf_tile_shared(T);
  const int mr = pf_map_index(nr), ms = pf_map_index(ns);
  const size_t gu_r = static_cast<size_t>(c.f / 8) * (d / 64) * kGroupBytes;
  const size_t gu_s = static_cast<size_t>(c.f_shared / 8) * (d / 64) * kGroupBytes;
  const int max_items = P / nr + E + 1;
  const int t_items = (T + ns - 1) / ns;
  // routed gate/up: expert-ordered rows -> GELU(gate) * up, fp16 [P][f]
  PfGemm a = pf_gemm_base(ctx);
  a.w = experts;
  a.w_stride = ctx->stride;
  a.nG = d / 64;
  a.items = ctx->pf_items;
  a.n_items_dev = ctx->pf_nitems;
  a.mode = PF_GU;
  a.out16 = ctx->pf_ar;
  a.f_out = c.f;
  if (ctx->pf_timeline && rel == 0) a.tl = ctx->pf_timeline;
  CK(launch_pf_gemm(nr, ctx->pf_map_xp[mr], a, c.f / 64, max_items, s));
  // routed down: per pair, fp32 [T*k][d]
  PfGemm r = pf_gemm_base(ctx);
  r.w = experts + gu_r;
  r.w_stride = ctx->stride;
  r.nG = c.f / 64;
  r.items = ctx->pf_items;
  r.n_items_dev = ctx->pf_nitems;
  r.mode = PF_DN_ROUTED;
  r.out32 = ctx->pf_ytok;
  r.pair_of_row = ctx->pf_rowpair;
  if (ctx->pf_timeline && rel == 0) r.tl = ctx->pf_timeline + 32;
  CK(launch_pf_gemm(nr, ctx->pf_map_ar[mr], r, d / 128, max_items, s));
  // shared down, then the combine: shared + routed in top-k order + residual
  PfGemm q = pf_gemm_base(ctx);
  q.w = L.shared + gu_s;
  q.nG = c.f_shared / 64;
  q.n_items = t_items;
  q.rows_total = T;
  q.mode = PF_DN_SHARED;
  q.out32 = ctx->pf_ys;
  if (ctx->pf_timeline && rel == 0) q.tl = ctx->pf_timeline + 48;
  CK(launch_pf_gemm(ns, ctx->pf_map_as[ms], q, d / 128, t_items, s));
  PROF(-1, s);
  PROF(6, s);
  CK(launch_pf_combine(ctx->pf_ys, ctx->pf_ytok, ctx->pf_gates, hin, hout, rel == n_rel - 1 ? y_last : nullptr,
                       dbg && ctx->dbg_y ? ctx->dbg_y + xo * d : nullptr, T, d, k, s));
  PROF(-1, s);
  return MOE_OK;
}

bool sg_use(const moe_ctx* ctx, int T) { return ctx->sg_ok && ctx->use_sg && T <= kSgMaxT; }

// The rest of a layer of at most kSgMaxT tokens after its routing and grouping
// (one item per active expert, expert e's record at experts + e * stride): the
// two small-batch GEMV launches and the combine (+ residual).
moe_status pf_layer_small_rest(moe_ctx* ctx, int l, int rel, int n_rel, const uint16_t* hin, uint16_t* hout, int T,
                               float* y_last, const uint8_t* experts, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  const LayerStore& L = ctx->L[l];
  const bool dbg = rel < ctx->dbg_layers;
  const size_t xo = static_cast<size_t>(rel) * T;
  SgParams g{};
  g.d = c.d;
  g.f = c.f;
  g.fs = c.f_shared;
  g.T = T;
  g.P = T * c.top_k;
  g.gelu = c.gelu_variant;
  g.experts = experts;
  g.stride = ctx->stride;
  g.shared = L.shared;
  g.items = ctx->pf_items;
  g.n_items = ctx->pf_nitems;
  g.row_pair = ctx->pf_rowpair;
  g.xv = ctx->sg_xv;
  g.xg = ctx->sg_xg;
  g.av_r = ctx->pf_ar;
  g.av_s = ctx->pf_as;
  g.y_r = ctx->pf_ytok;
  g.y_s = ctx->pf_ys;
  g.err = ctx->err_word;
  PROF(7, s);
  g.mode = SG_GU;
  CK(launch_sg(g, ctx->n_sm, s));
  g.mode = SG_DN;
  CK(launch_sg(g, ctx->n_sm, s));
  PROF(-1, s);
  PROF(6, s);
  CK(launch_pf_combine(ctx->pf_ys, ctx->pf_ytok, ctx->pf_gates, hin, hout, rel == n_rel - 1 ? y_last : nullptr,
                       dbg && ctx->dbg_y ? ctx->dbg_y + xo * c.d : nullptr, T, c.d, c.top_k, s));
  PROF(-1, s);
  return MOE_OK;
}

// A layer of at most kSgMaxT tokens: the routing and grouping, then the rest.
moe_status pf_layer_small(moe_ctx* ctx, int l, int rel, int n_rel, const uint16_t* hin, uint16_t* hout, int T,
                          const float* bias, float* y_last, cudaStream_t s) {
  moe_status st = pf_layer_route(ctx, l, rel, hin, T, bias, s, true);
  if (st != MOE_OK) return st;
  return pf_layer_small_rest(ctx, l, rel, n_rel, hin, hout, T, y_last, ctx->L[l].experts, s);
}

moe_status pf_layer(moe_ctx* ctx, int l, int rel, int n_rel, const uint16_t* hin, uint16_t* hout, int T,
                    const float* bias, float* y_last, cudaStream_t s) {
  if (sg_use(ctx, T)) return pf_layer_small(ctx, l, rel, n_rel, hin, hout, T, bias, y_last, s);
  moe_status st = pf_layer_route(ctx, l, rel, hin, T, bias, s);
  if (st != MOE_OK) return st;
  PROF(5, s);
  st = pf_layer_shared_gu(ctx, l, rel, T, s);
  if (st != MOE_OK) return st;
  return pf_layer_rest(ctx, l, rel, n_rel, hin, hout, T, y_last, ctx->L[l].experts, s);
}

// The tcgen05 path over [l0, l1) for T tokens.
moe_status pf_enqueue(moe_ctx* ctx, const void* h, int T, int l0, int l1, const float* logit_bias, void* h_out,
                      float* y_last, cudaStream_t s) {
  const int n_rel = l1 - l0;
  for (int rel = 0; rel < n_rel; ++rel) {
    const uint16_t* hin = rel == 0 ? static_cast<const uint16_t*>(h) : ctx->pf_h[(rel - 1) & 1];
    uint16_t* hout = rel == n_rel - 1 ? static_cast<uint16_t*>(h_out) : ctx->pf_h[rel & 1];
    moe_status st = pf_layer(ctx, l0 + rel, rel, n_rel, hin, hout, T, logit_bias, y_last, s);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

// Stages the union of layer l's experts picked by the chunk (pf_cnt_host[e] >
// 0) into the arena on the side stream: from the pinned host pool, or read from
// the expert file into the staging halves, k records at a time.
moe_status pf_stage_union(moe_ctx* ctx, int l, int T) {
  const int E = ctx->cfg.n_experts, k = ctx->cfg.top_k;
  const bool from_file = ctx->file_fd >= 0;
  const volatile int32_t* cnt = ctx->pf_cnt_host;
  int n = 0;
  for (int e = 0; e < E; ++e) {
    const int ne = cnt[e];
    if (ne < 0 || ne > T) return fail(ctx, MOE_ECUDA, "corrupt prefill pair count (%d for expert %d)", ne, e);
    if (ne == 0) continue;
    const uint8_t* src;
    if (from_file) {
      const int half = ctx->fhalf, m = n % k;
      // the copies out of this staging half are done before it is refilled
      if (m == 0) CK(cudaEventSynchronize(ctx->fev[half]));
      uint8_t* dst = ctx->fstage + (static_cast<size_t>(half) * k + m) * ctx->file_stride;
      moe_status st = file_read_record(ctx, l, e, dst);
      if (st != MOE_OK) return st;
      src = dst;
    } else {
      src = ctx->pool + (static_cast<size_t>(l) * E + e) * ctx->stride;
    }
    CK(cudaMemcpyAsync(ctx->pf_arena + static_cast<size_t>(e) * ctx->stride, src, ctx->expert_bytes,
                       cudaMemcpyHostToDevice, ctx->side));
    ctx->staged += ctx->expert_bytes;
    ++n;
    if (from_file && n % k == 0) {
      CK(cudaEventRecord(ctx->fev[ctx->fhalf], ctx->side));
      ctx->fhalf ^= 1;
    }
  }
  if (from_file && n % k != 0) {
    CK(cudaEventRecord(ctx->fev[ctx->fhalf], ctx->side));
    ctx->fhalf ^= 1;
  }
  return MOE_OK;
}

// Chunked prefill of a host-pool or expert-file context over [l0, l1): per
// layer, the chunk's T tokens are routed, the union of their experts is staged
// once into the arena, and the layer's grouped GEMMs run over it; the shared
// expert's gate/up runs while the union is staged.
moe_status pf_pool_run(moe_ctx* ctx, const void* h, int T, int l0, int l1, const float* logit_bias, void* h_out,
                       float* y_last, cudaStream_t s) {
  moe_status st = pf_alloc(ctx);
  if (st != MOE_OK) return st;
  g_chain_pdl = ctx->pdl && !ctx->profiling;
  const int E = ctx->cfg.n_experts;
  if (!ctx->pf_arena) {
    size_t nb = 0;
    uint8_t* arena = dalloc<uint8_t>(static_cast<size_t>(E) * ctx->stride, ctx->pf_owned, nb);
    if (!arena) return fail(ctx, MOE_ENOMEM, "prefill expert arena (%zu bytes)", static_cast<size_t>(E) * ctx->stride);
    if (cudaHostAlloc(reinterpret_cast<void**>(&ctx->pf_cnt_host), static_cast<size_t>(E) * 4,
                      cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      ctx->pf_cnt_host = nullptr;
      return fail(ctx, MOE_ENOMEM, "pinned prefill counts");
    }
    CK(cudaEventCreateWithFlags(&ctx->pf_ev_cnt, cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&ctx->pf_ev_read, cudaEventDisableTiming));
    ctx->device_bytes += nb;
    ctx->pf_arena = arena;
  }
  const int n_rel = l1 - l0;
  for (int rel = 0; rel < n_rel; ++rel) {
    const int l = l0 + rel;
    const uint16_t* hin = rel == 0 ? static_cast<const uint16_t*>(h) : ctx->pf_h[(rel - 1) & 1];
    uint16_t* hout = rel == n_rel - 1 ? static_cast<uint16_t*>(h_out) : ctx->pf_h[rel & 1];
    const bool small = sg_use(ctx, T);
    st = pf_layer_route(ctx, l, rel, hin, T, logit_bias, s, small);
    if (st != MOE_OK) return st;
    CK(cudaMemcpyAsync(ctx->pf_cnt_host, ctx->pf_cnt, static_cast<size_t>(E) * 4, cudaMemcpyDeviceToHost, s));
    CK(cudaEventRecord(ctx->pf_ev_cnt, s));
    if (!small) {   // the shared expert's gate/up runs while the union is staged
      PROF(5, s);
      st = pf_layer_shared_gu(ctx, l, rel, T, s);
      if (st != MOE_OK) return st;
    }
    st = wait_event(ctx, ctx->pf_ev_cnt, "prefill routing");
    if (st != MOE_OK) return st;
    // the arena is rewritten only after the GEMMs that read it last are done
    CK(cudaStreamWaitEvent(ctx->side, ctx->pf_ev_read, 0));
    st = pf_stage_union(ctx, l, T);
    if (st != MOE_OK) return st;
    CK(cudaEventRecord(ctx->ev_copy, ctx->side));
    CK(cudaStreamWaitEvent(s, ctx->ev_copy, 0));
    st = small ? pf_layer_small_rest(ctx, l, rel, n_rel, hin, hout, T, y_last, ctx->pf_arena, s)
               : pf_layer_rest(ctx, l, rel, n_rel, hin, hout, T, y_last, ctx->pf_arena, s);
    if (st != MOE_OK) return st;
    CK(cudaEventRecord(ctx->pf_ev_read, s));
  }
  return prof_collect(ctx, s);
}

moe_status pf_run(moe_ctx* ctx, const void* h, int T, int l0, int l1, const float* logit_bias, void* h_out,
                  float* y_last, cudaStream_t s) {
  moe_status st = pf_alloc(ctx);
  if (st != MOE_OK) return st;
  g_chain_pdl = ctx->pdl && !ctx->profiling;
  const moe_config& c = ctx->cfg;
  const bool dbg = dbg_on(ctx);
  if (ctx->profiling || dbg || T > kPfGraphMaxT || ctx->pf_timeline) {
    st = pf_enqueue(ctx, h, T, l0, l1, logit_bias, h_out, y_last, s);
    if (st != MOE_OK) return st;
    return prof_collect(ctx, s);
  }
  // small batches: one graph launch for all layers (the ~10 short kernels per layer would
  // otherwise cost more in launch gaps than in work); the caller's buffers are copied in and out
  const int n_rel = l1 - l0;
  if (!ctx->pf_gin) {
    size_t nb = 0;
    ctx->pf_gin = dalloc<uint16_t>(static_cast<size_t>(c.max_tokens) * c.d, ctx->pf_owned, nb);
    ctx->pf_gout = dalloc<uint16_t>(static_cast<size_t>(c.max_tokens) * c.d, ctx->pf_owned, nb);
    ctx->pf_gy = dalloc<float>(static_cast<size_t>(c.max_tokens) * c.d, ctx->pf_owned, nb);
    if (!ctx->pf_gin || !ctx->pf_gout || !ctx->pf_gy) return fail(ctx, MOE_ENOMEM, "graph staging buffers");
    ctx->device_bytes += nb;
  }
  if (logit_bias && !ctx->pf_gbias) {
    size_t nb = 0;
    ctx->pf_gbias = dalloc<float>(static_cast<size_t>(c.n_layers) * c.max_tokens * c.n_experts, ctx->pf_owned, nb);
    if (!ctx->pf_gbias) return fail(ctx, MOE_ENOMEM, "graph bias buffer");
    ctx->device_bytes += nb;
  }
  const size_t hb = static_cast<size_t>(T) * c.d * 2;
  CK(cudaMemcpyAsync(ctx->pf_gin, h, hb, cudaMemcpyDeviceToDevice, s));
  if (logit_bias)
    CK(cudaMemcpyAsync(ctx->pf_gbias, logit_bias, static_cast<size_t>(n_rel) * T * c.n_experts * 4,
                       cudaMemcpyDeviceToDevice, s));
  const auto key = std::make_tuple(T, l0, l1, logit_bias ? 1 : 0, y_last ? 1 : 0);
  auto it = ctx->pf_graphs.find(key);
  if (it == ctx->pf_graphs.end()) {
    cudaGraph_t g = nullptr;
    CK(cudaStreamBeginCapture(ctx->cap, cudaStreamCaptureModeThreadLocal));
    st = pf_enqueue(ctx, ctx->pf_gin, T, l0, l1, logit_bias ? ctx->pf_gbias : nullptr, ctx->pf_gout,
                    y_last ? ctx->pf_gy : nullptr, ctx->cap);
    cudaError_t e = cudaStreamEndCapture(ctx->cap, &g);
    if (st != MOE_OK) {
      if (g) cudaGraphDestroy(g);
      return st;
    }
    CK(e);
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    CK(e);
    it = ctx->pf_graphs.emplace(key, ex).first;
  }
  CK(cudaGraphLaunch(it->second, s));
  CK(cudaMemcpyAsync(h_out, ctx->pf_gout, hb, cudaMemcpyDeviceToDevice, s));
  if (y_last) CK(cudaMemcpyAsync(y_last, ctx->pf_gy, static_cast<size_t>(T) * c.d * 4, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

}  // namespace

moe_status moe_prefill(moe_ctx* ctx, const void* h, int T, int layer_begin, int layer_end, const float* logit_bias,
                       void* h_out, float* y_last, void* stream) {
  moe_status st = check_ready(ctx, layer_begin, layer_end);
  if (st != MOE_OK) return st;
  if (!h || !h_out) return fail(ctx, MOE_EINVAL, "NULL h / h_out");
  if (T < 1 || T > ctx->cfg.max_tokens) return fail(ctx, MOE_EINVAL, "T=%d outside [1, %d]", T, ctx->cfg.max_tokens);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(cudaSetDevice(ctx->device));
  if (ctx->residency == MOE_HOST_POOL || ctx->residency == MOE_FILE_POOL) {
    if (!(ctx->pf_ok && ctx->use_pf))
      return fail(ctx, MOE_EINVAL, "prefill of a host-pool context needs the tcgen05 path (d %% 128 == 0, "
                                   "n_experts <= 128)");
    return pf_pool_run(ctx, h, T, layer_begin, layer_end, logit_bias, h_out, y_last, s);
  }
  const int d = ctx->cfg.d;
  if (ctx->pf_ok && ctx->use_pf) return pf_run(ctx, h, T, layer_begin, layer_end, logit_bias, h_out, y_last, s);
  // otherwise: the batched decode kernels, kMaxDecodeB tokens at a time
  for (int t0 = 0; t0 < T; t0 += ctx->Bd) {
    const int B = std::min(ctx->Bd, T - t0);
    const uint16_t* hi = static_cast<const uint16_t*>(h) + static_cast<size_t>(t0) * d;
    uint16_t* ho = static_cast<uint16_t*>(h_out) + static_cast<size_t>(t0) * d;
    float* yl = y_last ? y_last + static_cast<size_t>(t0) * d : nullptr;
    DevCallArgs a = make_args(ctx, hi, ho, yl, logit_bias, B, T, t0);
    st = put_args(ctx, a, s);
    if (st != MOE_OK) return st;
    st = resident_run(ctx, B, layer_begin, layer_end, s);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_host_read_rate(const void* host_buf, uint64_t bytes, int reps, void* stream, double* gbs) {
  if (!host_buf || !gbs || bytes == 0 || bytes % 16 != 0 || reps < 1 ||
      reinterpret_cast<uintptr_t>(host_buf) % 16 != 0)
    return MOE_EINVAL;
  *gbs = 0.0;
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, host_buf) != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return MOE_EINVAL;   // not page-locked host memory the device can read
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return MOE_ECUDA;
  const void* src = attr.devicePointer ? attr.devicePointer : host_buf;
  unsigned* sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  moe_status st = MOE_ECUDA;
  float ms = 0.f;
  if (cudaMalloc(&sink, sizeof(unsigned)) == cudaSuccess && cudaEventCreate(&e0) == cudaSuccess &&
      cudaEventCreate(&e1) == cudaSuccess &&
      launch_host_read(src, static_cast<long long>(bytes), sink, n_sm, s) == cudaSuccess &&   // warm-up
      cudaEventRecord(e0, s) == cudaSuccess) {
    bool ok = true;
    for (int r = 0; r < reps && ok; ++r) ok = launch_host_read(src, static_cast<long long>(bytes), sink, n_sm, s) == cudaSuccess;
    if (ok && cudaEventRecord(e1, s) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
        cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess && ms > 0.f) {
      *gbs = static_cast<double>(bytes) * reps / (ms * 1e-3) / 1e9;
      st = MOE_OK;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (sink) cudaFree(sink);
  cudaGetLastError();
  return st;
}

moe_status moe_set_debug(moe_ctx* ctx, uint16_t* x_layers, int32_t* ids, float* gates, float* y_layers,
                         int max_layers) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (max_layers < 0) return fail(ctx, MOE_EINVAL, "negative max_layers");
  ctx->dbg_x = x_layers;
  ctx->dbg_ids = ids;
  ctx->dbg_gates = gates;
  ctx->dbg_y = y_layers;
  ctx->dbg_layers = max_layers;
  return MOE_OK;
}

moe_status moe_set_debug_logits(moe_ctx* ctx, int64_t* logits) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  ctx->dbg_logits = logits;
  return MOE_OK;
}

moe_status moe_sync(moe_ctx* ctx, void* stream) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  CK(cudaSetDevice(ctx->device));
  CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  CK(cudaStreamSynchronize(ctx->side));
  uint32_t w = 0;
  CK(cudaMemcpy(&w, ctx->err_word, 4, cudaMemcpyDeviceToHost));
  if (w) CK(cudaMemset(ctx->err_word, 0, 4));
  if (w & ERR_WAIT_TIMEOUT) return fail(ctx, MOE_ETIMEOUT, "a device wait ran out (error word 0x%x)", w);
  if (w & ERR_PLAN) return fail(ctx, MOE_ECUDA, "device plan overflow (error word 0x%x)", w);
  if (w & ERR_ROUTER_DOMAIN) return fail(ctx, MOE_EDOMAIN, "router input outside the exact fixed-point domain");
  if (w & ERR_PF_RANGE) return fail(ctx, MOE_EDOMAIN, "an fp16 matrix operand (prefill, or the clustered decode kernel) is outside [-65504, 65504]");
  if (w & ERR_LAUNCH_SHAPE)
    return fail(ctx, MOE_ECUDA, "clustered decode kernel ran without clusters of %d CTAs (error word 0x%x)", kCCluster, w);
  if (w & ERR_Y_RANGE) return fail(ctx, MOE_EDOMAIN, "decode: a partial FFN output is outside (-2^24, 2^24)");
  return MOE_OK;
}

moe_status moe_get_stats(moe_ctx* ctx, moe_stats* out) {
  if (!ctx || !out) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());
  std::vector<long long> cnt(static_cast<size_t>(ctx->cfg.n_layers) * 2);
  CK(cudaMemcpy(cnt.data(), ctx->lru_counts, cnt.size() * 8, cudaMemcpyDeviceToHost));
  memset(out, 0, sizeof(*out));
  for (int l = 0; l < ctx->cfg.n_layers; ++l) {
    out->hits += cnt[2 * l];
    out->misses += cnt[2 * l + 1];
  }
  out->steps = ctx->steps;
  out->staged_bytes = ctx->staged;
  out->file_read_bytes = ctx->file_read_bytes;
  out->host_tier_hits = ctx->host_hits;
  out->host_tier_bytes = ctx->hcache ? static_cast<int64_t>(ctx->cfg.n_layers) * ctx->n_host * ctx->file_stride : 0;
  out->n_slots = ctx->n_slots;
  out->expert_bytes = ctx->expert_bytes;
  // device-driven staging copies every miss once (the mode switch zeroed the counters)
  if (ctx->stage_device || ctx->stage_fused) out->staged_bytes += out->misses * ctx->expert_bytes;
  out->shared_bytes = ctx->shared_bytes;
  size_t dev = ctx->device_bytes;
  for (auto& Ls : ctx->L) {
    if (Ls.router_w) dev += static_cast<size_t>(ctx->cfg.n_experts) * ctx->cfg.d * 2;
    if (Ls.shared) dev += ctx->shared_bytes;
    if (Ls.experts) dev += static_cast<size_t>(ctx->cfg.n_experts) * ctx->stride;
    if (Ls.slots) dev += static_cast<size_t>(ctx->n_slots) * ctx->stride;
  }
  out->device_bytes = static_cast<int64_t>(dev);
  out->host_pool_bytes = static_cast<int64_t>(ctx->pool_bytes);
  return MOE_OK;
}

moe_status moe_get_cache_state(moe_ctx* ctx, int layer, int32_t* expert_of_slot, int64_t* last_use) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(ctx, MOE_EINVAL, "layer %d out of range", layer);
  if ((ctx->residency != MOE_HOST_POOL && ctx->residency != MOE_FILE_POOL) || ctx->n_slots == 0)
    return fail(ctx, MOE_ESTATE, "no slot cache");
  CK(cudaSetDevice(ctx->device));
  CK(cudaDeviceSynchronize());
  if (expert_of_slot)
    CK(cudaMemcpy(expert_of_slot, ctx->L[layer].expert_of_slot, ctx->n_slots * 4, cudaMemcpyDeviceToHost));
  if (last_use) CK(cudaMemcpy(last_use, ctx->L[layer].last_use, ctx->n_slots * 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_profile(moe_ctx* ctx, int enable) {
  if (!ctx) return MOE_EINVAL;
  if (ctx->poisoned) return fail(ctx, MOE_ESTATE, "context is poisoned: %s", ctx->err.c_str());
  ctx->profiling = enable != 0;
  ctx->prof_n = 0;
  return MOE_OK;
}

moe_status moe_get_profile(moe_ctx* ctx, moe_kernel_time* out, int n) {
  if (!ctx || !out || n < 0) return MOE_EINVAL;
  for (int i = 0; i < n && i < MOE_N_KERNEL_KINDS; ++i) {
    out[i] = ctx->prof[i];
    ctx->prof[i] = moe_kernel_time{};
  }
  return MOE_OK;
}

moe_status moe_test_hook(moe_ctx* ctx, int hook, int64_t value) {
  if (!ctx) return MOE_EINVAL;
  switch (hook) {
    case 1: ctx->hook_fail_copy = value != 0; return MOE_OK;
    case 2:
      if (value == -1) {
        ctx->hook_force_timeout = true;
        return MOE_OK;
      }
      if (value < 0) return fail(ctx, MOE_EINVAL, "negative wait limit");
      ctx->wait_limit_us = value;
      return MOE_OK;
    case 3: {  // programmatic dependent launch on/off
      const bool want = value != 0;
      if (want != ctx->pdl) {
        for (auto& kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
        ctx->graphs.clear();
        for (auto& kv : ctx->pf_graphs) cudaGraphExecDestroy(kv.second);
        ctx->pf_graphs.clear();
        ctx->pdl = want;
      }
      return MOE_OK;
    }
    case 8:  // event times of the prefill GEMMs' CTA (0, 0), first layer of a call, into [4][16] (0 = off)
      ctx->pf_timeline = reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
      return MOE_OK;
    case 7:  // tcgen05 batched prefill on/off; asking for it where it cannot run is an error
      if (value != 0 && !ctx->pf_ok)
        return fail(ctx, MOE_ESTATE, "tcgen05 prefill unavailable for this configuration or device");
      ctx->use_pf = value != 0;
      return MOE_OK;
    case 14:  // decode steps of 2 to kClusterLoopMaxB tokens: one clustered-kernel launch per token (on/off)
      ctx->c_loop = value != 0;
      return MOE_OK;
    case 13:  // small-batch GEMVs on/off for calls of at most kSgMaxT tokens on the grouped path
      if (value != 0 && !ctx->sg_ok)
        return fail(ctx, MOE_ESTATE, "small-batch GEMVs unavailable for this configuration or device");
      if ((value != 0) != ctx->use_sg) {   // cached graphs hold the other path
        for (auto& kv : ctx->pf_graphs) cudaGraphExecDestroy(kv.second);
        ctx->pf_graphs.clear();
        ctx->use_sg = value != 0;
      }
      return MOE_OK;
    case 9:  // clustered (1) or per-SM (0) persistent decode kernel; asking for one that cannot run is an error
      if ((value != 0 && !ctx->c_ok) || (value == 0 && !ctx->p_ok))
        return fail(ctx, MOE_ESTATE, "that persistent decode kernel is unavailable for this configuration or device");
      ctx->use_cluster = value != 0;
      return MOE_OK;
    case 4:  // persistent B = 1 decode kernel on/off; asking for it where it cannot run is an error
      if (value != 0 && !ctx->p_ok && !ctx->c_ok)
        return fail(ctx, MOE_ESTATE, "persistent decode kernel unavailable for this configuration or device");
      ctx->use_persistent = value != 0;
      return MOE_OK;
    case 10:  // bounded waits of the persistent decode kernels give up after `value` cycles (<= 0: the default, ~2 s)
      ctx->spin_limit = value > 0 ? value : 4000000000LL;
      return MOE_OK;
    case 11: {  // MOE_OK when the persistent kernels' launch words are at rest, else MOE_ESTATE (poisoned contexts too)
      CK(cudaDeviceSynchronize());
      std::vector<unsigned> w;
      std::vector<long long> yb;
      auto take = [&](const unsigned* src, size_t n) -> cudaError_t {
        if (!src || !n) return cudaSuccess;
        const size_t o = w.size();
        w.resize(o + n);
        return cudaMemcpy(w.data() + o, src, n * 4, cudaMemcpyDeviceToHost);
      };
      CK(take(ctx->p_exit, ctx->p_exit ? 2 : 0));
      CK(take(ctx->p_counters, ctx->p_counters ? static_cast<size_t>(ctx->p_n_counters) : 0));
      CK(take(ctx->c_counters, ctx->c_counters ? 2 : 0));
      if (ctx->c_ybuf) {
        yb.resize(static_cast<size_t>(3) * ctx->cfg.d);
        CK(cudaMemcpy(yb.data(), ctx->c_ybuf, yb.size() * 8, cudaMemcpyDeviceToHost));
      }
      for (unsigned v : w)
        if (v) return MOE_ESTATE;
      for (long long v : yb)
        if (v) return MOE_ESTATE;
      return MOE_OK;
    }
    case 12: {  // the clustered kernel's wait diagnostic (site << 16 | CTA, 0: none) into *(uint32_t*)value, then cleared
      if (!value || !ctx->c_counters) return fail(ctx, MOE_EINVAL, "hook 12 needs a host address and the clustered kernel");
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(reinterpret_cast<void*>(static_cast<uintptr_t>(value)), ctx->c_counters + 2, 4, cudaMemcpyDeviceToHost));
      CK(cudaMemset(ctx->c_counters + 2, 0, 4));
      return MOE_OK;
    }
    case 6:  // budget checks see `value` bytes of free device memory (-1: the real figure)
      ctx->hook_free_bytes = value;
      return MOE_OK;
    case 5:  // event timeline of the persistent kernel into a caller device buffer (0 = off)
      ctx->p_timeline = reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
      return MOE_OK;
    default: return fail(ctx, MOE_EINVAL, "unknown hook %d", hook);
  }
}

}  // extern "C"
