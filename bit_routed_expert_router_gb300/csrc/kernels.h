// Launchers of the libmoe kernels (host side).
#pragma once

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
};

size_t persistent_smem();
int persistent_max_tiles_per_cta();
int persistent_max_tasks();
cudaError_t persistent_attrs();
cudaError_t persistent_occupancy(int* blocks_per_sm);
cudaError_t launch_persistent(PParams& p, int grid, cudaStream_t s);

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
