// Structures shared by the libmoe host code and its kernels.
//
// Device weight layout of one expert (a permutation of the canonical bytes):
//
//   gate/up region: f/8 tiles of 8 rows; tile t holds gate rows 8t..8t+7 and
//   up rows 8t..8t+7 as the 16 rows of an m16 MMA tile.  A tile is d/64
//   groups of 576 bytes:
//     bytes [0, 512):   32 lanes x 16 bytes; lane l's 16 bytes are four
//                       32-bit words, one per k16 step of the group, each
//                       holding exactly the eight nibbles lane l needs as its
//                       bf16 A fragment: nibble i of the word sits at bits
//                       [4i, 4i+4); register r of the fragment takes nibbles
//                       r (low half) and r+4 (high half), so the word holds,
//                       for lane (g = l/4, t4 = l%4) and step base kb:
//                       gate: n0 = W[g][kb+2t4], n4 = W[g][kb+2t4+1],
//                             n2 = W[g][kb+2t4+8], n6 = W[g][kb+2t4+9];
//                       up:   n1, n5, n3, n7 at the same columns;
//                       down: n0/n4/n2/n6 from row g, n1/n5/n3/n7 from row g+8;
//     bytes [512, 576): 8 entries x 8 bytes: entry g = fp16 (scale, bias) of
//                       gate row 8t+g, then of up row 8t+g.
//   down region: d/16 tiles of 16 output rows; tile T is f/64 groups of 576
//   bytes: 512 bytes of fragments, then entry g = (scale, bias) of row 16T+g
//   and of row 16T+g+8.
//
// Totals equal the canonical sizes: 1.125*f*d + 0.5625*d*f bytes.
#pragma once

#include <cstdint>

namespace moe {

// Device error word bits (ORed by kernels, read and cleared by moe_sync).
enum : uint32_t {
  ERR_ROUTER_DOMAIN = 1u << 0,   // |W_r * x| >= 2^11 or a non-finite router input
  ERR_WAIT_TIMEOUT = 1u << 1,    // a bounded wait ran out
  ERR_PLAN = 1u << 2,            // plan capacity exceeded (should be unreachable)
  ERR_PF_RANGE = 1u << 3,        // an fp16 matrix operand would overflow (|v| >= 65504)
  ERR_Y_RANGE = 1u << 4,         // decode: a CTA's partial layer output beyond 2^24 (fixed-point sum range)
  ERR_LAUNCH_SHAPE = 1u << 5,    // the clustered kernel ran without its cluster shape (it returned at once)
};

constexpr int kGroup = 64;
constexpr int kGroupBytes = 576;       // one (tile, group) block
constexpr int kFragBytes = 512;        // fragment part of a block

struct DevCallArgs {                   // per-call pointers, written before each call
  const uint16_t* h_in;                // bf16 [B][d]
  uint16_t* h_out;                     // bf16 [B][d]
  float* y_last;                       // fp32 [B][d] or null
  const float* bias;                   // fp32 [L][B][E] or null
  uint16_t* dbg_x;                     // bf16 [L][B][d] or null
  int32_t* dbg_ids;                    // int32 [L][B][k] or null
  float* dbg_gates;                    // fp32 [L][B][k] or null
  float* dbg_y;                        // fp32 [L][B][d] or null
  int64_t* dbg_logits;                 // int64 [L][B][E] or null: router logits (bias included), 2^-40 units
  int32_t dbg_layers;
  int32_t B;                           // tokens of this launch
  int32_t tok_total;                   // tokens per layer in bias / debug buffers
  int32_t tok_off;                     // first token of this launch within them
  int64_t step;                        // LRU step counter (host-pool mode)
};

struct PlanHdr {
  int32_t n_active;                    // U: distinct experts picked by the B tokens
  int32_t n_miss;                      // host-pool: misses of this layer
  int32_t pad[2];
};

// Everything one kernel launch needs, passed by value.
struct KParams {
  // dimensions
  int d, f, fs, E, k, B, prenorm, gelu;
  float eps;
  int n_sc;                            // shared down chunks
  int cg;                              // groups per shared down chunk (= f/64)
  int layer;                           // absolute layer index
  int rel_layer;                       // layer - layer_begin of the call
  int first, last;                     // first / last layer of the call
  int pool;                            // 1 = host-pool mode
  int pass;                            // gate/up pass: -1 all, 0 shared+hits, 1 misses
  int n_slots;
  // weights of this layer (device)
  const uint16_t* router_w;            // fp16 [E][d]
  const uint8_t* shared;               // device layout
  const uint8_t* experts;              // resident base, or slot base in host-pool mode
  long long expert_stride;             // bytes
  int32_t* slot_of_expert;             // [E] host-pool mode
  int32_t* expert_of_slot;             // [N]
  long long* last_use;                 // [N]
  long long* lru_counts;               // [L][2] hits, misses
  int policy;                          // 0 LRU, 1 LFU (host-pool mode)
  long long* use_count;                // [E] whole-run picks per expert of this layer (LFU)
  int32_t* host_rec;                   // mapped host [L][1 + 2k + 4k] record of this layer
  // residual stream
  const uint16_t* h_src;               // layer input (null: read call args h_in)
  uint16_t* h_dst;                     // layer output (null: write call args h_out)
  // scratch
  const DevCallArgs* args;
  uint16_t* x_perm;                    // bf16 fragments [B][d]
  float* xg;                           // [B][d/64]
  long long* logits;                   // [B][E]
  int32_t* ids;                        // [B][k]
  float* gates;                        // [B][k]
  int32_t* tok_cnt;                    // [B]
  int32_t* all_cnt;                    // [1]
  PlanHdr* plan;
  int32_t* act_expert;                 // [B*k]
  int32_t* act_off;
  int32_t* act_cnt;
  int32_t* act_pass;
  int32_t* pair_tok;                   // [B*k]
  float* pair_gate;
  int32_t* pos_of;                     // [B][k]
  uint16_t* a_s;                       // hi/lo fragments [B][fs*2]
  uint16_t* a_r;                       // [B*k][f*2]
  float* asum_s;                       // [B][fs/8][2]
  float* asum_r;                       // [B*k][f/8][2]
  float* part_s;                       // [n_sc][B][d]
  float* y_r;                          // [B*k][d]
  int32_t* row_cnt;                    // [d/16]
  uint32_t* err;
};

}  // namespace moe
