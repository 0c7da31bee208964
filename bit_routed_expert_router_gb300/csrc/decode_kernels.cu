// Decode-path kernels of libmoe (sm_103a).
//
// Per layer the host enqueues three kernels:
//   k_router  - (optional RMS norm), exact fixed-point router logits, top-k
//               with lower-index ties, softmax gates over the picked k (the
//               TurboFieldfare video transcript: eight of the experts are
//               picked per token), the per-layer LRU slot step in host-pool
//               mode, and the token-by-expert plan;
//   k_gateup  - fused int4 gate+up GEMV with GELU(gate)*up for the shared
//               expert, which every token runs, and every picked expert; int4
//               affine groups of 64 (write-up section "Vectorization helped
//               when it respected the storage layout");
//   k_down    - int4 down GEMV per (16-row tile, source) and, by the last
//               source to finish a tile, the fixed-order router-weighted
//               combine y = y_shared + sum_j gate_j y_j and the residual.
//
// Work is split the way the TurboFieldfare write-up found fastest for its
// routed-MoE kernel (section "MoE needed parallel work, reuse, and coarse
// overlap": resident workgroups taking rows until the dispatch is done): many
// independent warps, each owning a row tile of one expert, instead of several
// lanes cooperating on one expert.  On sm_103a a
// warp stages its whole tile into shared memory with one bulk (TMA-engine)
// copy, then runs the int4 dot products on the tensor cores: nibbles become
// bf16 (128 + q) operands in registers, the 128 offset and the affine
// (scale, bias) are applied per group in fp32.
#include "common.cuh"
#include "internal.h"
#include "kernels.h"
#include "staging.h"

#include <climits>

namespace moe {

// ------------------------------------------------------------------ router

__device__ __forceinline__ void build_plan_and_lru(const KParams& p, const DevCallArgs* A, int B);

__global__ void __launch_bounds__(256) k_router(KParams p) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm_raw);
  __shared__ float red[8];
  __shared__ int s_flag;
  const int b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d;

  pdl_wait();
  pdl_trigger();
  const DevCallArgs* A = p.args;
  const int B = A->B;
  const uint16_t* h = (p.h_src ? p.h_src : A->h_in) + static_cast<size_t>(b) * d;

  float ss = 0.f;
  for (int i = tid; i < d; i += 256) {
    const uint16_t v = h[i];
    xs[i] = v;
    const float fv = bf16_bits_to_float(v);
    ss += fv * fv;
  }
  if (p.prenorm) {
#pragma unroll
    for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float r = 1.0f / sqrtf(tot / static_cast<float>(d) + p.eps);
    for (int i = tid; i < d; i += 256) xs[i] = float_to_bf16_bits(bf16_bits_to_float(xs[i]) * r);
  }
  __syncthreads();

  // logits: warp w owns expert blockIdx.x*8 + w
  const int e = blockIdx.x * 8 + warp;
  if (e < p.E) {
    const uint4* wr = reinterpret_cast<const uint4*>(p.router_w + static_cast<size_t>(e) * d);
    const uint4* xv4 = reinterpret_cast<const uint4*>(xs);
    Fix40 fx;
    bool bad = false;
    for (int c = lane; c < d / 8; c += 32) {
      const uint4 wv = __ldg(wr + c);
      const uint4 xv = xv4[c];
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
    if (lane == 0) {
      if (A->bias) {
        const float bv = A->bias[(static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off + b) * p.E + e];
        if (!(fabsf(bv) < 1048576.f)) {
          atomicOr(p.err, ERR_ROUTER_DOMAIN);
        } else {
          acc += __float2ll_rn(bv * 1099511627776.0f);
        }
      }
      p.logits[static_cast<size_t>(b) * p.E + e] = acc;
      __threadfence();
    }
  }

  if (blockIdx.x == 0) {
    // B-operand fragments of x: per (group G, t4, step st) the four bf16
    // x[64G+16st+2t4 + {0,1,8,9}].
    uint2* xp = reinterpret_cast<uint2*>(p.x_perm + static_cast<size_t>(b) * d);
    for (int idx = tid; idx < d / 4; idx += 256) {
      const int st = idx & 3, t4 = (idx >> 2) & 3, G = idx >> 4;
      const int base = 64 * G + 16 * st + 2 * t4;
      uint2 v;
      v.x = static_cast<uint32_t>(xs[base]) | (static_cast<uint32_t>(xs[base + 1]) << 16);
      v.y = static_cast<uint32_t>(xs[base + 8]) | (static_cast<uint32_t>(xs[base + 9]) << 16);
      xp[idx] = v;
    }
    for (int G = tid; G < d / 64; G += 256) {
      float s = 0.f;
      for (int i = 0; i < 64; ++i) s += bf16_bits_to_float(xs[64 * G + i]);
      p.xg[static_cast<size_t>(b) * (d / 64) + G] = s;
    }
    if (A->dbg_x && p.rel_layer < A->dbg_layers) {
      uint16_t* dx = A->dbg_x + (static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off + b) * d;
      for (int i = tid; i < d; i += 256) dx[i] = xs[i];
    }
    __threadfence();
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&p.tok_cnt[b], 1);
    s_flag = (old == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  // ---- last CTA of token b: top-k + gates (warp 0)
  if (warp == 0) {
    const int E = p.E, k = p.k;
    long long v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ee = lane + 32 * i;
      v[i] = (ee < E) ? __ldcg(&p.logits[static_cast<size_t>(b) * E + ee]) : LLONG_MIN;
      if (ee < E && A->dbg_logits && p.rel_layer < A->dbg_layers)
        A->dbg_logits[(static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off + b) * E + ee] = v[i];
    }
    unsigned taken = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i >= E) taken |= 1u << i;
    int my_id = 0;
    long long my_v = 0;
    for (int j = 0; j < k; ++j) {
      long long bv = LLONG_MIN;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!(taken & (1u << i))) {
          const int ee = lane + 32 * i;
          if (v[i] > bv || (v[i] == bv && ee < be)) {
            bv = v[i];
            be = ee;
          }
        }
      }
#pragma unroll
      for (int m = 16; m; m >>= 1) {
        const long long ov = shfl_xor_i64(bv, m);
        const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, m);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == be) taken |= 1u << i;
      if (lane == j) {
        my_id = be;
        my_v = bv;
      }
    }
    const long long top = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    float ex = 0.f;
    if (lane < k) ex = expf(__ll2float_rn(my_v - top) * 9.094947017729282e-13f);  // 2^-40
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
    if (lane < k) {
      const float g = ex / sum;
      p.ids[b * k + lane] = my_id;
      p.gates[b * k + lane] = g;
      if (p.rel_layer < A->dbg_layers) {
        if (A->dbg_ids) A->dbg_ids[(static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off + b) * k + lane] = my_id;
        if (A->dbg_gates) A->dbg_gates[(static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off + b) * k + lane] = g;
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) {
    p.tok_cnt[b] = 0;
    __threadfence();
    const int old = atomicAdd(p.all_cnt, 1);
    s_flag = (old == B - 1);
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  if (tid == 0) *p.all_cnt = 0;
  build_plan_and_lru(p, A, B);
}

// Per-layer LRU step (host-pool mode, one token) and the token-by-expert plan.
// Runs in the single CTA that finished last.
__device__ __forceinline__ void build_plan_and_lru(const KParams& p, const DevCallArgs* A, int B) {
  __shared__ int cnt_e[256];
  __shared__ int u_of_e[256];
  __shared__ int s_hit[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k, nP = B * k;

  if (p.pool && warp == 0) {
    // Slot cache over this layer's slots (B == 1): hits refresh; misses in
    // top-k order take, among slots untouched this step, the smallest
    // (last_use, slot) under LRU, or (use count of its expert, last_use, slot)
    // under LFU (an empty slot counts -1).
    const int N = p.n_slots;
    const long long t = A->step;
    const bool lfu = p.policy == 1;
    int eos[8];
    long long lu[8], uc[8];
    unsigned used = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = lane + 32 * i;
      eos[i] = (s < N) ? p.expert_of_slot[s] : -1;
      lu[i] = (s < N) ? p.last_use[s] : LLONG_MAX;
      uc[i] = (!lfu || s >= N) ? 0 : (eos[i] >= 0 ? p.use_count[eos[i]] : -1);
      if (s >= N) used |= 1u << i;
    }
    int n_hit = 0, n_miss = 0;
    int32_t* rec = p.host_rec + static_cast<size_t>(p.rel_layer) * (1 + 6 * k);
    for (int j = 0; j < k; ++j) {
      const int ej = __ldcg(&p.ids[j]);
      const int s = p.slot_of_expert[ej];
      const int hit = s >= 0;
      if (hit) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (lane + 32 * i == s) {
            used |= 1u << i;
            lu[i] = t;
          }
        ++n_hit;
      }
      if (lane == 0) s_hit[j] = hit;
    }
    __syncwarp();
    for (int j = 0; j < k; ++j) {
      const int ej = __ldcg(&p.ids[j]);
      int slot, ev = -1;
      if (s_hit[j]) {
        slot = p.slot_of_expert[ej];
      } else {
        long long bc = LLONG_MAX, bv = LLONG_MAX;
        int bs = INT_MAX;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int s = lane + 32 * i;
          const bool better = uc[i] < bc || (uc[i] == bc && (lu[i] < bv || (lu[i] == bv && s < bs)));
          if (!(used & (1u << i)) && better) {
            bc = uc[i];
            bv = lu[i];
            bs = s;
          }
        }
#pragma unroll
        for (int m = 16; m; m >>= 1) {
          const long long oc = shfl_xor_i64(bc, m);
          const long long ov = shfl_xor_i64(bv, m);
          const int os = __shfl_xor_sync(0xFFFFFFFFu, bs, m);
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
        ev = __shfl_sync(0xFFFFFFFFu, my_ev, bs & 31);
        if (lane == 0) {
          if (ev >= 0) p.slot_of_expert[ev] = -1;
          p.slot_of_expert[ej] = bs;
          rec[1 + 2 * n_miss] = ej;
          rec[2 + 2 * n_miss] = bs;
        }
        ++n_miss;
      }
      if (lane == 0) {
        int32_t* tr = rec + 1 + 2 * k + 4 * j;
        tr[0] = ej;
        tr[1] = s_hit[j];
        tr[2] = slot;
        tr[3] = ev;
      }
      __syncwarp();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = lane + 32 * i;
      if (s < N) {
        p.expert_of_slot[s] = eos[i];
        p.last_use[s] = lu[i];
      }
    }
    if (lane == 0 && lfu)
      for (int j = 0; j < k; ++j) p.use_count[__ldcg(&p.ids[j])] += 1;
    if (lane == 0) {
      rec[0] = n_miss;
      p.plan->n_miss = n_miss;
      p.lru_counts[2 * p.layer + 0] += n_hit;
      p.lru_counts[2 * p.layer + 1] += n_miss;
    }
    __threadfence_system();
  }
  if (!p.pool && tid < 32) s_hit[tid] = 1;

  for (int ee = tid; ee < E; ee += blockDim.x) cnt_e[ee] = 0;
  __syncthreads();
  for (int q = tid; q < nP; q += blockDim.x) atomicAdd(&cnt_e[__ldcg(&p.ids[q])], 1);
  __syncthreads();
  if (tid == 0) {
    int U = 0, off = 0;
    for (int ee = 0; ee < E; ++ee) {
      const int c = cnt_e[ee];
      u_of_e[ee] = -1;
      if (c > 0) {
        p.act_expert[U] = ee;
        p.act_off[U] = off;
        p.act_cnt[U] = c;
        u_of_e[ee] = U;
        off += c;
        ++U;
      }
    }
    p.plan->n_active = U;
  }
  __syncthreads();
  for (int q = tid; q < nP; q += blockDim.x) {
    const int ee = __ldcg(&p.ids[q]);
    int rank = 0;
    for (int q2 = 0; q2 < q; ++q2) rank += (__ldcg(&p.ids[q2]) == ee);
    const int u = u_of_e[ee];
    const int pos = p.act_off[u] + rank;
    p.pair_tok[pos] = q / k;
    p.pair_gate[pos] = __ldcg(&p.gates[q]);
    p.pos_of[q] = pos;
    if (p.pool) p.act_pass[u] = s_hit[q % k] ? 0 : 1;
    else p.act_pass[u] = 0;
  }
  __threadfence();
}

// ------------------------------------------------------------------ gate/up

__device__ __forceinline__ float gelu_f(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

// Index (in bf16 elements) of intermediate element r, part `par` (0 hi, 1 lo),
// inside one token's fragment block of the down B operand.
__device__ __forceinline__ int a_frag_index(int r, int par) {
  const int G = r >> 6, st = (r >> 4) & 3, w = r & 15;
  const int t4 = (w & 7) >> 1, pos = ((w >> 3) << 1) | (w & 1);
  return ((((G * 2 + par) * 4 + t4) * 4 + st) << 2) + pos;
}

template <int NB>
__global__ void __launch_bounds__(kGuWarps * 32) k_gateup(KParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int nG = p.d / 64;
  const int tile_bytes = nG * kGroupBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm) + warp;
  uint8_t* buf = sm + 128 + static_cast<size_t>(warp) * tile_bytes;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  pdl_wait();
  pdl_trigger();
  const int B = p.args->B;
  const int U = p.plan->n_active;
  const int nS = p.fs / 8, tR = p.f / 8;
  const int n_items = nS + U * tR;
  uint32_t phase = 0;

  for (int item = blockIdx.x * kGuWarps + warp; item < n_items; item += gridDim.x * kGuWarps) {
    const uint8_t* src;
    int ntok, off = 0, tile, K;
    bool routed;
    if (item < nS) {
      if (p.pass == 1) continue;
      tile = item;
      src = p.shared + static_cast<size_t>(tile) * tile_bytes;
      ntok = B;
      routed = false;
      K = p.fs;
    } else {
      const int u = (item - nS) / tR;
      tile = (item - nS) - u * tR;
      if (p.pass >= 0 && p.act_pass[u] != p.pass) continue;
      const int ex = p.act_expert[u];
      const long long loc = p.pool ? p.slot_of_expert[ex] : ex;
      src = p.experts + loc * p.expert_stride + static_cast<size_t>(tile) * tile_bytes;
      ntok = p.act_cnt[u];
      off = p.act_off[u];
      routed = true;
      K = p.f;
    }
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, tile_bytes);
      bulk_g2s(buf, src, tile_bytes, bar);
    }

    // token of this lane's B column (g) and of its two C columns (2t4, 2t4+1)
    const uint4* xrow[NB];
    int ctok[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int col = nb * 8 + g;
      xrow[nb] = nullptr;
      if (col < ntok) {
        const int tok = routed ? p.pair_tok[off + col] : col;
        xrow[nb] = reinterpret_cast<const uint4*>(p.x_perm + static_cast<size_t>(tok) * p.d);
      }
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int c2 = nb * 8 + 2 * t4 + hc;
        ctok[nb][hc] = (c2 < ntok) ? (routed ? p.pair_tok[off + c2] : c2) : -1;
      }
    }
    float gacc[NB][2], uacc[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) gacc[nb][0] = gacc[nb][1] = uacc[nb][0] = uacc[nb][1] = 0.f;

    if (!mbar_wait_bounded(bar, phase, p.err)) {
      mbar_wait_bounded(bar, phase, p.err);  // give the copy in flight a second bounded chance
      return;
    }
    phase ^= 1;

    for (int G = 0; G < nG; ++G) {
      const uint8_t* blk = buf + G * kGroupBytes;
      const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
      const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
      const float sg = half_lo(sbv.x), bg = half_hi(sbv.x);
      const float su = half_lo(sbv.y), bu = half_hi(sbv.y);
      const float bg2 = fmaf(-128.f, sg, bg), bu2 = fmaf(-128.f, su, bu);
      uint4 xb[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if (xrow[nb]) {
          const uint4* src4 = xrow[nb] + (G * 4 + t4) * 2;
          xb[nb][0] = __ldg(src4);
          xb[nb][1] = __ldg(src4 + 1);
        } else {
          xb[nb][0] = make_uint4(0, 0, 0, 0);
          xb[nb][1] = make_uint4(0, 0, 0, 0);
        }
      }
      float c[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) c[nb][0] = c[nb][1] = c[nb][2] = c[nb][3] = 0.f;
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        uint32_t a[4];
        nibbles_to_bf16x2(qw[st], a);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint4& v = xb[nb][st >> 1];
          const uint32_t b0 = (st & 1) ? v.z : v.x;
          const uint32_t b1 = (st & 1) ? v.w : v.y;
          mma_bf16(c[nb], a, b0, b1);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const float X0 = ctok[nb][0] >= 0 ? __ldg(&p.xg[static_cast<size_t>(ctok[nb][0]) * nG + G]) : 0.f;
        const float X1 = ctok[nb][1] >= 0 ? __ldg(&p.xg[static_cast<size_t>(ctok[nb][1]) * nG + G]) : 0.f;
        gacc[nb][0] += sg * c[nb][0] + bg2 * X0;
        gacc[nb][1] += sg * c[nb][1] + bg2 * X1;
        uacc[nb][0] += su * c[nb][2] + bu2 * X0;
        uacc[nb][1] += su * c[nb][3] + bu2 * X1;
      }
    }

    // epilogue: a = GELU(gate) * up for row 8*tile+g, split into bf16 hi + lo
    const int r = tile * 8 + g;
    uint16_t* abase = routed ? p.a_r : p.a_s;
    float* sbase = routed ? p.asum_r : p.asum_s;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int col = nb * 8 + 2 * t4 + hc;
        const bool valid = col < ntok;
        const float av = gelu_f(gacc[nb][hc], p.gelu) * uacc[nb][hc];
        const uint16_t hi = float_to_bf16_bits(av);
        const uint16_t lo = float_to_bf16_bits(av - bf16_bits_to_float(hi));
        const int slot = routed ? off + col : col;
        if (valid) {
          uint16_t* ab = abase + static_cast<size_t>(slot) * (2 * K);
          ab[a_frag_index(r, 0)] = hi;
          ab[a_frag_index(r, 1)] = lo;
        }
        float sh = valid ? bf16_bits_to_float(hi) : 0.f;
        float sl = valid ? bf16_bits_to_float(lo) : 0.f;
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
          sh += __shfl_xor_sync(0xFFFFFFFFu, sh, m);
          sl += __shfl_xor_sync(0xFFFFFFFFu, sl, m);
        }
        if (valid && g == 0) {
          float* sp = sbase + (static_cast<size_t>(slot) * (K / 8) + tile) * 2;
          sp[0] = sh;
          sp[1] = sl;
        }
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ down + combine

template <int NB4>
__global__ void __launch_bounds__(kDnWarps * 32) k_down(KParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int cg = p.cg;
  const int buf_bytes = cg * kGroupBytes;
  constexpr int kTok = NB4 * 4;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm) + warp;
  uint8_t* buf = sm + 128 + static_cast<size_t>(warp) * buf_bytes;
  float* As = reinterpret_cast<float*>(sm + 128 + static_cast<size_t>(kDnWarps) * buf_bytes) +
              static_cast<size_t>(warp) * cg * kTok;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  pdl_wait();
  pdl_trigger();
  const DevCallArgs* A = p.args;
  const int B = A->B;
  const int U = p.plan->n_active;
  const int d = p.d;
  const int per_tile = p.n_sc + U;
  const int n_items = (d / 16) * per_tile;
  const int nGs = p.fs / 64, nGr = p.f / 64;
  const size_t gu_s = static_cast<size_t>(p.fs / 8) * (d / 64) * kGroupBytes;
  const size_t gu_r = static_cast<size_t>(p.f / 8) * (d / 64) * kGroupBytes;
  uint32_t phase = 0;

  for (int item = blockIdx.x * kDnWarps + warp; item < n_items; item += gridDim.x * kDnWarps) {
    const int T = item / per_tile;
    const int pidx = item - T * per_tile;
    const uint8_t* src;
    int ntok, off = 0, g0, ng, K;
    bool routed;
    if (pidx < p.n_sc) {
      g0 = pidx * cg;
      ng = min(cg, nGs - g0);
      src = p.shared + gu_s + (static_cast<size_t>(T) * nGs + g0) * kGroupBytes;
      ntok = B;
      routed = false;
      K = p.fs;
    } else {
      const int u = pidx - p.n_sc;
      const int ex = p.act_expert[u];
      const long long loc = p.pool ? p.slot_of_expert[ex] : ex;
      g0 = 0;
      ng = nGr;
      src = p.experts + loc * p.expert_stride + gu_r + static_cast<size_t>(T) * nGr * kGroupBytes;
      ntok = p.act_cnt[u];
      off = p.act_off[u];
      routed = true;
      K = p.f;
    }
    const int bytes = ng * kGroupBytes;
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(buf, src, bytes, bar);
    }

    const uint16_t* abase = routed ? p.a_r : p.a_s;
    const float* sbase = routed ? p.asum_r : p.asum_s;
    // per (group, token) sums of the hi+lo operand values, for the bias term
    for (int idx = lane; idx < ng * ntok; idx += 32) {
      const int G = idx / ntok, col = idx - G * ntok;
      const int slot = routed ? off + col : col;
      const float4* s4 = reinterpret_cast<const float4*>(sbase + (static_cast<size_t>(slot) * (K / 8) + (g0 + G) * 8) * 2);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = s4[i];
        s += v.x + v.y;
        s += v.z + v.w;
      }
      As[G * kTok + col] = s;
    }
    // B-operand rows of this lane: column g = (token g/2, part g&1)
    const uint4* arow[NB4];
#pragma unroll
    for (int nb = 0; nb < NB4; ++nb) {
      const int col = nb * 4 + (g >> 1);
      arow[nb] = nullptr;
      if (col < ntok) {
        const int slot = routed ? off + col : col;
        arow[nb] = reinterpret_cast<const uint4*>(abase + static_cast<size_t>(slot) * (2 * K));
      }
    }
    float y0[NB4], y1[NB4];
#pragma unroll
    for (int nb = 0; nb < NB4; ++nb) y0[nb] = y1[nb] = 0.f;
    __syncwarp();

    if (!mbar_wait_bounded(bar, phase, p.err)) {
      mbar_wait_bounded(bar, phase, p.err);
      return;
    }
    phase ^= 1;

    for (int G = 0; G < ng; ++G) {
      const uint8_t* blk = buf + G * kGroupBytes;
      const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
      const uint2 sbv = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
      const float s0 = half_lo(sbv.x), b0 = half_hi(sbv.x);
      const float s1 = half_lo(sbv.y), b1 = half_hi(sbv.y);
      const float b0c = fmaf(-128.f, s0, b0), b1c = fmaf(-128.f, s1, b1);
      uint4 ab[NB4][2];
#pragma unroll
      for (int nb = 0; nb < NB4; ++nb) {
        if (arow[nb]) {
          const uint4* s4 = arow[nb] + (((g0 + G) * 2 + (g & 1)) * 4 + t4) * 2;
          ab[nb][0] = __ldg(s4);
          ab[nb][1] = __ldg(s4 + 1);
        } else {
          ab[nb][0] = make_uint4(0, 0, 0, 0);
          ab[nb][1] = make_uint4(0, 0, 0, 0);
        }
      }
      float c[NB4][4];
#pragma unroll
      for (int nb = 0; nb < NB4; ++nb) c[nb][0] = c[nb][1] = c[nb][2] = c[nb][3] = 0.f;
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        uint32_t a[4];
        nibbles_to_bf16x2(qw[st], a);
#pragma unroll
        for (int nb = 0; nb < NB4; ++nb) {
          const uint4& v = ab[nb][st >> 1];
          const uint32_t bb0 = (st & 1) ? v.z : v.x;
          const uint32_t bb1 = (st & 1) ? v.w : v.y;
          mma_bf16(c[nb], a, bb0, bb1);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB4; ++nb) {
        const int col = nb * 4 + t4;
        const float Asum = (col < ntok) ? As[G * kTok + col] : 0.f;
        y0[nb] += s0 * (c[nb][0] + c[nb][1]) + b0c * Asum;
        y1[nb] += s1 * (c[nb][2] + c[nb][3]) + b1c * Asum;
      }
    }

    const int row0 = T * 16 + g;
#pragma unroll
    for (int nb = 0; nb < NB4; ++nb) {
      const int col = nb * 4 + t4;
      if (col < ntok) {
        float* dst = routed ? p.y_r + static_cast<size_t>(off + col) * d
                            : p.part_s + (static_cast<size_t>(pidx) * B + col) * d;
        dst[row0] = y0[nb];
        dst[row0 + 8] = y1[nb];
      }
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = (atomicAdd(&p.row_cnt[T], 1) == per_tile - 1);
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      __threadfence();
      const uint16_t* hin = p.h_src ? p.h_src : A->h_in;
      uint16_t* hout = p.h_dst ? p.h_dst : A->h_out;
      const int k = p.k;
      for (int idx = lane; idx < B * 16; idx += 32) {
        const int b = idx >> 4, row = T * 16 + (idx & 15);
        float y = 0.f;
        for (int c2 = 0; c2 < p.n_sc; ++c2) y += __ldcg(&p.part_s[(static_cast<size_t>(c2) * B + b) * d + row]);
        for (int j = 0; j < k; ++j) {
          const int pos = p.pos_of[b * k + j];
          y += p.pair_gate[pos] * __ldcg(&p.y_r[static_cast<size_t>(pos) * d + row]);
        }
        const size_t o = static_cast<size_t>(b) * d + row;
        hout[o] = float_to_bf16_bits(bf16_bits_to_float(hin[o]) + y);
        if (p.last && A->y_last) A->y_last[o] = y;
        if (A->dbg_y && p.rel_layer < A->dbg_layers)
          A->dbg_y[(static_cast<size_t>(p.rel_layer) * A->tok_total + A->tok_off) * d + o] = y;
      }
      if (lane == 0) p.row_cnt[T] = 0;
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ repack

__device__ __forceinline__ uint32_t nib_at(const uint8_t* q, int row_bytes, int r, int c) {
  return (q[static_cast<size_t>(r) * row_bytes + (c >> 1)] >> ((c & 1) * 4)) & 0xFu;
}

// Canonical gate/up [f][d] -> device tiles (see internal.h).
__global__ void k_repack_gu(const uint8_t* gq, const uint16_t* gsb, const uint8_t* uq, const uint16_t* usb,
                            int d, int f, uint8_t* dst) {
  const int nG = d / 64;
  const long long n_words = static_cast<long long>(f / 8) * nG * 128;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_words;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int st = static_cast<int>(idx & 3), lane = static_cast<int>((idx >> 2) & 31);
    const long long tg = idx >> 7;
    const int G = static_cast<int>(tg % nG), t = static_cast<int>(tg / nG);
    const int g = lane >> 2, t4 = lane & 3;
    const int r = t * 8 + g, kb = 64 * G + 16 * st + 2 * t4;
    const int rb = d / 2;
    const uint32_t w = nib_at(gq, rb, r, kb) | (nib_at(uq, rb, r, kb) << 4) | (nib_at(gq, rb, r, kb + 8) << 8) |
                       (nib_at(uq, rb, r, kb + 8) << 12) | (nib_at(gq, rb, r, kb + 1) << 16) |
                       (nib_at(uq, rb, r, kb + 1) << 20) | (nib_at(gq, rb, r, kb + 9) << 24) |
                       (nib_at(uq, rb, r, kb + 9) << 28);
    uint8_t* blk = dst + (static_cast<size_t>(t) * nG + G) * kGroupBytes;
    *reinterpret_cast<uint32_t*>(blk + lane * 16 + st * 4) = w;
    if (st == 0 && t4 == 0) {
      const size_t si = (static_cast<size_t>(r) * nG + G) * 2;
      uint16_t* o = reinterpret_cast<uint16_t*>(blk + kFragBytes + g * 8);
      o[0] = gsb[si];
      o[1] = gsb[si + 1];
      o[2] = usb[si];
      o[3] = usb[si + 1];
    }
  }
}

// Canonical down [d][f] -> device tiles (see internal.h).
__global__ void k_repack_dn(const uint8_t* dq, const uint16_t* dsb, int d, int f, uint8_t* dst) {
  const int nG = f / 64;
  const long long n_words = static_cast<long long>(d / 16) * nG * 128;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_words;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int st = static_cast<int>(idx & 3), lane = static_cast<int>((idx >> 2) & 31);
    const long long tg = idx >> 7;
    const int G = static_cast<int>(tg % nG), T = static_cast<int>(tg / nG);
    const int g = lane >> 2, t4 = lane & 3;
    const int R = T * 16 + g, kb = 64 * G + 16 * st + 2 * t4;
    const int rb = f / 2;
    const uint32_t w = nib_at(dq, rb, R, kb) | (nib_at(dq, rb, R + 8, kb) << 4) | (nib_at(dq, rb, R, kb + 8) << 8) |
                       (nib_at(dq, rb, R + 8, kb + 8) << 12) | (nib_at(dq, rb, R, kb + 1) << 16) |
                       (nib_at(dq, rb, R + 8, kb + 1) << 20) | (nib_at(dq, rb, R, kb + 9) << 24) |
                       (nib_at(dq, rb, R + 8, kb + 9) << 28);
    uint8_t* blk = dst + (static_cast<size_t>(T) * nG + G) * kGroupBytes;
    *reinterpret_cast<uint32_t*>(blk + lane * 16 + st * 4) = w;
    if (st == 0 && t4 == 0) {
      const size_t s0 = (static_cast<size_t>(R) * nG + G) * 2;
      const size_t s1 = (static_cast<size_t>(R + 8) * nG + G) * 2;
      uint16_t* o = reinterpret_cast<uint16_t*>(blk + kFragBytes + g * 8);
      o[0] = dsb[s0];
      o[1] = dsb[s0 + 1];
      o[2] = dsb[s1];
      o[3] = dsb[s1 + 1];
    }
  }
}

// ------------------------------------------------------------------ launchers

static cudaError_t launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          KParams* p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {p};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

size_t gateup_smem(int d) { return 128 + static_cast<size_t>(kGuWarps) * (d / 64) * kGroupBytes; }
size_t down_smem(int cg, int nb4) {
  return 128 + static_cast<size_t>(kDnWarps) * cg * kGroupBytes + static_cast<size_t>(kDnWarps) * cg * nb4 * 4 * 4;
}

int pick_nb(int B) { return B <= 8 ? 1 : 4; }
int pick_nb4(int B) { return B <= 4 ? 1 : 8; }

// Allow every kernel the device's opt-in shared-memory maximum; launches
// request only what their shapes need.
cudaError_t set_kernel_attrs(int max_smem) {
  const void* fns[] = {(const void*)k_gateup<1>, (const void*)k_gateup<4>, (const void*)k_down<1>,
                       (const void*)k_down<8>, (const void*)k_router};
  for (auto f : fns) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, f);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_router(KParams& p, int B, cudaStream_t s, bool pdl) {
  dim3 grid((p.E + 7) / 8, B);
  return launch((const void*)k_router, grid, dim3(256), static_cast<size_t>(p.d) * 2, s, pdl, &p);
}

cudaError_t launch_gateup(KParams& p, int B, int max_items, int n_sm, cudaStream_t s, bool pdl) {
  const int nb = pick_nb(B);
  const int want = (max_items + kGuWarps - 1) / kGuWarps;
  const int grid = want < 2 * n_sm ? want : 2 * n_sm;
  const void* fn = nb == 1 ? (const void*)k_gateup<1> : (const void*)k_gateup<4>;
  return launch(fn, dim3(grid > 0 ? grid : 1), dim3(kGuWarps * 32), gateup_smem(p.d), s, pdl, &p);
}

cudaError_t launch_down(KParams& p, int B, int max_items, int n_sm, cudaStream_t s, bool pdl) {
  const int nb4 = pick_nb4(B);
  const int want = (max_items + kDnWarps - 1) / kDnWarps;
  const int grid = want < 4 * n_sm ? want : 4 * n_sm;
  const void* fn = nb4 == 1 ? (const void*)k_down<1> : (const void*)k_down<8>;
  return launch(fn, dim3(grid > 0 ? grid : 1), dim3(kDnWarps * 32), down_smem(p.cg, nb4), s, pdl, &p);
}

namespace {

// Device-driven staging of a layer's misses (no host round trip): block row y
// copies the record of miss y from the pinned host pool, read through the host
// link as mapped memory, into its slot, eight 16-byte loads in flight per
// thread to cover the link's latency.  A malformed record sets ERR_PLAN and
// is skipped.
__global__ void __launch_bounds__(256) k_stage_misses(const int32_t* rec, const uint8_t* pool_layer, uint8_t* slots,
                                                      long long stride, long long n16, int E, int n_slots, int k,
                                                      uint32_t* err) {
  const int m = blockIdx.y;
  const int n_miss = rec[0];
  const bool lead = blockIdx.x == 0 && threadIdx.x == 0;
  if (n_miss < 0 || n_miss > k) {
    if (lead && m == 0) atomicOr(err, ERR_PLAN);
    return;
  }
  if (m >= n_miss) return;
  const int ex = rec[1 + 2 * m], slot = rec[2 + 2 * m];
  if (ex < 0 || ex >= E || slot < 0 || slot >= n_slots) {
    if (lead) atomicOr(err, ERR_PLAN);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(pool_layer + static_cast<long long>(ex) * stride);
  uint4* dst = reinterpret_cast<uint4*>(slots + static_cast<long long>(slot) * stride);
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 7 * step < n16; i += 8 * step) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = src[i + u * step];
#pragma unroll
    for (int u = 0; u < 8; ++u) dst[i + u * step] = v[u];
  }
  for (; i < n16; i += step) dst[i] = src[i];
}

// Reads n16 16-byte words of pinned host memory through the host link (the
// way the fused host-pool step reads its misses: plain loads, eight in flight
// per thread) and folds them into one word, so the reads cannot be dropped.
__global__ void __launch_bounds__(256) k_host_read(const uint4* src, long long n16, unsigned* sink) {
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  unsigned acc = 0;
  for (; i + 7 * step < n16; i += 8 * step) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = src[i + u * step];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += step) acc ^= src[i].x ^ src[i].y ^ src[i].z ^ src[i].w;
  if (acc == 0x9E3779B9u) atomicAdd(sink, 1u);   // almost never taken; keeps the loads
}

}  // namespace

cudaError_t launch_stage_misses(const int32_t* rec, const uint8_t* pool_layer, uint8_t* slots, long long stride,
                                long long bytes, int E, int n_slots, int k, uint32_t* err, int n_sm, cudaStream_t s) {
  if (bytes % 16 != 0 || stride % 16 != 0) return cudaErrorInvalidValue;
  int per_miss = 4 * n_sm / k;
  per_miss = per_miss < 1 ? 1 : (per_miss > 128 ? 128 : per_miss);
  k_stage_misses<<<dim3(per_miss, k), 256, 0, s>>>(rec, pool_layer, slots, stride, bytes / 16, E, n_slots, k, err);
  return cudaGetLastError();
}

cudaError_t launch_host_read(const void* src, long long bytes, unsigned* sink, int n_sm, cudaStream_t s) {
  if (bytes % 16 != 0) return cudaErrorInvalidValue;
  k_host_read<<<4 * n_sm, 256, 0, s>>>(static_cast<const uint4*>(src), bytes / 16, sink);
  return cudaGetLastError();
}

cudaError_t launch_repack(const uint8_t* gq, const uint16_t* gsb, const uint8_t* uq, const uint16_t* usb,
                          const uint8_t* dq, const uint16_t* dsb, int d, int f, uint8_t* dst, cudaStream_t s) {
  const size_t gu_bytes = static_cast<size_t>(f / 8) * (d / 64) * kGroupBytes;
  k_repack_gu<<<1024, 256, 0, s>>>(gq, gsb, uq, usb, d, f, dst);
  k_repack_dn<<<1024, 256, 0, s>>>(dq, dsb, d, f, dst + gu_bytes);
  return cudaGetLastError();
}

}  // namespace moe
