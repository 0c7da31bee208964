// Small-batch grouped GEMVs of libmoe (sm_103a): the routed-MoE FFN of at most
// 32 tokens, after the prefill path's routing and expert grouping.
//
// With a few tokens per expert every int4 weight is used once or twice, so the
// layer is bound by reading and unpacking weights, not by multiply throughput
// (TurboFieldfare write-up, "Splitting the work improved attention and
// prefill": the batched routed MoE).  The tcgen05 grouped GEMM writes every
// dequantised fp16 tile into tensor memory before it multiplies; here the
// weights go from a shared-memory ring straight into mma.sync A fragments
// (nibbles OR-ed under the fp16 exponent of 1024, the affine of each group
// applied in fp32), and the tokens of an expert fill the eight B columns of
// m16n8k16.  Two launches per layer:
//   SG_GU  gate/up tiles (8 gate + 8 up rows over d) of the shared expert, for
//          all T tokens, and of every active expert, for the tokens of its
//          pairs (the x rows of those tokens, which the prefill path's norm
//          step writes per token, read through the expert-ordered pair list):
//          a = GELU(gate) * up rounded to fp16, in expert order and in the
//          fragment order the down launch reads;
//   SG_DN  down tiles: per stage the shared expert's 16-row tile over all f_s
//          columns, or an active expert's 16-row tiles over its f columns
//          (as many as one ring slot holds); outputs per token (shared) and per
//          (token, top-k position) pair (routed), which the prefill combine
//          adds in top-k order with the residual.
// Both are persistent, as the write-up's routed-MoE kernel kept its
// workgroups resident until the whole dispatch was done (section "MoE needed
// parallel work, reuse, and coarse overlap"): one CTA per SM takes the shared
// expert's stages dealt round robin and then a contiguous range of the routed
// stages; a producer lane streams the CTA's stages into a ring of
// shared-memory slots with 1-D bulk copies; four quads of four consumer warps
// take them in turn (stage j to quad j mod 4).  Within a quad the warps
// split the int4 groups of a tile and the last one to finish adds the four
// partials in warp order (deterministic), except for routed down stages,
// where each warp owns whole 16-row tiles.
//
// B operands are rows in fragment order: for each 64-element group G and lane
// quarter t4 eight 32-bit words (k16 step st, half h) holding elements
// 64 G + 16 st + 8 h + 2 t4 + {0, 1}, so a lane loads its fragments of one
// group as two 16-byte words.  The group sums that the affine needs come from
// the x rows' precomputed sums (gate/up) or from one more MMA with an all-ones
// A operand (down: column sums of a), so no atomics enter any sum.  The unpack
// of the int4 words and the MMA are one asm block (mma_nib, common.cuh).
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kNC = 16;                       // consumer warps
constexpr int kQW = 4;                        // warps per quad
constexpr int kNQ = kNC / kQW;
constexpr int kNS = 6;                        // ring slots
constexpr int kXcBytes = 12 * 64 * kSgMaxG * 2; // B-row cache: twelve x rows of d = 2816 (or more, shorter rows)
constexpr int kXcItems = 8;                   // experts the cache holds rows of
constexpr int kSlotBytes = kSgMaxG * kGroupBytes;
constexpr int kMaxNB = kSgMaxT / 8;           // blocks of eight token columns
constexpr int kThreads = 32 * (kNC + 1);
constexpr unsigned kFull = 0xFFFFFFFFu;
#ifndef SG_UNROLL
#define SG_UNROLL 4
#endif
constexpr int kUnroll = SG_UNROLL;            // int4 groups a warp's loop keeps in flight

struct Smem {
  alignas(128) uint8_t ring[kNS][kSlotBytes];
  alignas(128) uint8_t xc[kXcBytes];            // B rows (and, gate/up, their group sums) of the CTA's experts
  alignas(16) float xcg[kXcBytes / 128];        // group sums of cached x rows (one float per 64 fp16)
  alignas(8) uint64_t xbar;                     // the cache is filled
  int xc_item[kXcItems];                        // routed item whose rows the cache holds
  int xc_off[kXcItems];                         // their byte offset in xc (row r of the item at + r * row bytes)
  int n_xc;
  alignas(8) uint64_t full[kNS];
  alignas(8) uint64_t empty[kNS];
  int cnt[kNS];
};
static_assert(sizeof(Smem) + 128 <= 227 * 1024, "shared memory per CTA");
static_assert(offsetof(Smem, ring) % 128 == 0 && kSlotBytes % 16 == 0, "bulk copy targets");

enum : int { ST_GU = 0, ST_DN_SHARED = 1, ST_DN_ROUTED = 2 };

struct Stage {
  const uint8_t* src;
  int bytes;
  int kind;
  int tile;       // gate/up: tile index (intermediate rows 8 tile .. + 7); down: first 16-row tile
  int nrt;        // routed down: 16-row tiles in the stage
  int row0;       // routed: first row of the expert in the expert-ordered matrices
  int ntok;       // token columns
  int item;       // routed: the item (active expert) index
};

__device__ __forceinline__ int routed_rt(const SgParams& p) { return min(p.d / 16, kSgMaxG / (p.f / 64)); }

// Stages of the launch: nS of the shared expert, then nR of the active experts.
__device__ __forceinline__ void n_stages(const SgParams& p, int n_items, int& nS, int& nR) {
  if (p.mode == SG_GU) {
    nS = p.fs / 8;
    nR = n_items * (p.f / 8);
    return;
  }
  const int R = p.d / 16, rt = routed_rt(p);
  nS = R;
  nR = n_items * ((R + rt - 1) / rt);
}

// The CTA's stages: the shared ones dealt round robin over the CTAs (each
// multiplies all T tokens), then a contiguous range of the routed ones, so
// consecutive stages of a CTA mostly belong to one expert and its token rows
// stay in the L1 cache.
struct CtaStages {
  int nS, G, c, n_sh, r0, n;
  __device__ int stage(int j) const { return j < n_sh ? c + j * G : nS + r0 + (j - n_sh); }
};
__device__ __forceinline__ CtaStages cta_stages(const SgParams& p, int n_items) {
  CtaStages cs;
  int nR;
  n_stages(p, n_items, cs.nS, nR);
  cs.G = static_cast<int>(gridDim.x);
  cs.c = static_cast<int>(blockIdx.x);
  cs.n_sh = cs.c < cs.nS ? (cs.nS - cs.c + cs.G - 1) / cs.G : 0;
  cs.r0 = static_cast<int>(static_cast<long long>(nR) * cs.c / cs.G);
  const int r1 = static_cast<int>(static_cast<long long>(nR) * (cs.c + 1) / cs.G);
  cs.n = cs.n_sh + (r1 - cs.r0);
  return cs;
}

// Stage s of the launch (the same on the producer and the consumer side).
__device__ Stage stage_of(const SgParams& p, int s) {
  const int nGd = p.d / 64, nGf = p.f / 64, nGs = p.fs / 64;
  Stage st;
  st.nrt = 1;
  st.item = -1;
  if (p.mode == SG_GU) {
    const int nS = p.fs / 8, per = p.f / 8;
    const int tile_bytes = nGd * kGroupBytes;
    st.kind = ST_GU;
    st.bytes = tile_bytes;
    if (s < nS) {
      st.tile = s;
      st.row0 = -1;
      st.ntok = p.T;
      st.src = p.shared + static_cast<size_t>(s) * tile_bytes;
    } else {
      const int u = (s - nS) / per;
      st.item = u;
      st.tile = (s - nS) - u * per;
      const int e = __ldg(&p.items[3 * u]);
      st.row0 = __ldg(&p.items[3 * u + 1]);
      st.ntok = __ldg(&p.items[3 * u + 2]);
      st.src = p.experts + static_cast<long long>(e) * p.stride + static_cast<size_t>(st.tile) * tile_bytes;
    }
    return st;
  }
  const int R = p.d / 16, rt = routed_rt(p), per = (R + rt - 1) / rt;
  if (s < R) {
    const size_t gu_s = static_cast<size_t>(p.fs / 8) * nGd * kGroupBytes;
    st.kind = ST_DN_SHARED;
    st.tile = s;
    st.row0 = -1;
    st.ntok = p.T;
    st.bytes = nGs * kGroupBytes;
    st.src = p.shared + gu_s + static_cast<size_t>(s) * nGs * kGroupBytes;
  } else {
    const size_t gu_r = static_cast<size_t>(p.f / 8) * nGd * kGroupBytes;
    const int u = (s - R) / per, i = (s - R) - u * per;
    st.item = u;
    const int e = __ldg(&p.items[3 * u]);
    st.kind = ST_DN_ROUTED;
    st.tile = i * rt;
    st.nrt = min(rt, R - st.tile);
    st.row0 = __ldg(&p.items[3 * u + 1]);
    st.ntok = __ldg(&p.items[3 * u + 2]);
    st.bytes = st.nrt * nGf * kGroupBytes;
    st.src = p.experts + static_cast<long long>(e) * p.stride + gu_r + static_cast<size_t>(st.tile) * nGf * kGroupBytes;
  }
  return st;
}

// Bounded wait on a local mbarrier phase by a whole warp (the lanes decide
// together); false after about two seconds, with the error word flagged.
__device__ bool wait_warp(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(kFull, clock64() - t0 > kSpinLimitCycles)) {
      if ((threadIdx.x & 31) == 0) atomicOr(err, ERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Groups [G0, G1) of 16 weight rows (`blk`: the slot block of group G0, one
// 576-byte block per group) times eight token columns of the B rows: `brow` is
// this lane's column (fragment order), `xg0` / `xg1` the rows of group sums of
// the lane's two accumulator columns 2 t4, 2 t4 + 1.  Columns past the last
// token repeat a valid row; their results are never used.  Returns the lane's
// sums (row g, column 2 t4), (row g, 2 t4 + 1), (row g + 8, 2 t4),
// (row g + 8, 2 t4 + 1), each s P + (b - 1024 s) X for the rows held as
// 1024 + q and (s / 16) P + (b - 64 s) X for those held as 1024 + 16 q, X the
// column's group sum: from xg, or with kOnesSum from an MMA of the B columns
// with an all-ones A operand.  kSmemB: the B rows and sums are in this CTA's
// cache in shared memory (else global memory, read through the L1 cache).
// m16n8k16 fp16 MMA without the volatile qualifier, so the compiler may
// interleave the MMAs of several groups.
__device__ __forceinline__ void mma16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with a zero accumulator in (one zero register for all four inputs).
__device__ __forceinline__ void mma16z(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

template <bool kOnesSum, bool kSmemB>
__device__ __forceinline__ float4 tile_dot(const uint8_t* blk, int G0, int G1, const uint4* brow, const float* xg0,
                                           const float* xg1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
  const uint32_t one[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};   // fp16 1.0 pairs
  const uint8_t* wq = blk + lane * 16;
  const uint8_t* ws = blk + kFragBytes + g * 8;
  const uint4* bp = brow + (G0 * 4 + t4) * 2;
#pragma unroll kUnroll
  for (int G = G0; G < G1; ++G) {
    const uint4 q = *reinterpret_cast<const uint4*>(wq);
    const uint2 sbv = *reinterpret_cast<const uint2*>(ws);
    const uint4 x01 = kSmemB ? bp[0] : __ldg(bp), x23 = kSmemB ? bp[1] : __ldg(bp + 1);
    wq += kGroupBytes;
    ws += kGroupBytes;
    bp += 8;
    float X0 = 0.f, X1 = 0.f;
    if (!kOnesSum) {
      X0 = kSmemB ? xg0[G] : __ldg(xg0 + G);
      X1 = kSmemB ? xg1[G] : __ldg(xg1 + G);
    }
    float c0[4], c1[4];
    mma_nib<true>(c0, q.x, x01.x, x01.y);
    mma_nib<true>(c1, q.y, x01.z, x01.w);
    mma_nib<false>(c0, q.z, x23.x, x23.y);
    mma_nib<false>(c1, q.w, x23.z, x23.w);
    if (kOnesSum) {   // column sums of B: two chains of two MMAs
      float s0[4], s1[4];
      mma16z(s0, one, x01.x, x01.y);
      mma16z(s1, one, x01.z, x01.w);
      mma16(s0, one, x23.x, x23.y);
      mma16(s1, one, x23.z, x23.w);
      X0 = s0[0] + s1[0];
      X1 = s0[1] + s1[1];
    }
    const float sA = half_lo(sbv.x), oA = half_hi(sbv.x), sB = half_lo(sbv.y), oB = half_hi(sbv.y);
    const float bA = fmaf(-1024.f, sA, oA), bB = fmaf(-64.f, sB, oB), sB16 = sB * 0.0625f;
    r0 += sA * (c0[0] + c1[0]) + bA * X0;
    r1 += sA * (c0[1] + c1[1]) + bA * X1;
    r2 += sB16 * (c0[2] + c1[2]) + bB * X0;
    r3 += sB16 * (c0[3] + c1[3]) + bB * X1;
  }
  return make_float4(r0, r1, r2, r3);
}

__device__ __forceinline__ float gelu_of(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

// Position (fp16 elements) of element i of a row in fragment order.
__device__ __forceinline__ int frag_pos(int i) {
  const int G = i >> 6, w = i & 63, st = w >> 4, h = (w >> 3) & 1, t4 = (w & 7) >> 1;
  return ((((G * 4 + t4) * 4 + st) * 2 + h) << 1) | (w & 1);
}

// Where warp qw of the quad leaves its partial sums of token block nb (32
// lanes x float4) in the slot it has multiplied: behind the stage's weights
// when the slot has room there for every warp's blocks, else inside the
// warp's own groups (then at least six, 3,456 bytes), which only this warp
// reads and has finished reading.
constexpr int kPartBytes = 32 * 16;
__device__ __forceinline__ float4* part_at(Smem& S, int slot, int nG, int G0, int qw, int nb) {
  uint8_t* base = S.ring[slot];
  if (nG * kGroupBytes + kQW * kMaxNB * kPartBytes <= kSlotBytes)
    return reinterpret_cast<float4*>(base + kSlotBytes - kQW * kMaxNB * kPartBytes + (qw * kMaxNB + nb) * kPartBytes);
  return reinterpret_cast<float4*>(base + static_cast<size_t>(G0) * kGroupBytes + nb * kPartBytes);
}

// Byte offset of routed item u's B rows in the CTA's cache, or -1.
__device__ __forceinline__ int xc_find(const Smem& S, int u) {
  for (int i = 0; i < S.n_xc; ++i)
    if (S.xc_item[i] == u) return S.xc_off[i];
  return -1;
}

// The results of token block nb of a split stage: a = GELU(gate) * up in fp16
// at its fragment-order place (gate/up), or the shared expert's output rows
// (down).  r holds (row g, column c0), (row g, c0 + 1), (row g + 8, c0),
// (row g + 8, c0 + 1), c0 = nb * 8 + 2 t4.
__device__ __forceinline__ void emit(const SgParams& p, const Stage& st, bool gu, int nb, float4 r) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int c0 = nb * 8 + 2 * t4;
  if (gu) {
    // gate row g (r.x, r.y) and up row g (r.z, r.w) of intermediate row 8 tile + g
    const int i = 8 * st.tile + g, F = st.row0 >= 0 ? p.f : p.fs;
    uint16_t* av = st.row0 >= 0 ? p.av_r + static_cast<size_t>(st.row0) * p.f : p.av_s;
    const float a0 = gelu_of(r.x, p.gelu) * r.z, a1 = gelu_of(r.y, p.gelu) * r.w;
    const bool v0 = c0 < st.ntok, v1 = c0 + 1 < st.ntok;
    if ((v0 && !(fabsf(a0) < 65504.f)) || (v1 && !(fabsf(a1) < 65504.f))) atomicOr(p.err, ERR_PF_RANGE);
    const int pos = frag_pos(i);
    if (v0) av[static_cast<size_t>(c0) * F + pos] = __half_as_ushort(__float2half_rn(a0));
    if (v1) av[static_cast<size_t>(c0 + 1) * F + pos] = __half_as_ushort(__float2half_rn(a1));
  } else {
    const int row = 16 * st.tile + g;
    if (c0 < st.ntok) {
      p.y_s[static_cast<size_t>(c0) * p.d + row] = r.x;
      p.y_s[static_cast<size_t>(c0) * p.d + row + 8] = r.z;
    }
    if (c0 + 1 < st.ntok) {
      p.y_s[static_cast<size_t>(c0 + 1) * p.d + row] = r.y;
      p.y_s[static_cast<size_t>(c0 + 1) * p.d + row + 8] = r.w;
    }
  }
}

// One token block of a split stage over groups [G0, G1): B rows from the
// CTA's cache (routed gate/up whose rows it holds) or global memory.
__device__ __forceinline__ float4 split_block(const SgParams& p, Smem& S, const Stage& st, bool gu, int xoff,
                                             const uint8_t* blk, int G0, int G1, int nb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  // columns past the last token repeat its row (their results are not used)
  const int last_col = st.ntok - 1;
  const int col = min(nb * 8 + g, last_col), c0 = min(nb * 8 + 2 * t4, last_col), c1 = min(c0 + 1, last_col);
  if (xoff >= 0) {   // routed gate/up with its x rows (and sums) in the cache
    const int rb = p.d * 2;
    const uint4* brow = reinterpret_cast<const uint4*>(S.xc + xoff + col * rb);
    return tile_dot<false, true>(blk, G0, G1, brow, S.xcg + (xoff + c0 * rb) / 128, S.xcg + (xoff + c1 * rb) / 128);
  }
  // gate/up: the token rows of x (an active expert's column c is the token of
  // its pair row0 + c; the shared expert's column c is token c); down: the
  // shared a rows
  if (gu) {
    const int k = p.P / p.T;
    const int tc = st.row0 >= 0 ? __ldg(&p.row_pair[st.row0 + col]) / k : col;
    const int t0 = st.row0 >= 0 ? __ldg(&p.row_pair[st.row0 + c0]) / k : c0;
    const int t1 = st.row0 >= 0 ? __ldg(&p.row_pair[st.row0 + c1]) / k : c1;
    const uint4* brow = reinterpret_cast<const uint4*>(p.xv + static_cast<size_t>(tc) * p.d);
    const int nGd = p.d / 64;
    return tile_dot<false, false>(blk, G0, G1, brow, p.xg + static_cast<size_t>(t0) * nGd,
                                  p.xg + static_cast<size_t>(t1) * nGd);
  }
  const uint4* brow = reinterpret_cast<const uint4*>(p.av_s + static_cast<size_t>(col) * p.fs);
  return tile_dot<true, false>(blk, G0, G1, brow, nullptr, nullptr);
}

// A stage of 16 weight rows over nG int4 groups (gate/up tiles and shared down
// tiles).  With four blocks of token columns each warp of the quad takes one
// block over every group and writes its results; otherwise the warps split the
// groups ([qw * cg, (qw + 1) * cg)) for every block, and the last warp to
// finish adds the four partials in warp order and writes the results.
__device__ void stage_split(const SgParams& p, Smem& S, int slot, const Stage& st, int qw) {
  const int lane = threadIdx.x & 31;
  const bool gu = st.kind == ST_GU;
  const int nG = gu ? p.d / 64 : p.fs / 64;
  const int nbu = (st.ntok + 7) >> 3;
  const int xoff = gu && st.row0 >= 0 ? xc_find(S, st.item) : -1;
  if (nbu == kQW) {
    emit(p, st, gu, qw, split_block(p, S, st, gu, xoff, S.ring[slot], 0, nG, qw));
    return;
  }
  const int cg = (nG + kQW - 1) / kQW, G0 = min(nG, qw * cg), G1 = min(nG, G0 + cg);
  const uint8_t* blk = S.ring[slot] + static_cast<size_t>(G0) * kGroupBytes;
  float4 rr[kMaxNB];
#pragma unroll
  for (int nb = 0; nb < kMaxNB; ++nb) {
    rr[nb] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nb < nbu) rr[nb] = split_block(p, S, st, gu, xoff, blk, G0, G1, nb);
  }
  // every read of this warp's groups is done: its partials may overwrite them
  __syncwarp();
#pragma unroll
  for (int nb = 0; nb < kMaxNB; ++nb)
    if (nb < nbu) part_at(S, slot, nG, G0, qw, nb)[lane] = rr[nb];
  fence_proxy_async_smem();   // generic writes into a bulk-copy target, before the slot is refilled
  __threadfence_block();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&S.cnt[slot], 1) == kQW - 1;
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __threadfence_block();
  for (int nb = 0; nb < nbu; ++nb) {
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kQW; ++w) {
      const int Gw = min(nG, w * cg);
      const volatile float* v = reinterpret_cast<const volatile float*>(part_at(S, slot, nG, Gw, w, nb) + lane);
      r.x += v[0];
      r.y += v[1];
      r.z += v[2];
      r.w += v[3];
    }
    emit(p, st, gu, nb, r);
  }
  __syncwarp();
  if (lane == 0) S.cnt[slot] = 0;
}

// Routed down stage: warp qw owns the stage's 16-row tiles qw, qw + 4, ...
// over all f/64 groups; outputs go to the rows of the tokens' pairs.
__device__ void stage_down_routed(const SgParams& p, Smem& S, int slot, const Stage& st, int qw) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nGf = p.f / 64, nbu = (st.ntok + 7) >> 3;
  const int xoff = xc_find(S, st.item);
  for (int j = qw; j < st.nrt; j += kQW) {
    const uint8_t* blk = S.ring[slot] + static_cast<size_t>(j) * nGf * kGroupBytes;
    const int row = 16 * (st.tile + j) + g;
    for (int nb = 0; nb < nbu; ++nb) {
      const int col = min(nb * 8 + g, st.ntok - 1), c0 = nb * 8 + 2 * t4;   // past the last token: its row again
      float4 r;
      if (xoff >= 0) {
        r = tile_dot<true, true>(blk, 0, nGf, reinterpret_cast<const uint4*>(S.xc + xoff + col * p.f * 2), nullptr,
                                 nullptr);
      } else {
        const uint4* brow = reinterpret_cast<const uint4*>(p.av_r + static_cast<size_t>(st.row0 + col) * p.f);
        r = tile_dot<true, false>(blk, 0, nGf, brow, nullptr, nullptr);
      }
      if (c0 < st.ntok) {
        float* y = p.y_r + static_cast<size_t>(__ldg(&p.row_pair[st.row0 + c0])) * p.d;
        y[row] = r.x;
        y[row + 8] = r.z;
      }
      if (c0 + 1 < st.ntok) {
        float* y = p.y_r + static_cast<size_t>(__ldg(&p.row_pair[st.row0 + c0 + 1])) * p.d;
        y[row] = r.y;
        y[row + 8] = r.w;
      }
    }
  }
}

// The producer lane fills the CTA's B-row cache: the rows of the active
// experts its routed stages belong to (x rows and their group sums for gate/up,
// rows of a for down), as many whole experts as fit, with bulk copies that
// complete on xbar.
__device__ void fill_cache(const SgParams& p, Smem& S, const CtaStages& cs) {
  const bool gu = p.mode == SG_GU;
  const int nGd = p.d / 64;
  const int rb = gu ? p.d * 2 : p.f * 2;                        // bytes per row
  int per;
  if (gu) {
    per = p.f / 8;
  } else {
    const int R = p.d / 16, rt = routed_rt(p);
    per = (R + rt - 1) / rt;
  }
  const int nr = cs.n - cs.n_sh;                                 // routed stages of the CTA
  int n = 0, used = 0;
  uint32_t bytes = 0;
  // gate/up sums are copied too, which needs 16-byte aligned rows of them
  if (nr > 0 && (!gu || nGd % 4 == 0)) {
    const int u0 = cs.r0 / per, u1 = (cs.r0 + nr - 1) / per;
    for (int u = u0; u <= u1 && n < kXcItems; ++u) {
      const int rows = __ldg(&p.items[3 * u + 2]);
      if (used + rows * rb > kXcBytes) break;
      S.xc_item[n] = u;
      S.xc_off[n] = used;
      ++n;
      used += rows * rb;
      bytes += static_cast<uint32_t>(rows * rb + (gu ? rows * nGd * 4 : 0));
    }
  }
  S.n_xc = n;
  mbar_arrive_expect_tx(&S.xbar, bytes);   // release: the table above is visible to the waiters
  for (int i = 0; i < n; ++i) {
    const int u = S.xc_item[i], row0 = __ldg(&p.items[3 * u + 1]), rows = __ldg(&p.items[3 * u + 2]);
    if (!gu) {   // the item's rows of a, contiguous in expert order
      bulk_g2s(S.xc + S.xc_off[i], reinterpret_cast<const uint8_t*>(p.av_r) + static_cast<size_t>(row0) * rb,
               static_cast<uint32_t>(rows * rb), &S.xbar);
      continue;
    }
    // gate/up: the x rows (and group sums) of the item's tokens, one copy each
    const int k = p.P / p.T;
    for (int c = 0; c < rows; ++c) {
      const int tok = __ldg(&p.row_pair[row0 + c]) / k;
      bulk_g2s(S.xc + S.xc_off[i] + c * rb, reinterpret_cast<const uint8_t*>(p.xv) + static_cast<size_t>(tok) * rb,
               static_cast<uint32_t>(rb), &S.xbar);
      bulk_g2s(S.xcg + (S.xc_off[i] + c * rb) / 128, p.xg + static_cast<size_t>(tok) * nGd,
               static_cast<uint32_t>(nGd * 4), &S.xbar);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_small_batch(SgParams p) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the ring at a 128-byte boundary (the allocation has 128 bytes to spare)
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kQW);
      S.cnt[i] = 0;
    }
    mbar_init(&S.xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const CtaStages cs = cta_stages(p, *p.n_items);
  if (warp == kNC) {
    // producer: the B-row cache, then the CTA's stages j = 0, 1, ... in order
    if (lane != 0) return;
    fill_cache(p, S, cs);
    int j = 0;
    for (; j < cs.n; ++j) {
      const int slot = j % kNS;
      if (!mbar_wait_bounded(&S.empty[slot], ((j / kNS) & 1u) ^ 1u, p.err)) break;
      const Stage st = stage_of(p, cs.stage(j));
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(st.bytes));
      bulk_g2s(S.ring[slot], st.src, static_cast<uint32_t>(st.bytes), &S.full[slot]);
    }
    // copies still in flight complete before the CTA leaves (bounded)
    for (int v = max(0, j - kNS); v < j; ++v) mbar_wait_bounded(&S.full[v % kNS], (v / kNS) & 1u, p.err);
    mbar_wait_bounded(&S.xbar, 0u, p.err);
    return;
  }
  const int quad = warp / kQW, qw = warp % kQW;
  bool cache_ready = false;
  for (int j = quad; j < cs.n; j += kNQ) {
    const int slot = j % kNS;
    if (!wait_warp(&S.full[slot], (j / kNS) & 1u, p.err)) return;
    const Stage st = stage_of(p, cs.stage(j));
    if (st.item >= 0 && !cache_ready) {   // the first routed stage of this warp: the cache must be complete
      if (!wait_warp(&S.xbar, 0u, p.err)) return;
      cache_ready = true;
    }
    if (st.kind == ST_DN_ROUTED) stage_down_routed(p, S, slot, st, qw);
    else stage_split(p, S, slot, st, qw);
    __syncwarp();
    if (lane == 0) mbarrier_arrive(&S.empty[slot]);
  }
}

}  // namespace

bool sg_shape_ok(int d, int f, int fs) {
  return d % 64 == 0 && f % 64 == 0 && fs % 64 == 0 && d / 64 <= kSgMaxG && fs / 64 <= kSgMaxG &&
         f / 64 <= kSgMaxG && d >= 16;
}

size_t sg_smem() { return sizeof(Smem) + 128; }

cudaError_t sg_set_attrs() {
  return cudaFuncSetAttribute((const void*)k_small_batch, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sg_smem()));
}

cudaError_t launch_sg(const SgParams& p, int n_sm, cudaStream_t s) {
  return launch_chain(k_small_batch, dim3(n_sm), dim3(kThreads), sg_smem(), s, p);
}

}  // namespace moe
