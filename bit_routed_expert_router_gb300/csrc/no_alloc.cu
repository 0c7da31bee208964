// moe_route_noalloc: routing (logits, top-k, gates) that allocates nothing.
//
// Some callers cannot call cudaMalloc at the point where they need routing:
// hosts that reserve all device memory up front and forbid any allocation
// afterwards (a framework allocator with a hard budget, an embedded or
// real-time serving loop), because cudaMalloc can block, can synchronise the
// device and can fail under memory pressure at the worst moment.  This entry
// point serves them: the caller passes inputs and outputs, and the only
// global memory the kernel uses beyond them is a fixed file-scope device
// array, which every GPU that loads this library holds until the process
// exits.
//
// The arithmetic is the same as the router phase of moe_decode_step: optional
// RMS normalisation of h to bf16, exact fixed-point logits (every fp16 x bf16
// product rounded half-to-even onto the 2^-40 grid and summed in int64),
// top-k with ties to the lower expert index, softmax gates over the k picked.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "moe.h"

#include <climits>

namespace {

constexpr int kNaMaxB = MOE_ROUTE_NOALLOC_MAX_B;
constexpr int kNaMaxE = 256;

// Scratch: int64 logits [kNaMaxB][kNaMaxE] followed by one CTA counter per token.
// 131,328 bytes.  Shared by every call on a device; calls that overlap on the
// GPU race on it.
constexpr size_t kNaLogitBytes = sizeof(long long) * kNaMaxB * kNaMaxE;
constexpr size_t kNaScratchBytes = kNaLogitBytes + sizeof(int) * kNaMaxB;
static __device__ __align__(256) unsigned char g_route_scratch[kNaScratchBytes];

__global__ void __launch_bounds__(256) k_route_noalloc(const uint16_t* __restrict__ router_w,
                                                       const uint16_t* __restrict__ h, const float* bias, int d,
                                                       int E, int k, int prenorm, float eps, int32_t* ids,
                                                       float* gates, unsigned char* scratch) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm_raw);
  __shared__ float red[8];
  __shared__ int s_last;
  long long* logits = reinterpret_cast<long long*>(scratch);
  int* cnt = reinterpret_cast<int*>(scratch + kNaLogitBytes);
  const int b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint16_t* hb = h + static_cast<size_t>(b) * d;

  float ss = 0.f;
  for (int i = tid; i < d; i += 256) {
    const uint16_t v = hb[i];
    xs[i] = v;
    const float fv = moe::bf16_bits_to_float(v);
    ss += fv * fv;
  }
  if (prenorm) {
#pragma unroll
    for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float r = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
    for (int i = tid; i < d; i += 256) xs[i] = moe::float_to_bf16_bits(moe::bf16_bits_to_float(xs[i]) * r);
  }
  __syncthreads();

  const int e = blockIdx.x * 8 + warp;
  if (e < E) {
    const uint4* wr = reinterpret_cast<const uint4*>(router_w + static_cast<size_t>(e) * d);
    const uint4* xv4 = reinterpret_cast<const uint4*>(xs);
    long long acc = 0;
    for (int c = lane; c < d / 8; c += 32) {
      const uint4 wv = __ldg(wr + c);
      const uint4 xv = xv4[c];
      const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float pw = hh ? moe::half_hi(wa[i]) : moe::half_lo(wa[i]);
          const float px =
              moe::bf16_bits_to_float(static_cast<uint16_t>(hh ? (xa[i] >> 16) : (xa[i] & 0xFFFFu)));
          const float prod = pw * px;
          if (fabsf(prod) < 2048.f) acc += __float2ll_rn(prod * 1099511627776.0f);
        }
      }
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) acc += moe::shfl_xor_i64(acc, m);
    if (lane == 0) {
      if (bias) {
        const float bv = bias[static_cast<size_t>(b) * E + e];
        if (fabsf(bv) < 1048576.f) acc += __float2ll_rn(bv * 1099511627776.0f);
      }
      logits[static_cast<size_t>(b) * kNaMaxE + e] = acc;
      __threadfence();
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = (atomicAdd(&cnt[b], 1) == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();

  long long v[8];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ee = lane + 32 * i;
    v[i] = (ee < E) ? __ldcg(&logits[static_cast<size_t>(b) * kNaMaxE + ee]) : LLONG_MIN;
    if (ee >= E) taken |= 1u << i;
  }
  int my_id = 0;
  long long my_v = 0;
  for (int j = 0; j < k; ++j) {
    long long bv = LLONG_MIN;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ee = lane + 32 * i;
      if (!(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && ee < be))) {
        bv = v[i];
        be = ee;
      }
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) {
      const long long ov = moe::shfl_xor_i64(bv, m);
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
  if (lane < k) ex = expf(__ll2float_rn(my_v - top) * 9.094947017729282e-13f);
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
  if (lane < k) {
    ids[b * k + lane] = my_id;
    gates[b * k + lane] = ex / sum;
  }
}

// Device address of g_route_scratch, looked up once per device.
constexpr int kMaxDevices = 64;
std::mutex g_na_mutex;
unsigned char* g_na_ptr[kMaxDevices] = {};

}  // namespace

extern "C" moe_status moe_route_noalloc(const moe_config* cfg, const uint16_t* router_w, const void* h, int B,
                                        const float* logit_bias, int32_t* ids, float* gates, void* stream) {
  if (!cfg || !router_w || !h || !ids || !gates) return MOE_EINVAL;
  if (cfg->group != 64 || cfg->d <= 0 || cfg->d % 64 || cfg->d > 3072) return MOE_EINVAL;
  if (cfg->n_experts < 1 || cfg->n_experts > kNaMaxE) return MOE_EINVAL;
  if (cfg->top_k < 1 || cfg->top_k > cfg->n_experts || cfg->top_k > 32) return MOE_EINVAL;
  if (cfg->prenorm != 0 && cfg->prenorm != 1) return MOE_EINVAL;
  if (B < 1 || B > kNaMaxB) return MOE_EINVAL;
  // the kernel reads router rows and hidden rows 16 bytes at a time
  if ((reinterpret_cast<uintptr_t>(router_w) | reinterpret_cast<uintptr_t>(h)) & 15u) return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(gates) |
       reinterpret_cast<uintptr_t>(logit_bias)) & 3u)
    return MOE_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ECUDA;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (!g_na_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ECUDA;
      g_na_ptr[dev] = static_cast<unsigned char*>(p);
    }
    scratch = g_na_ptr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the per-token CTA counters must start at zero on every call
  if (cudaMemsetAsync(scratch + kNaLogitBytes, 0, sizeof(int) * B, s) != cudaSuccess) return MOE_ECUDA;
  dim3 grid((cfg->n_experts + 7) / 8, B);
  k_route_noalloc<<<grid, 256, static_cast<size_t>(cfg->d) * 2, s>>>(
      router_w, static_cast<const uint16_t*>(h), logit_bias, cfg->d, cfg->n_experts, cfg->top_k, cfg->prenorm,
      cfg->norm_eps, ids, gates, scratch);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}
