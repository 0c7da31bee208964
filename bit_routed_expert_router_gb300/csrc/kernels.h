// Launchers of the libmoe kernels (host side).
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

constexpr int kGuWarps = 4;     // warps per gate/up CTA, one row tile each
constexpr int kDnWarps = 8;     // warps per down CTA
constexpr int kMaxDecodeB = 32; // tokens per decode launch

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
