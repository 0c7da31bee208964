// Device-driven staging of host-pool misses (decode_kernels.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// Copies one layer's slot-cache misses from the pinned host pool into their
// slots on stream s: rec is the layer's miss record ([0] = n_miss, then
// (expert, slot) pairs, written by the router kernel), pool_layer the layer's
// records in mapped pinned host memory, at `stride` bytes; bytes % 16 == 0.
// A malformed record sets ERR_PLAN in *err and is skipped.
cudaError_t launch_stage_misses(const int32_t* rec, const uint8_t* pool_layer, uint8_t* slots, long long stride,
                                long long bytes, int E, int n_slots, int k, uint32_t* err, int n_sm, cudaStream_t s);

// Reads `bytes` (a multiple of 16) of pinned host memory at src through the
// host link with plain loads from every SM (the fused host-pool step's read
// pattern); sink is a device word the reads are folded into.
cudaError_t launch_host_read(const void* src, long long bytes, unsigned* sink, int n_sm, cudaStream_t s);

}  // namespace moe
