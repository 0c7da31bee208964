// Test shim: the expert file tier's host-only code (expert_file.cu) built with
// the host compiler, so its bookkeeping can be checked without a GPU.
#include <cstdint>

#include "expert_file.h"

extern "C" int shim_host_tier_lru_step(int n_rec, int32_t* expert_of_rec, long long* last_use,
                                       int32_t* rec_of_expert, const int32_t* ids, int n, long long t,
                                       int32_t* rec, int32_t* hit, int32_t* evicted, char* touched) {
  return moe::host_tier_lru_step(n_rec, expert_of_rec, last_use, rec_of_expert, ids, n, t, rec, hit, evicted,
                                 touched);
}
