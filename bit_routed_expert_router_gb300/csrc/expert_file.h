// Expert file tier (host): bounded parallel pread / pwrite (expert_file.cu).
#pragma once

#include <cstdint>

namespace moe {

struct FilePool;

int pio_all(int fd, bool write, uint64_t offset, void* buf, uint64_t bytes);
FilePool* file_pool_create(int n_threads);   // null if its threads cannot be started
void file_pool_destroy(FilePool* fp);
// One transfer of [offset, offset + bytes) split into `chunk`-byte pieces over
// the pool's threads; returns 0 or an errno value.
int file_pool_transfer(FilePool* fp, int fd, bool write, uint64_t offset, void* buf, uint64_t bytes, uint64_t chunk);

// The host tier's bookkeeping for one layer (the slot cache's LRU rules one
// level down).  expert_of_rec[n_rec] (-1 = empty), last_use[n_rec] (-1 =
// empty), rec_of_expert[E] (-1 = not held); ids[0..n) are the step's requests
// (the slot cache's misses, distinct, in top-k order), t the step counter,
// touched[n_rec] scratch.  Requests the tier holds refresh their record
// (last_use = t, hit[m] = 1); the others, in order, take the record with the
// smallest (last_use, index) among those the step has not touched (hit[m] = 0,
// evicted[m] = the expert it held or -1).  rec[m] is the record holding ids[m]
// afterwards.  Returns the number of non-hits, or -1 if n > n_rec.
int host_tier_lru_step(int n_rec, int32_t* expert_of_rec, long long* last_use, int32_t* rec_of_expert,
                       const int32_t* ids, int n, long long t, int32_t* rec, int32_t* hit, int32_t* evicted,
                       char* touched);

}  // namespace moe
