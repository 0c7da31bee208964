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

}  // namespace moe
