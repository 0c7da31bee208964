// Expert file tier: bounded parallel pread / pwrite of expert records.
//
// The TurboFieldfare write-up streams routed experts from the model file with
// explicit reads ("Explicit reads made expert streaming work": each miss is
// read with a bounded number of parallel pread calls into the layer's slot,
// instead of relying on memory-mapped page faults).  Here the file holds every
// (layer, expert) record in the device layout at a 4096-byte stride; a miss is
// read in chunks by a small persistent pool of host threads into pinned
// staging memory, from which the staging copy to the device slot is issued.
//
// Host code only (no kernels).
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cerrno>
#include <condition_variable>
#include <cstdint>
#include <mutex>
#include <thread>
#include <vector>

#include "expert_file.h"
#include "moe.h"

namespace moe {

// Reads or writes [offset, offset + bytes) in full (restarting after short
// transfers and EINTR).  Returns 0, or an errno value (EIO for a transfer that
// ended early at end of file).
int pio_all(int fd, bool write, uint64_t offset, void* buf, uint64_t bytes) {
  uint8_t* p = static_cast<uint8_t*>(buf);
  while (bytes > 0) {
    const ssize_t n = write ? ::pwrite(fd, p, static_cast<size_t>(bytes), static_cast<off_t>(offset))
                            : ::pread(fd, p, static_cast<size_t>(bytes), static_cast<off_t>(offset));
    if (n < 0) {
      if (errno == EINTR) continue;
      return errno;
    }
    if (n == 0) return EIO;
    p += n;
    offset += static_cast<uint64_t>(n);
    bytes -= static_cast<uint64_t>(n);
  }
  return 0;
}

// A fixed set of worker threads; run() splits one transfer into chunks, hands
// them out and returns when all are done (the calling thread works too).
struct FilePool {
  explicit FilePool(int n_threads) {
    for (int i = 0; i + 1 < n_threads; ++i) workers.emplace_back([this] { loop(); });
  }
  ~FilePool() {
    {
      std::lock_guard<std::mutex> g(mu);
      stop = true;
    }
    cv.notify_all();
    for (auto& t : workers) t.join();
  }

  int run(int fd, bool write, uint64_t offset, void* buf, uint64_t bytes, uint64_t chunk) {
    std::unique_lock<std::mutex> g(mu);
    job_fd = fd;
    job_write = write;
    job_off = offset;
    job_buf = static_cast<uint8_t*>(buf);
    job_bytes = bytes;
    job_chunk = chunk > 0 ? chunk : bytes;
    next = 0;
    n_chunks = bytes == 0 ? 0 : (bytes + job_chunk - 1) / job_chunk;
    done = 0;
    err = 0;
    ++generation;
    cv.notify_all();
    g.unlock();
    work();
    g.lock();
    done_cv.wait(g, [this] { return done == n_chunks; });
    return err;
  }

 private:
  void loop() {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> g(mu);
    for (;;) {
      cv.wait(g, [&] { return stop || generation != seen; });
      if (stop) return;
      seen = generation;
      g.unlock();
      work();
      g.lock();
    }
  }

  // Takes chunks until none is left.
  void work() {
    for (;;) {
      uint64_t i;
      {
        std::lock_guard<std::mutex> g(mu);
        if (next >= n_chunks) return;
        i = next++;
      }
      const uint64_t o = i * job_chunk;
      const uint64_t n = o + job_chunk <= job_bytes ? job_chunk : job_bytes - o;
      const int e = pio_all(job_fd, job_write, job_off + o, job_buf + o, n);
      std::lock_guard<std::mutex> g(mu);
      if (e != 0 && err == 0) err = e;
      if (++done == n_chunks) done_cv.notify_all();
    }
  }

  std::vector<std::thread> workers;
  std::mutex mu;
  std::condition_variable cv, done_cv;
  bool stop = false;
  uint64_t generation = 0;
  int job_fd = -1;
  bool job_write = false;
  uint64_t job_off = 0, job_bytes = 0, job_chunk = 0, next = 0, n_chunks = 0, done = 0;
  uint8_t* job_buf = nullptr;
  int err = 0;
};

int host_tier_lru_step(int n_rec, int32_t* expert_of_rec, long long* last_use, int32_t* rec_of_expert,
                       const int32_t* ids, int n, long long t, int32_t* rec, int32_t* hit, int32_t* evicted,
                       char* touched) {
  if (n > n_rec) return -1;
  for (int i = 0; i < n_rec; ++i) touched[i] = 0;
  for (int m = 0; m < n; ++m) {
    const int r = rec_of_expert[ids[m]];
    hit[m] = r >= 0;
    evicted[m] = -1;
    rec[m] = r;
    if (r >= 0) {
      last_use[r] = t;
      touched[r] = 1;
    }
  }
  int n_new = 0;
  for (int m = 0; m < n; ++m) {
    if (hit[m]) continue;
    int v = -1;
    for (int i = 0; i < n_rec; ++i)
      if (!touched[i] && (v < 0 || last_use[i] < last_use[v])) v = i;
    evicted[m] = expert_of_rec[v];
    if (expert_of_rec[v] >= 0) rec_of_expert[expert_of_rec[v]] = -1;
    expert_of_rec[v] = ids[m];
    rec_of_expert[ids[m]] = v;
    last_use[v] = t;
    touched[v] = 1;
    rec[m] = v;
    ++n_new;
  }
  return n_new;
}

// Null when the threads cannot be started (no exception leaves the library).
FilePool* file_pool_create(int n_threads) {
  try {
    return new FilePool(n_threads < 1 ? 1 : n_threads);
  } catch (...) {
    return nullptr;
  }
}
void file_pool_destroy(FilePool* fp) { delete fp; }
int file_pool_transfer(FilePool* fp, int fd, bool write, uint64_t offset, void* buf, uint64_t bytes, uint64_t chunk) {
  return fp->run(fd, write, offset, buf, bytes, chunk);
}

}  // namespace moe

extern "C" moe_status moe_pread_parallel(const char* path, uint64_t offset, uint64_t bytes, void* dst, int n_threads,
                                         uint64_t chunk_bytes) {
  if (!path || (!dst && bytes > 0) || n_threads < 1 || n_threads > 64) return MOE_EINVAL;
  const int fd = ::open(path, O_RDONLY);
  if (fd < 0) return MOE_EINVAL;
  moe::FilePool* pool = moe::file_pool_create(n_threads);
  if (!pool) {
    ::close(fd);
    return MOE_ENOMEM;
  }
  const int e = pool->run(fd, false, offset, dst, bytes, chunk_bytes);
  moe::file_pool_destroy(pool);
  ::close(fd);
  return e == 0 ? MOE_OK : MOE_EIO;
}
