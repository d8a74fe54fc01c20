// Launch counting and optional per-kernel CUDA-event timing.
//
// Every kernel launch of the library goes through KDA_LAUNCH, which bumps a
// process-wide counter and, while timing is enabled, records a CUDA event pair
// on the launching stream around the launch.  kda_timing_collect() waits for
// the recorded events and returns the elapsed time per kernel name.
#include <mutex>
#include <string.h>
#include <vector>

#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {
namespace {

struct Record {
  const char *name;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_timing = false;
unsigned long long g_launches = 0;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;
thread_local int t_open = -1;  // index of the record opened by inst_begin on this thread

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

void inst_begin(const char *name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_launches;
  t_open = -1;
  if (!g_timing) return;
  Record r{name, take_event(), take_event()};
  if (r.start == nullptr || r.stop == nullptr) return;
  cudaEventRecord(r.start, s);
  g_records.push_back(r);
  t_open = (int)g_records.size() - 1;
}

void inst_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (t_open >= 0 && t_open < (int)g_records.size()) cudaEventRecord(g_records[t_open].stop, s);
  t_open = -1;
}

}  // namespace kda

namespace kda {
namespace {

// One thread waits, with a bounded wait, on an mbarrier that nothing arrives
// on: the wait gives up after `polls` polls and raises *err.
__global__ void bounded_wait_probe_kernel(int *err, long polls) {
  __shared__ uint64_t bar;
  umma::bar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  umma::bar_wait(&bar, 0, err, polls);
}

}  // namespace
}  // namespace kda

extern "C" {

kda_status kda_debug_bounded_wait(int *err, long long polls, void *stream) {
  if (err == nullptr || polls < 1 || polls > (1LL << 24)) {
    kda::set_last_error("kda_debug_bounded_wait: err must be a device int and 1 <= polls <= 2^24");
    return KDA_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  KDA_LAUNCH("bounded_wait_probe_kernel", s, kda::bounded_wait_probe_kernel<<<1, 1, 0, s>>>(err, (long)polls));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    kda::set_last_error(cudaGetErrorString(e));
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

unsigned long long kda_launch_count(void) {
  std::lock_guard<std::mutex> lk(kda::g_mu);
  return kda::g_launches;
}

int kda_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(kda::g_mu);
  const int prev = kda::g_timing ? 1 : 0;
  kda::g_timing = on != 0;
  return prev;
}

int kda_timing_collect(int max_kernels, char *names, size_t name_stride, double *total_ms,
                       int *launches) {
  std::lock_guard<std::mutex> lk(kda::g_mu);
  std::vector<const char *> seen;
  std::vector<double> ms;
  std::vector<int> cnt;
  for (auto &r : kda::g_records) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      t = -1.f;
    size_t i = 0;
    while (i < seen.size() && strcmp(seen[i], r.name) != 0) ++i;
    if (i == seen.size()) {
      seen.push_back(r.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[i] += t;
    cnt[i] += 1;
    kda::g_pool.push_back(r.start);
    kda::g_pool.push_back(r.stop);
  }
  kda::g_records.clear();
  const int n = (int)seen.size();
  for (int i = 0; i < n && i < max_kernels; ++i) {
    if (names != nullptr && name_stride > 0) {
      strncpy(names + (size_t)i * name_stride, seen[i], name_stride - 1);
      names[(size_t)i * name_stride + name_stride - 1] = 0;
    }
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = cnt[i];
  }
  return n;
}

}  // extern "C"
