// Status plumbing of the C ABI: per-thread error messages, the device error word, ig_check.
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "ig_common.cuh"

namespace ig {

namespace {
thread_local char g_msg[512] = "";
constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;
// streams bound to a subset of the SMs (a green context), with that subset's size
std::vector<std::pair<cudaStream_t, int>> g_stream_sms;
std::atomic<int> g_n_stream_sms{0};
}  // namespace

// Per device: [0] the error word (bits IG_DEVERR_* set by guarded kernels), [1] the iteration
// limit of the score kernels' first bounded wait (ig_set_wait_limit).
__device__ int g_device_error_word[2] = {0, kDefaultWaitIters};

ig_status fail(ig_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

ig_status cuda_fail(cudaError_t e, const char* what) {
  return fail(IG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

int stream_sms(cudaStream_t st) {
  if (st && g_n_stream_sms.load(std::memory_order_acquire) > 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const auto& e : g_stream_sms)
      if (e.first == st) return e.second;
  }
  return 0;
}

int sm_count(cudaStream_t st) {
  const int n = stream_sms(st);
  return n > 0 ? n : sm_count();
}

int fetch_grid(cudaStream_t st) {
  // on a stream of its own SM partition the fetch takes two CTAs on every SM of it; sharing
  // all SMs with the compute stream, a quarter of them (38 on a GB300) already moves ~185 GB/s
  // over the host link, and more CTAs only slow the compute stream down
  const int n = stream_sms(st);
  return n > 0 ? 2 * n : (sm_count() / 4 > 0 ? sm_count() / 4 : 1);
}

void register_stream_sms(cudaStream_t st, int sms) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_stream_sms.emplace_back(st, sms);
  g_n_stream_sms.store((int)g_stream_sms.size(), std::memory_order_release);
}

void unregister_stream_sms(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (size_t i = 0; i < g_stream_sms.size(); ++i)
    if (g_stream_sms[i].first == st) {
      g_stream_sms.erase(g_stream_sms.begin() + (long)i);
      break;
    }
  g_n_stream_sms.store((int)g_stream_sms.size(), std::memory_order_release);
}

namespace {
std::atomic<uint64_t> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void count_launches(int64_t n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace ig

extern "C" uint64_t ig_launch_count(void) { return ig::g_launches.load(); }

extern "C" const char* ig_last_error(void) { return ig::g_msg; }

extern "C" int ig_version(void) { return 100; }

extern "C" ig_status ig_set_wait_limit(int max_iters) {
  int* w = ig::error_word();
  if (!w) return ig::fail(IG_ERR_CUDA, "ig_set_wait_limit: no device error word");
  const int v = max_iters < 0 ? ig::kDefaultWaitIters : max_iters;
  cudaError_t e = cudaMemcpy(w + 1, &v, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return ig::cuda_fail(e, "ig_set_wait_limit");
  return IG_OK;
}

extern "C" ig_status ig_check(void* stream) {
  cudaStream_t s = ig::as_stream(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return ig::cuda_fail(e, "ig_check: stream synchronize");
  int* w = ig::error_word();
  if (!w) return ig::fail(IG_ERR_CUDA, "ig_check: no device error word");
  int v = 0;
  e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return ig::cuda_fail(e, "ig_check: read error word");
  if (v) {
    int zero = 0;
    e = cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return ig::cuda_fail(e, "ig_check: clear error word");
  }
  if (v & IG_DEVERR_TIMEOUT) return ig::fail(IG_ERR_TIMEOUT, "a bounded in-kernel wait ran out (word 0x%x)", v);
  if (v & IG_DEVERR_INDEX) return ig::fail(IG_ERR_INVALID, "an in-kernel index guard tripped (word 0x%x)", v);
  return IG_OK;
}
