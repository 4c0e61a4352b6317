// Shared helpers of the sm_103a kernels: status handling, the device error word, half
// conversions, and the PTX wrappers for mbarriers and bulk (TMA) copies.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/ig.h"

namespace ig {

// Sets the calling thread's last-error message and returns `st`.
ig_status fail(ig_status st, const char* fmt, ...);

// Maps a CUDA error to IG_ERR_CUDA with a message naming `what`.
ig_status cuda_fail(cudaError_t e, const char* what);

// Device pointer of the error word of the current device; the word after it holds the
// iteration limit of the score kernels' first bounded wait (ig_set_wait_limit).
int* error_word();

// Default iteration limit of a bounded mbarrier wait (far longer than any copy takes).
constexpr int kDefaultWaitIters = 1 << 22;

// Number of SMs of the current device (cached per device).
int sm_count();

// Number of SMs work on `st` may use: the size of its SM partition when the stream belongs to
// one (ig_sm_split_create), else the device's count.  Grids are sized by it.
int sm_count(cudaStream_t st);
// SMs of the partition `st` belongs to, 0 when it has none.
int stream_sms(cudaStream_t st);
// Default grid of the host-link fetch kernels launched on `st`.
int fetch_grid(cudaStream_t st);
void register_stream_sms(cudaStream_t st, int sms);
void unregister_stream_sms(cudaStream_t st);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Counts one kernel launch of this library (ig_launch_count); count_launches adds n (n may be
// negative: launches recorded into a graph have not run).
void count_launch();
void count_launches(int64_t n);

#define IG_CHECK_LAUNCH(what)                                   \
  do {                                                          \
    cudaError_t e_ = cudaGetLastError();                        \
    if (e_ != cudaSuccess) return ::ig::cuda_fail(e_, what);    \
    ::ig::count_launch();                                       \
  } while (0)

#define IG_REQUIRE(cond, ...)                                   \
  do {                                                          \
    if (!(cond)) return ::ig::fail(IG_ERR_INVALID, __VA_ARGS__); \
  } while (0)

// Launches `kern` with programmatic stream serialization: it may start while the kernel before
// it in the stream is still running (which lets it begin once that kernel's CTAs have signalled
// pdl_trigger()), so it must call pdl_wait() before reading anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ----------------------------------------------------------------------------------------
// Device side
// ----------------------------------------------------------------------------------------
// Programmatic dependent launch: the kernel after this one in the stream (launched with
// launch_pdl) may be scheduled once every CTA of this grid has issued pdl_trigger() ...
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// ... and a kernel launched that way waits here until the grid before it has completed and its
// memory operations are visible (a no-op for a kernel launched without the attribute).  Every
// such kernel waits before it exits, so that completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void raise_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// One bounded probe of phase `parity`; true once the phase has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` with an iteration limit; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t max_iters = (uint32_t)kDefaultWaitIters) {
  for (uint32_t i = 0; i < max_iters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// The host-set limit of a score kernel's first wait for its copies (ig_set_wait_limit), read
// from the word after the error word.  A give-up path must still drain its copies with the
// default limit before the CTA leaves.
__device__ __forceinline__ uint32_t wait_limit(const int* err) {
  if (!err) return (uint32_t)kDefaultWaitIters;
  const int v = *(reinterpret_cast<const volatile int*>(err) + 1);
  return v < 0 ? (uint32_t)kDefaultWaitIters : (uint32_t)v;
}

// An L2 policy that marks the lines it touches first for eviction: for data read once per
// step (the partial key cache, the projection weight), so that it does not push out data read
// again soon (the staged rows the attention reads).  Speculation + selection of an OPT-30B
// layer alone: 68.4 -> 63.9 us.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor TMA) copy global -> shared, completing on `bar` with `bytes` of tx, under
// the L2 policy `pol`.  src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// 16-byte read-only load that does not allocate in L1 (streams through L2).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 8- and 4-byte read-only loads that do not allocate in L1
__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Sum of S split partials p[0], p[stride], ... added in that order (the same fp32 sum as a
// plain loop): the loads are issued 8 at a time before their adds, so they overlap.
__device__ __forceinline__ float sum_splits(const float* __restrict__ p, size_t stride, int S) {
  float a = 0.f;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = s0 + i < S ? __ldg(p + (size_t)(s0 + i) * stride) : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (s0 + i < S) a += v[i];
  }
  return a;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

}  // namespace ig
