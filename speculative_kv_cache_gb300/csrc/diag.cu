// Diagnostics of the speculation and of the pool (not steps of the method): eviction misses
// under a capacity limit (InfiniGen paper-graph summary, section 3.4, "KV Cache Pool
// Management Under Memory Pressure", and the pool-limit study it calls for: how often the
// selection wants a token the pool has evicted, and how much of the selected weight that is).
#include <math.h>

#include "ig_common.cuh"

namespace ig {
namespace {

// One warp per (b, h): the head's selected tokens idx[0..cnt) over token-indexed scores;
// m = their maximum score; count the tokens not resident and the share of exp(s - m) on them.
__global__ void k_eviction_misses(int units, int H, int Lcap, const float* __restrict__ scores,
                                  const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
                                  const uint8_t* __restrict__ resident, int32_t* __restrict__ miss_cnt,
                                  float* __restrict__ miss_mass, int* err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= units) return;
  const int b = warp / H;
  int c = cnt[warp];
  if (c < 0 || c > Lcap) {
    if (lane == 0) raise_error(err, IG_DEVERR_INDEX);
    c = c < 0 ? 0 : Lcap;
  }
  const float* s = scores + (size_t)warp * Lcap;
  const int32_t* ix = idx + (size_t)warp * Lcap;
  const uint8_t* res = resident + (size_t)b * Lcap;
  float m = -INFINITY;
  for (int j = lane; j < c; j += 32) {
    const int t = ix[j];
    if (t >= 0 && t < Lcap) m = fmaxf(m, s[t]);
  }
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float all = 0.f, gone = 0.f;
  int n = 0;
  for (int j = lane; j < c; j += 32) {
    const int t = ix[j];
    if (t < 0 || t >= Lcap) {
      raise_error(err, IG_DEVERR_INDEX);
      continue;
    }
    const float w = expf(s[t] - m);
    all += w;
    if (!res[t]) {
      gone += w;
      ++n;
    }
  }
  for (int o = 16; o; o >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, o);
    gone += __shfl_xor_sync(0xffffffffu, gone, o);
    n += __shfl_xor_sync(0xffffffffu, n, o);
  }
  if (lane == 0) {
    miss_cnt[warp] = n;
    miss_mass[warp] = all > 0.f ? gone / all : 0.f;
  }
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" ig_status ig_eviction_misses(void* stream, int B, int H, int Lcap, const float* scores,
                                        const int32_t* idx, const int32_t* cnt,
                                        const uint8_t* resident, int32_t* miss_cnt,
                                        float* miss_mass) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE((long long)B * H * Lcap < (1ll << 31), "B*H*Lcap must stay below 2^31");
  IG_REQUIRE(scores && idx && cnt && resident && miss_cnt && miss_mass, "null pointer argument");
  const int units = B * H;
  const int threads = 256;
  const int blocks = (units * 32 + threads - 1) / threads;
  k_eviction_misses<<<blocks, threads, 0, as_stream(stream)>>>(units, H, Lcap, scores, idx, cnt, resident,
                                                                miss_cnt, miss_mass, error_word());
  IG_CHECK_LAUNCH("eviction-miss launch");
  return IG_OK;
}
