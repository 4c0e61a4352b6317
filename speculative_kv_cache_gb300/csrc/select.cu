// Selection of the tokens each head prefetches (InfiniGen paper-graph summary, section 3.4,
// "Decoding Stage", Step 3 threshold, Step 4 multi-head averaging, Step 5 transfer cap; and
// the normalized threshold alpha' = alpha / sigma its follow-up work proposes).
//
// One CTA per (sequence, head).  The per-head maximum is a warp-shuffle reduction followed by
// a reduction over warps; the chosen tokens are compacted in ascending order with a warp
// ballot + popc prefix and a scan over warp totals.  A count limit (cap, or the head-averaged
// count) is met exactly with an MSB-first radix select on order-preserving keys of the fp32
// scores, ties going to the lower token index.
#include <math.h>

#include "ig_common.cuh"

namespace ig {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

// Order-preserving map float -> uint32 (larger float, larger key).  NaN never reaches it.
__device__ __forceinline__ uint32_t fkey(float s) {
  uint32_t u = (s == 0.0f) ? 0u : __float_as_uint(s);  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
  float fred[kSelWarps];
  int ired[kSelWarps];
  int wscan[kSelWarps];
  int wscan_eq[kSelWarps];
  unsigned int hist[256];
  uint32_t prefix;
  int remaining;
  int total;
};

__device__ float block_max(float v, SelShared& sh) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh.fred[warp] = v;
  __syncthreads();
  float r = -INFINITY;
  for (int w = 0; w < kSelWarps; ++w) r = fmaxf(r, sh.fred[w]);
  return r;
}

__device__ int block_sum(int v, SelShared& sh) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh.ired[warp] = v;
  __syncthreads();
  int r = 0;
  for (int w = 0; w < kSelWarps; ++w) r += sh.ired[w];
  return r;
}

__device__ float block_fsum(float v, SelShared& sh) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh.fred[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < kSelWarps; ++w) r += sh.fred[w];
  return r;
}

// Finds the n-th largest key among valid tokens (n >= 1, n <= number of valid tokens).
// Returns the key; *need_eq = how many tokens holding exactly that key are to be kept
// (the lowest-index ones).
__device__ uint32_t radix_select(const float* s, int L, int n, int* need_eq, SelShared& sh) {
  if (threadIdx.x == 0) {
    sh.prefix = 0;
    sh.remaining = n;
  }
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += kSelThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh.prefix;
    for (int t = threadIdx.x; t < L; t += kSelThreads) {
      const float v = s[t];
      if (isnan(v)) continue;
      const uint32_t kk = fkey(v);
      if ((kk & mask) == prefix) atomicAdd(&sh.hist[(kk >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int rem = sh.remaining;
      int above = 0;
      int dsel = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        const int c = (int)sh.hist[dgt];
        if (above + c >= rem) {
          dsel = dgt;
          break;
        }
        above += c;
      }
      sh.remaining = rem - above;
      sh.prefix = prefix | ((uint32_t)dsel << shift);
    }
    mask |= 0xffu << shift;
  }
  __syncthreads();
  *need_eq = sh.remaining;
  return sh.prefix;
}

// Ordered compaction.  mode 0: keep valid tokens with (m - s) < alpha or s tied with the
// maximum.  mode 1: keep valid tokens with key > kstar, plus the first need_eq tokens with
// key == kstar.
__device__ int compact(const float* s, int L, int mode, float m, float alpha, uint32_t kstar,
                       int need_eq, int32_t* idx_out, uint8_t* used_b, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  int running = 0, running_eq = 0;
  for (int base = 0; base < L; base += kSelThreads) {
    const int t = base + threadIdx.x;
    bool f = false, eq = false;
    if (t < L) {
      const float v = s[t];
      if (!isnan(v)) {
        if (mode == 0) {
          f = (m - v) < alpha || (m - v) == 0.f;
        } else {
          const uint32_t kk = fkey(v);
          f = kk > kstar;
          eq = kk == kstar;
        }
      }
    }
    if (mode == 1) {
      const unsigned be = __ballot_sync(0xffffffffu, eq);
      __syncthreads();
      if (lane == 0) sh.wscan_eq[warp] = __popc(be);
      __syncthreads();
      int before = running_eq + __popc(be & lt);
      int tot = 0;
      for (int w = 0; w < kSelWarps; ++w) {
        const int c = sh.wscan_eq[w];
        if (w < warp) before += c;
        tot += c;
      }
      running_eq += tot;
      if (eq && before < need_eq) f = true;
    }
    const unsigned bf = __ballot_sync(0xffffffffu, f);
    __syncthreads();
    if (lane == 0) sh.wscan[warp] = __popc(bf);
    __syncthreads();
    int pos = running + __popc(bf & lt);
    int tot = 0;
    for (int w = 0; w < kSelWarps; ++w) {
      const int c = sh.wscan[w];
      if (w < warp) pos += c;
      tot += c;
    }
    if (f) {
      idx_out[pos] = t;
      if (used_b) used_b[t] = 1;
    }
    running += tot;
  }
  return running;
}

// pass: 0 = threshold (+ optional cap) and write; 1 = head-avg counting only; 2 = head-avg write.
// normalized (pass 0): the threshold is alpha times the head's score standard deviation.
__global__ void __launch_bounds__(kSelThreads) k3_select(const float* __restrict__ scores,
                                                         const int* __restrict__ L_valid, int H,
                                                         int Lcap, float alpha, int normalized,
                                                         double cap_frac,
                                                         int pass, int32_t* __restrict__ idx,
                                                         int32_t* __restrict__ cnt,
                                                         uint8_t* __restrict__ used,
                                                         int32_t* __restrict__ counts_ws, int* err) {
  __shared__ SelShared sh;
  const int bh = blockIdx.x, b = bh / H;
  int L = L_valid[b];
  if (L < 0 || L > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    L = L < 0 ? 0 : Lcap;
  }
  const float* s = scores + (size_t)bh * Lcap;
  int32_t* io = idx + (size_t)bh * Lcap;
  uint8_t* ub = used ? used + (size_t)b * Lcap : nullptr;
  const int capn = cap_frac >= 1.0 ? L : (int)floor(cap_frac * (double)L + 0.5);

  float m = -INFINITY;
  int nv = 0;
  for (int t = threadIdx.x; t < L; t += kSelThreads) {
    const float v = s[t];
    if (!isnan(v)) {
      m = fmaxf(m, v);
      ++nv;
    }
  }
  m = block_max(m, sh);
  nv = block_sum(nv, sh);

  if (pass == 2) {
    int tot = 0;
    for (int h = 0; h < H; ++h) tot += counts_ws[(size_t)b * H + h];
    int cbar = (2 * tot + H) / (2 * H);
    if (cbar < 1) cbar = 1;
    if (cbar > capn) cbar = capn;
    const int n = min(cbar, nv);
    int kept = 0;
    if (n > 0) {
      int need_eq = 0;
      const uint32_t kstar = radix_select(s, L, n, &need_eq, sh);
      kept = compact(s, L, 1, 0.f, 0.f, kstar, need_eq, io, ub, sh);
    }
    if (threadIdx.x == 0) cnt[bh] = kept;
    return;
  }

  if (normalized && nv > 0) {  // alpha in units of the population std of the valid scores
    float a = 0.f;
    for (int t = threadIdx.x; t < L; t += kSelThreads) {
      const float v = s[t];
      if (!isnan(v)) a += v;
    }
    const float mean = block_fsum(a, sh) / (float)nv;
    float q = 0.f;
    for (int t = threadIdx.x; t < L; t += kSelThreads) {
      const float v = s[t];
      if (!isnan(v)) q = fmaf(v - mean, v - mean, q);
    }
    alpha = alpha * sqrtf(block_fsum(q, sh) / (float)nv);
  }
  int nthr = 0;
  if (nv > 0) {
    int c = 0;
    for (int t = threadIdx.x; t < L; t += kSelThreads) {
      const float v = s[t];
      if (!isnan(v) && ((m - v) < alpha || (m - v) == 0.f)) ++c;
    }
    nthr = block_sum(c, sh);
  }
  if (pass == 1) {
    if (threadIdx.x == 0) counts_ws[bh] = nthr;
    return;
  }
  int kept = 0;
  if (nthr > 0) {
    if (nthr <= capn) {
      kept = compact(s, L, 0, m, alpha, 0u, 0, io, ub, sh);
    } else if (capn > 0) {
      int need_eq = 0;
      const uint32_t kstar = radix_select(s, L, capn, &need_eq, sh);
      kept = compact(s, L, 1, 0.f, 0.f, kstar, need_eq, io, ub, sh);
    }
  }
  if (threadIdx.x == 0) cnt[bh] = kept;
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" size_t ig_select_workspace_bytes(int B, int H) {
  if (B <= 0 || H <= 0) return 0;
  return round_up((size_t)B * H * sizeof(int32_t), 256);
}

extern "C" ig_status ig_select(void* stream, int B, int H, int Lcap, const float* scores,
                               const int32_t* L_valid, float alpha, int policy, float cap_frac,
                               int32_t* idx, int32_t* cnt, uint8_t* used, void* workspace,
                               size_t workspace_bytes) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE(scores && L_valid && idx && cnt, "null pointer argument");
  IG_REQUIRE(alpha > 0.f, "alpha must be > 0 (got %g)", (double)alpha);
  IG_REQUIRE(!(cap_frac < 0.f) && !isnan(cap_frac), "cap_frac must be >= 0");
  IG_REQUIRE(policy == IG_SEL_THRESHOLD || policy == IG_SEL_HEAD_AVG || policy == IG_SEL_NORMALIZED,
             "unknown policy %d", policy);
  cudaStream_t s = as_stream(stream);
  int* err = error_word();
  if (used) {
    cudaError_t e = cudaMemsetAsync(used, 0, (size_t)B * Lcap, s);
    if (e != cudaSuccess) return cuda_fail(e, "clear used flags");
  }
  const double cf = (double)cap_frac;
  if (policy == IG_SEL_THRESHOLD || policy == IG_SEL_NORMALIZED) {
    k3_select<<<B * H, kSelThreads, 0, s>>>(scores, L_valid, H, Lcap, alpha, policy == IG_SEL_NORMALIZED, cf, 0,
                                            idx, cnt, used, nullptr, err);
    IG_CHECK_LAUNCH("select launch");
    return IG_OK;
  }
  const size_t need = ig_select_workspace_bytes(B, H);
  if (!workspace || workspace_bytes < need)
    return fail(IG_ERR_CAPACITY, "head-averaged selection needs %zu workspace bytes", need);
  int32_t* counts = static_cast<int32_t*>(workspace);
  k3_select<<<B * H, kSelThreads, 0, s>>>(scores, L_valid, H, Lcap, alpha, 0, cf, 1, idx, cnt, used,
                                          counts, err);
  IG_CHECK_LAUNCH("select (count) launch");
  k3_select<<<B * H, kSelThreads, 0, s>>>(scores, L_valid, H, Lcap, alpha, 0, cf, 2, idx, cnt, used,
                                          counts, err);
  IG_CHECK_LAUNCH("select (head-avg) launch");
  return IG_OK;
}
