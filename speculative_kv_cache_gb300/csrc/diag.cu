// Diagnostics of the speculation and of the pool (not steps of the method), the studies the
// InfiniGen paper-graph summary's critique asks for:
//   * eviction misses under a capacity limit (section 3.4, "KV Cache Pool Management Under
//     Memory Pressure"): how often selection wants a token the pool has evicted;
//   * speculation fidelity (section 3.4, "Decoding Stage"; the skew ablation of Fig 13): how
//     well the set speculated at layer i-1 matches layer i's real attention, and how much of
//     the q.k magnitude the partial columns capture with and without the skew.
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

constexpr int kDiagThreads = 256;
constexpr int kMaxRecallTokens = 16384;  // real logits of one head in shared memory (64 KB)

template <int VPR>
__device__ __forceinline__ float group_sum(float s) {
#pragma unroll
  for (int o = VPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Block-wide reductions over kDiagThreads threads (every thread calls; red has 32 floats).
__device__ float block_max(float v, float* red) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = -INFINITY;
  for (int i = 0; i < kDiagThreads / 32; ++i) r = fmaxf(r, red[i]);
  return r;
}
__device__ float block_sum(float v, float* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < kDiagThreads / 32; ++i) r += red[i];
  return r;
}

// fp32 -> uint32 whose unsigned order is the float order (-0 and +0 adjacent)
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Real logits z_t = scale q . K_t of one head for t < L into z[] (shared), d/8 lanes per row.
template <int D>
__device__ void head_logits(const __half* __restrict__ q, const __half* __restrict__ K, int L, float scale,
                            float* z) {
  constexpr int VPR = D / 8, RPW = 32 / VPR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, v = lane % VPR, sub = lane / VPR;
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4*>(q + v * 8);
    const __half2* h = reinterpret_cast<const __half2*>(&qv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      qf[2 * i] = f.x * scale;
      qf[2 * i + 1] = f.y * scale;
    }
  }
  // warp-uniform trip count: rows past L compute on zeros and are not stored
  for (int t0 = warp * RPW; t0 < L; t0 += (kDiagThreads / 32) * RPW) {
    const int t = t0 + sub;
    float acc = 0.f;
    if (t < L) {
      const uint4 kv = *reinterpret_cast<const uint4*>(K + (size_t)t * D + v * 8);
      const __half2* h = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        acc = fmaf(qf[2 * i], f.x, acc);
        acc = fmaf(qf[2 * i + 1], f.y, acc);
      }
    }
    acc = group_sum<VPR>(acc);
    if (t < L && v == 0) z[t] = acc;
  }
  __syncthreads();
}

// One CTA per (b, h): recall@c and weight recall of the speculated set against the real
// logits (definitions in include/ig.h).
template <int D>
__global__ void __launch_bounds__(kDiagThreads) k_attention_recall(
    int H, int Lcap, float scale, const __half* __restrict__ q, const __half* __restrict__ K,
    const int32_t* __restrict__ L_valid, const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
    float* __restrict__ recall, float* __restrict__ weight, int* err) {
  extern __shared__ float z[];  // [Lcap]
  __shared__ float red[32];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh_digit, sh_above;
  const int u = blockIdx.x, b = u / H;
  int L = L_valid[b];
  if (L < 0 || L > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    L = L < 0 ? 0 : Lcap;
  }
  int c = cnt[u];
  if (c < 0 || c > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    c = c < 0 ? 0 : Lcap;
  }
  if (c == 0 || L == 0) {
    if (threadIdx.x == 0) {
      recall[u] = 0.f;
      weight[u] = 0.f;
    }
    return;
  }
  head_logits<D>(q + (size_t)u * D, K + (size_t)u * Lcap * D, L, scale, z);
  float m = -INFINITY;
  for (int t = threadIdx.x; t < L; t += kDiagThreads) m = fmaxf(m, z[t]);
  const float M = block_max(m, red);
  float e = 0.f;
  for (int t = threadIdx.x; t < L; t += kDiagThreads) e += expf(z[t] - M);
  const float S = block_sum(e, red);
  // the c-th largest logit (c capped at L): MSB-first radix select on the ordered keys
  const int want = c < L ? c : L;
  uint32_t prefix = 0, mask = 0;
  int rem = want;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kDiagThreads) hist[i] = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < L; t += kDiagThreads) {
      const uint32_t key = ordered(z[t]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t above = 0;
      int dgt = 255;
      for (; dgt > 0; --dgt) {
        if (above + hist[dgt] >= (uint32_t)rem) break;
        above += hist[dgt];
      }
      sh_digit = (uint32_t)dgt;
      sh_above = above;
    }
    __syncthreads();
    prefix |= sh_digit << shift;
    mask |= 255u << shift;
    rem -= (int)sh_above;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // key of the want-th largest logit
  float hits = 0.f, w = 0.f;
  const int32_t* ix = idx + (size_t)u * Lcap;
  for (int j = threadIdx.x; j < c; j += kDiagThreads) {
    const int t = ix[j];
    if (t < 0 || t >= L) {
      raise_error(err, IG_DEVERR_INDEX);
      continue;
    }
    hits += ordered(z[t]) >= thr ? 1.f : 0.f;
    w += expf(z[t] - M);
  }
  hits = block_sum(hits, red);
  w = block_sum(w, red);
  if (threadIdx.x == 0) {
    recall[u] = hits / (float)c;
    weight[u] = w / S;
  }
}

// One CTA per (b, h): sum_t sum_{c in S} |q_c K_tc| / sum_t sum_c |q_c K_tc| over t < L.
template <int D>
__global__ void __launch_bounds__(kDiagThreads) k_captured_fraction(
    int H, int k, int Lcap, const __half* __restrict__ q, const __half* __restrict__ K,
    const int32_t* __restrict__ L_valid, const int32_t* __restrict__ cols, float* __restrict__ frac, int* err) {
  constexpr int VPR = D / 8, RPW = 32 / VPR;
  __shared__ float red[32];
  __shared__ float sq[D], in_s[D];
  const int u = blockIdx.x, b = u / H, h = u % H;
  int L = L_valid[b];
  if (L < 0 || L > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    L = L < 0 ? 0 : Lcap;
  }
  for (int i = threadIdx.x; i < D; i += kDiagThreads) {
    sq[i] = fabsf(__half2float(q[(size_t)u * D + i]));
    in_s[i] = 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += kDiagThreads) {
    const int col = cols[h * k + i];
    if (col < 0 || col >= D) raise_error(err, IG_DEVERR_INDEX);
    else in_s[col] = 1.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, v = lane % VPR, sub = lane / VPR;
  float qa[8], ms[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qa[i] = sq[v * 8 + i];
    ms[i] = in_s[v * 8 + i];
  }
  float tot = 0.f, part = 0.f;
  const __half* Kh = K + (size_t)u * Lcap * D;
  for (int t = warp * RPW + sub; t < L; t += (kDiagThreads / 32) * RPW) {
    const uint4 kv = *reinterpret_cast<const uint4*>(Kh + (size_t)t * D + v * 8);
    const __half2* hh = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(hh[i]);
      const float a = qa[2 * i] * fabsf(f.x), bb = qa[2 * i + 1] * fabsf(f.y);
      tot += a + bb;
      part += ms[2 * i] * a + ms[2 * i + 1] * bb;
    }
  }
  tot = block_sum(tot, red);
  part = block_sum(part, red);
  if (threadIdx.x == 0) frac[u] = tot > 0.f ? part / tot : 0.f;
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" ig_status ig_attention_recall(void* stream, int B, int H, int d, int Lcap, float scale,
                                         const uint16_t* q, const uint16_t* K, const int32_t* L_valid,
                                         const int32_t* idx, const int32_t* cnt, float* recall,
                                         float* weight) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128 (got %d)", d);
  IG_REQUIRE(Lcap <= kMaxRecallTokens, "Lcap %d exceeds %d", Lcap, kMaxRecallTokens);
  IG_REQUIRE(q && K && L_valid && idx && cnt && recall && weight, "null pointer argument");
  IG_REQUIRE(aligned(q, 16) && aligned(K, 16), "q and K must be 16-byte aligned");
  const size_t smem = (size_t)Lcap * sizeof(float);
  cudaStream_t st = as_stream(stream);
  auto qh = reinterpret_cast<const __half*>(q);
  auto Kh = reinterpret_cast<const __half*>(K);
  cudaError_t e = cudaSuccess;
  if (d == 128) {
    if (smem > 48 * 1024) e = cudaFuncSetAttribute(k_attention_recall<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "recall smem attribute");
    k_attention_recall<128><<<B * H, kDiagThreads, smem, st>>>(H, Lcap, scale, qh, Kh, L_valid, idx, cnt, recall,
                                                               weight, error_word());
  } else {
    if (smem > 48 * 1024) e = cudaFuncSetAttribute(k_attention_recall<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "recall smem attribute");
    k_attention_recall<64><<<B * H, kDiagThreads, smem, st>>>(H, Lcap, scale, qh, Kh, L_valid, idx, cnt, recall,
                                                              weight, error_word());
  }
  IG_CHECK_LAUNCH("recall launch");
  return IG_OK;
}

extern "C" ig_status ig_captured_fraction(void* stream, int B, int H, int d, int k, int Lcap,
                                          const uint16_t* q, const uint16_t* K, const int32_t* L_valid,
                                          const int32_t* cols, float* frac) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0 && k > 0 && k <= d, "bad sizes");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128 (got %d)", d);
  IG_REQUIRE(q && K && L_valid && cols && frac, "null pointer argument");
  IG_REQUIRE(aligned(q, 16) && aligned(K, 16), "q and K must be 16-byte aligned");
  cudaStream_t st = as_stream(stream);
  auto qh = reinterpret_cast<const __half*>(q);
  auto Kh = reinterpret_cast<const __half*>(K);
  if (d == 128)
    k_captured_fraction<128><<<B * H, kDiagThreads, 0, st>>>(H, k, Lcap, qh, Kh, L_valid, cols, frac, error_word());
  else
    k_captured_fraction<64><<<B * H, kDiagThreads, 0, st>>>(H, k, Lcap, qh, Kh, L_valid, cols, frac, error_word());
  IG_CHECK_LAUNCH("captured-fraction launch");
  return IG_OK;
}

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
