// Attention over the prefetched rows (InfiniGen paper-graph summary, section 3.4, Inference
// Controller) and the dense layer-0 attention ("Why InfiniGen starts speculation from Layer 1").
//
// Decode attention has one query row per head, so it is a bandwidth-bound pass over the
// gathered K and V rows, not a tensor-core contraction.  A row of d fp16 values is read by
// d/8 lanes with 16-byte loads; each lane group keeps an fp32 online softmax (running max,
// running sum, partial output) over its rows, kUnroll rows in flight, and the groups are merged
// in shared memory.  When there are too few (b, h) units to fill the GPU, the rows of each
// head are split across CTAs and a second kernel merges the partial (max, sum, output).
#include <math.h>

#include "ig_common.cuh"

namespace ig {
namespace {

constexpr int kAttThreads = 128;
constexpr int kAttUnroll = 4;
constexpr int kMaxAttSplits = 16;

inline int att_splits_max(int Lcap) {
  int s = Lcap / 64;
  return s < 1 ? 1 : (s > kMaxAttSplits ? kMaxAttSplits : s);
}

template <int D>
__device__ __forceinline__ float row_dot(const float (&q)[8], uint4 kv) {
  float2 a = h2_to_f2(kv.x), b = h2_to_f2(kv.y), c = h2_to_f2(kv.z), e = h2_to_f2(kv.w);
  float s = q[0] * a.x;
  s = fmaf(q[1], a.y, s);
  s = fmaf(q[2], b.x, s);
  s = fmaf(q[3], b.y, s);
  s = fmaf(q[4], c.x, s);
  s = fmaf(q[5], c.y, s);
  s = fmaf(q[6], e.x, s);
  s = fmaf(q[7], e.y, s);
  constexpr int VPR = D / 8;
#pragma unroll
  for (int o = VPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

__device__ __forceinline__ void online_add(float z, uint4 vv, float& m, float& l, float (&acc)[8]) {
  const float mn = fmaxf(m, z);
  const float corr = __expf(m - mn);   // m = -inf at start: exp(-inf) = 0
  const float p = __expf(z - mn);
  l = l * corr + p;
  float2 a = h2_to_f2(vv.x), b = h2_to_f2(vv.y), c = h2_to_f2(vv.z), e = h2_to_f2(vv.w);
  const float vals[8] = {a.x, a.y, b.x, b.y, c.x, c.y, e.x, e.y};
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vals[i], acc[i] * corr);
  m = mn;
}

// cnt_per_seq: the row count of (b, h) is cnt[b] (dense) instead of cnt[b * H + h].
template <int D>
__global__ void __launch_bounds__(kAttThreads) k5_attend(
    const __half* __restrict__ q, const __half* __restrict__ Kg, const __half* __restrict__ Vg,
    const int32_t* __restrict__ cnt, int cnt_per_seq, int H, int Lcap, float scale,
    const __half* __restrict__ k_new, const __half* __restrict__ v_new, float* __restrict__ out,
    float* __restrict__ ws, int splits, int* err) {
  constexpr int VPR = D / 8;                  // lanes per row
  constexpr int RPW = 32 / VPR;               // rows per warp step
  constexpr int NG = (kAttThreads / 32) * RPW;  // lane groups per CTA
  __shared__ float sm_m[NG], sm_l[NG];
  __shared__ float sm_acc[NG][D];
  const int bh = blockIdx.y, split = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v = lane % VPR, g = warp * RPW + lane / VPR;
  int c = cnt_per_seq ? cnt[bh / H] : cnt[bh];
  if (c < 0 || c > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    c = c < 0 ? 0 : Lcap;
  }
  const int per = (c + splits - 1) / splits;
  const int j0 = split * per;
  const int j1 = min(c, j0 + per);

  float qf[8];
  {
    uint4 qv = *reinterpret_cast<const uint4*>(q + (size_t)bh * D + v * 8);
    float2 a = h2_to_f2(qv.x), b = h2_to_f2(qv.y), cc = h2_to_f2(qv.z), e = h2_to_f2(qv.w);
    qf[0] = a.x * scale; qf[1] = a.y * scale; qf[2] = b.x * scale; qf[3] = b.y * scale;
    qf[4] = cc.x * scale; qf[5] = cc.y * scale; qf[6] = e.x * scale; qf[7] = e.y * scale;
  }
  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  const uint4* Kb = reinterpret_cast<const uint4*>(Kg + (size_t)bh * Lcap * D) + v;
  const uint4* Vb = reinterpret_cast<const uint4*>(Vg + (size_t)bh * Lcap * D) + v;
  // The trip count is uniform across each warp (the shuffles in row_dot take the full mask);
  // a lane group whose row is past the end computes on zeros and skips the update.
  const int sub = lane / VPR;
  for (int jw = j0 + warp * RPW; jw < j1; jw += NG * kAttUnroll) {
    uint4 kv[kAttUnroll], vv[kAttUnroll];
#pragma unroll
    for (int u = 0; u < kAttUnroll; ++u) {
      const int jj = jw + sub + u * NG;
      kv[u] = make_uint4(0, 0, 0, 0);
      vv[u] = make_uint4(0, 0, 0, 0);
      if (jj < j1) {
        kv[u] = __ldg(Kb + (size_t)jj * VPR);
        vv[u] = __ldg(Vb + (size_t)jj * VPR);
      }
    }
#pragma unroll
    for (int u = 0; u < kAttUnroll; ++u) {
      const int jj = jw + sub + u * NG;
      const float z = row_dot<D>(qf, kv[u]);
      if (jj < j1) online_add(z, vv[u], m, l, acc);
    }
  }
  if (split == 0 && k_new != nullptr && warp == 0) {
    uint4 kv = *reinterpret_cast<const uint4*>(k_new + (size_t)bh * D + v * 8);
    uint4 vv = *reinterpret_cast<const uint4*>(v_new + (size_t)bh * D + v * 8);
    const float z = row_dot<D>(qf, kv);
    if (g == 0) online_add(z, vv, m, l, acc);
  }
  if (v == 0) {
    sm_m[g] = m;
    sm_l[g] = l;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sm_acc[g][v * 8 + i] = acc[i];
  __syncthreads();
  float M = -INFINITY;
  for (int i = 0; i < NG; ++i) M = fmaxf(M, sm_m[i]);
  float Lsum = 0.f;
  for (int i = 0; i < NG; ++i)
    if (sm_m[i] != -INFINITY) Lsum += sm_l[i] * __expf(sm_m[i] - M);
  for (int dd = threadIdx.x; dd < D; dd += kAttThreads) {
    float o = 0.f;
    for (int i = 0; i < NG; ++i)
      if (sm_m[i] != -INFINITY) o += sm_acc[i][dd] * __expf(sm_m[i] - M);
    if (splits == 1) {
      out[(size_t)bh * D + dd] = Lsum > 0.f ? o / Lsum : 0.f;
    } else {
      float* w = ws + ((size_t)bh * splits + split) * (D + 2);
      w[2 + dd] = o;
      if (dd == 0) {
        w[0] = M;
        w[1] = Lsum;
      }
    }
  }
}

template <int D>
__global__ void k5_combine(const float* __restrict__ ws, int splits, float* __restrict__ out) {
  const int bh = blockIdx.x;
  const float* w = ws + (size_t)bh * splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, w[(size_t)s * (D + 2)]);
  float Lsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = w[(size_t)s * (D + 2)];
    if (ms != -INFINITY) Lsum += w[(size_t)s * (D + 2) + 1] * __expf(ms - M);
  }
  for (int dd = threadIdx.x; dd < D; dd += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float ms = w[(size_t)s * (D + 2)];
      if (ms != -INFINITY) o += w[(size_t)s * (D + 2) + 2 + dd] * __expf(ms - M);
    }
    out[(size_t)bh * D + dd] = Lsum > 0.f ? o / Lsum : 0.f;
  }
}

template <int D>
ig_status launch_attend(cudaStream_t st, int B, int H, int Lcap, float scale, const uint16_t* q,
                        const uint16_t* K, const uint16_t* V, const int32_t* cnt, int per_seq,
                        const uint16_t* kn, const uint16_t* vn, float* out, void* ws,
                        size_t ws_bytes) {
  const int units = B * H;
  const int sms = sm_count();
  int splits = 1;
  if (units < 2 * sms) {
    splits = (4 * sms + units - 1) / units;
    const int smax = att_splits_max(Lcap);
    if (splits > smax) splits = smax;
  }
  if (splits > 1) {
    const size_t need = (size_t)units * splits * (D + 2) * sizeof(float);
    if (!ws || ws_bytes < need) splits = 1;  // no room to split: one CTA per head
  }
  dim3 grid(splits, units);
  k5_attend<D><<<grid, kAttThreads, 0, st>>>(
      reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(K),
      reinterpret_cast<const __half*>(V), cnt, per_seq, H, Lcap, scale,
      reinterpret_cast<const __half*>(kn), reinterpret_cast<const __half*>(vn), out,
      static_cast<float*>(ws), splits, error_word());
  IG_CHECK_LAUNCH("attention launch");
  if (splits > 1) {
    k5_combine<D><<<units, D, 0, st>>>(static_cast<const float*>(ws), splits, out);
    IG_CHECK_LAUNCH("attention combine launch");
  }
  return IG_OK;
}

ig_status attend_common(void* stream, int B, int H, int d, int Lcap, float scale,
                        const uint16_t* q, const uint16_t* K, const uint16_t* V,
                        const int32_t* cnt, int per_seq, const uint16_t* kn, const uint16_t* vn,
                        float* out, void* ws, size_t ws_bytes) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128 (got %d)", d);
  IG_REQUIRE(q && K && V && cnt && out, "null pointer argument");
  IG_REQUIRE((kn == nullptr) == (vn == nullptr), "k_new and v_new go together");
  IG_REQUIRE(aligned(q, 16) && aligned(K, 16) && aligned(V, 16), "q, K, V must be 16-byte aligned");
  IG_REQUIRE(!kn || (aligned(kn, 16) && aligned(vn, 16)), "k_new, v_new must be 16-byte aligned");
  IG_REQUIRE(!ws || aligned(ws, 256), "workspace must be 256-byte aligned");
  cudaStream_t s = as_stream(stream);
  if (d == 128)
    return launch_attend<128>(s, B, H, Lcap, scale, q, K, V, cnt, per_seq, kn, vn, out, ws, ws_bytes);
  return launch_attend<64>(s, B, H, Lcap, scale, q, K, V, cnt, per_seq, kn, vn, out, ws, ws_bytes);
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" size_t ig_attend_workspace_bytes(int B, int H, int d, int Lcap) {
  if (B <= 0 || H <= 0 || d <= 0 || Lcap <= 0) return 0;
  return round_up((size_t)B * H * att_splits_max(Lcap) * (d + 2) * sizeof(float), 256);
}

extern "C" ig_status ig_sparse_attend(void* stream, int B, int H, int d, int Lcap, float scale,
                                      const uint16_t* q, const uint16_t* Kg, const uint16_t* Vg,
                                      const int32_t* cnt, const uint16_t* k_new,
                                      const uint16_t* v_new, float* out, void* workspace,
                                      size_t workspace_bytes) {
  return attend_common(stream, B, H, d, Lcap, scale, q, Kg, Vg, cnt, 0, k_new, v_new, out,
                       workspace, workspace_bytes);
}

extern "C" ig_status ig_dense_attend(void* stream, int B, int H, int d, int Lcap, float scale,
                                     const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                     const int32_t* L_valid, const uint16_t* k_new,
                                     const uint16_t* v_new, float* out, void* workspace,
                                     size_t workspace_bytes) {
  return attend_common(stream, B, H, d, Lcap, scale, q, K, V, L_valid, 1, k_new, v_new, out,
                       workspace, workspace_bytes);
}
