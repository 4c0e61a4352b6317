// Attention over the prefetched rows (InfiniGen paper-graph summary, section 3.4, Inference
// Controller) and the dense layer-0 attention ("Why InfiniGen starts speculation from Layer 1").
//
// Decode attention has one query row per head, so it is a bandwidth-bound pass over the
// gathered K and V rows, not a tensor-core contraction.  A row of d fp16 values is read by
// d/8 lanes with 16-byte loads; each lane group keeps an fp32 online softmax (running max,
// running sum, partial output) over its rows with kUnroll rows in flight.
//
// Balance: the number of rows per head varies a lot (the threshold keeps a few tokens for a
// peaked head and most of them for a flat one), so heads are not mapped to CTAs.  Every CTA
// scans the per-head counts in shared memory and takes an equal share of ALL rows, in head
// order; for each head segment it meets, it writes one partial (max, sum, unnormalised output)
// to the workspace at index head + CTA (unique: CTA ranges and head ranges are both
// increasing).  A combine kernel merges each head's partials, adds the current token's own
// key/value, and normalises.  No atomics; the result does not depend on timing.
#include <math.h>

#include "ig_common.cuh"

namespace ig {
namespace {

constexpr int kAttThreads = 128;
constexpr int kAttUnroll = 4;
constexpr int kMaxAttCtas = 1024;   // upper bound of the balanced grid (sizes the workspace)
constexpr int kMaxAttUnits = 16384; // (units + 1) ints of shared memory for the scan

__device__ __forceinline__ float lane_dot(const float (&q)[8], uint4 kv) {
  float2 a = h2_to_f2(kv.x), b = h2_to_f2(kv.y), c = h2_to_f2(kv.z), e = h2_to_f2(kv.w);
  float s = q[0] * a.x;
  s = fmaf(q[1], a.y, s);
  s = fmaf(q[2], b.x, s);
  s = fmaf(q[3], b.y, s);
  s = fmaf(q[4], c.x, s);
  s = fmaf(q[5], c.y, s);
  s = fmaf(q[6], e.x, s);
  s = fmaf(q[7], e.y, s);
  return s;
}

// dot of a d-wide row held by VPR consecutive lanes (full-warp shuffles; every lane calls)
template <int VPR>
__device__ __forceinline__ float group_sum(float s) {
#pragma unroll
  for (int o = VPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

__device__ __forceinline__ void online_add(float z, uint4 vv, float& m, float& l, float (&acc)[8]) {
  const float mn = fmaxf(m, z);
  const float corr = __expf(m - mn);  // m = -inf at start: exp(-inf) = 0
  const float p = __expf(z - mn);
  l = l * corr + p;
  float2 a = h2_to_f2(vv.x), b = h2_to_f2(vv.y), c = h2_to_f2(vv.z), e = h2_to_f2(vv.w);
  const float vals[8] = {a.x, a.y, b.x, b.y, c.x, c.y, e.x, e.y};
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vals[i], acc[i] * corr);
  m = mn;
}

// Exclusive scan of the clamped per-unit row counts into pre[0..units] (pre[units] = R).
// cnt_per_seq: the count of unit u is cnt[u / H] (dense attention) instead of cnt[u].
__device__ void scan_counts(const int32_t* cnt, int cnt_per_seq, int H, int units, int Lcap, int* pre,
                            int* wsum, int* err) {
  const int per = (units + kAttThreads - 1) / kAttThreads;
  const int u0 = threadIdx.x * per;
  int local = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) {
    int c = cnt_per_seq ? cnt[u / H] : cnt[u];
    if (c < 0 || c > Lcap) {
      raise_error(err, IG_DEVERR_INDEX);
      c = c < 0 ? 0 : Lcap;
    }
    pre[u + 1] = c;
    local += c;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += wsum[w];
  if (threadIdx.x == 0) pre[0] = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) {
    run += pre[u + 1];
    pre[u + 1] = run;
  }
  __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kAttThreads) k5_attend(
    const __half* __restrict__ q, const __half* __restrict__ Kg, const __half* __restrict__ Vg,
    const int32_t* __restrict__ cnt, int cnt_per_seq, int H, int Lcap, int units, float scale,
    float* __restrict__ ws, int* err) {
  constexpr int VPR = D / 8;                    // lanes per row
  constexpr int RPW = 32 / VPR;                 // rows per warp step
  constexpr int NG = (kAttThreads / 32) * RPW;  // lane groups per CTA
  extern __shared__ int pre[];                  // [units + 1]
  __shared__ int wsum[kAttThreads / 32];
  __shared__ float sm_m[NG], sm_l[NG];
  __shared__ float sm_acc[NG][D];
  scan_counts(cnt, cnt_per_seq, H, units, Lcap, pre, wsum, err);
  const long long R = pre[units];
  int r0 = (int)(R * blockIdx.x / gridDim.x);
  const int r1 = (int)(R * (blockIdx.x + 1) / gridDim.x);
  if (r0 >= r1) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v = lane % VPR, sub = lane / VPR, g = warp * RPW + sub;
  int u;
  {
    int lo = 0, hi = units;  // first unit whose rows end after r0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid + 1] <= r0) lo = mid + 1; else hi = mid;
    }
    u = lo;
  }
  while (r0 < r1) {
    const int seg_end = min(r1, pre[u + 1]);
    const int j0 = r0 - pre[u], j1 = seg_end - pre[u];
    float qf[8];
    {
      uint4 qv = *reinterpret_cast<const uint4*>(q + (size_t)u * D + v * 8);
      float2 a = h2_to_f2(qv.x), b = h2_to_f2(qv.y), cc = h2_to_f2(qv.z), e = h2_to_f2(qv.w);
      qf[0] = a.x * scale; qf[1] = a.y * scale; qf[2] = b.x * scale; qf[3] = b.y * scale;
      qf[4] = cc.x * scale; qf[5] = cc.y * scale; qf[6] = e.x * scale; qf[7] = e.y * scale;
    }
    float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    const uint4* Kb = reinterpret_cast<const uint4*>(Kg + (size_t)u * Lcap * D) + v;
    const uint4* Vb = reinterpret_cast<const uint4*>(Vg + (size_t)u * Lcap * D) + v;
    // warp-uniform trip count (the shuffles take the full mask); a group past the end
    // computes on zeros and skips the update
    for (int jw = j0 + warp * RPW; jw < j1; jw += NG * kAttUnroll) {
      uint4 kv[kAttUnroll], vv[kAttUnroll];
#pragma unroll
      for (int x = 0; x < kAttUnroll; ++x) {
        const int jj = jw + sub + x * NG;
        kv[x] = make_uint4(0, 0, 0, 0);
        vv[x] = make_uint4(0, 0, 0, 0);
        if (jj < j1) {
          kv[x] = __ldg(Kb + (size_t)jj * VPR);
          vv[x] = __ldg(Vb + (size_t)jj * VPR);
        }
      }
#pragma unroll
      for (int x = 0; x < kAttUnroll; ++x) {
        const int jj = jw + sub + x * NG;
        const float z = group_sum<VPR>(lane_dot(qf, kv[x]));
        if (jj < j1) online_add(z, vv[x], m, l, acc);
      }
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
    float* w = ws + ((size_t)u + blockIdx.x) * (D + 2);
    for (int dd = threadIdx.x; dd < D; dd += kAttThreads) {
      float o = 0.f;
      for (int i = 0; i < NG; ++i)
        if (sm_m[i] != -INFINITY) o += sm_acc[i][dd] * __expf(sm_m[i] - M);
      w[2 + dd] = o;
    }
    if (threadIdx.x == 0) {
      float Ls = 0.f;
      for (int i = 0; i < NG; ++i)
        if (sm_m[i] != -INFINITY) Ls += sm_l[i] * __expf(sm_m[i] - M);
      w[0] = M;
      w[1] = Ls;
    }
    __syncthreads();  // smem is reused by the next segment
    r0 = seg_end;
    while (u < units - 1 && pre[u + 1] <= r0) ++u;
  }
}

// CTA of the balanced grid whose row range holds row r (the last c with start(c) <= r).
__device__ __forceinline__ int cta_of(long long r, long long R, int G) {
  int c = (int)((r * G) / R);
  while (c + 1 < G && (R * (c + 1)) / G <= r) ++c;
  while (c > 0 && (R * c) / G > r) --c;
  return c;
}

// One CTA (d threads) per head: merges the partials of the CTAs that covered its rows, adds
// the current token, normalises.
template <int D>
__global__ void __launch_bounds__(D) k5_combine(const float* __restrict__ ws, const int32_t* __restrict__ cnt,
                                                int cnt_per_seq, int H, int Lcap, int units, int G,
                                                const __half* __restrict__ q,
                                                const __half* __restrict__ k_new,
                                                const __half* __restrict__ v_new, float scale,
                                                float* __restrict__ out) {
  __shared__ float red[D / 32];
  __shared__ long long sh_lo, sh_R;
  const int u = blockIdx.x, dd = threadIdx.x;
  // rows before this head and in total (clamped counts, as in the main kernel)
  long long before = 0, total = 0;
  for (int x = threadIdx.x; x < units; x += D) {
    int c = cnt_per_seq ? cnt[x / H] : cnt[x];
    c = c < 0 ? 0 : (c > Lcap ? Lcap : c);
    total += c;
    if (x < u) before += c;
  }
  for (int o = 16; o; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  __shared__ long long sb[D / 32], st[D / 32];
  if ((threadIdx.x & 31) == 0) {
    sb[threadIdx.x >> 5] = before;
    st[threadIdx.x >> 5] = total;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long b = 0, t = 0;
    for (int i = 0; i < D / 32; ++i) {
      b += sb[i];
      t += st[i];
    }
    sh_lo = b;
    sh_R = t;
  }
  __syncthreads();
  const long long lo = sh_lo, R = sh_R;
  int c = cnt_per_seq ? cnt[u / H] : cnt[u];
  c = c < 0 ? 0 : (c > Lcap ? Lcap : c);
  float M = -INFINITY, Ls = 0.f, o = 0.f;
  if (c > 0) {
    // CTAs c0..c1 cover this head's rows; those with an empty range (fewer rows than CTAs)
    // wrote nothing and are skipped
    const int c0 = cta_of(lo, R, G), c1 = cta_of(lo + c - 1, R, G);
    for (int cc = c0; cc <= c1; ++cc)
      if ((R * cc) / G < (R * (cc + 1)) / G) M = fmaxf(M, ws[((size_t)u + cc) * (D + 2)]);
    for (int cc = c0; cc <= c1; ++cc) {
      if ((R * cc) / G == (R * (cc + 1)) / G) continue;
      const float* w = ws + ((size_t)u + cc) * (D + 2);
      if (w[0] == -INFINITY) continue;
      const float f = __expf(w[0] - M);
      Ls += w[1] * f;
      o += w[2 + dd] * f;
    }
  }
  if (k_new) {
    // the current token's own key and value (always attended)
    float part = __half2float(q[(size_t)u * D + dd]) * scale * __half2float(k_new[(size_t)u * D + dd]);
    for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((dd & 31) == 0) red[dd >> 5] = part;
    __syncthreads();
    float z = 0.f;
    for (int i = 0; i < D / 32; ++i) z += red[i];
    const float Mn = fmaxf(M, z);
    const float f = (M == -INFINITY) ? 0.f : __expf(M - Mn);
    const float p = __expf(z - Mn);
    Ls = Ls * f + p;
    o = o * f + p * __half2float(v_new[(size_t)u * D + dd]);
    M = Mn;
  }
  out[(size_t)u * D + dd] = Ls > 0.f ? o / Ls : 0.f;
}

inline int att_grid() {
  int g = 4 * sm_count();
  return g > kMaxAttCtas ? kMaxAttCtas : g;
}

template <int D>
ig_status launch_attend(cudaStream_t st, int B, int H, int Lcap, float scale, const uint16_t* q,
                        const uint16_t* K, const uint16_t* V, const int32_t* cnt, int per_seq,
                        const uint16_t* kn, const uint16_t* vn, float* out, void* ws) {
  const int units = B * H;
  const int G = att_grid();
  const size_t smem = (size_t)(units + 1) * sizeof(int);
  if (smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k5_attend<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "attention smem attribute");
  }
  k5_attend<D><<<G, kAttThreads, smem, st>>>(
      reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(K),
      reinterpret_cast<const __half*>(V), cnt, per_seq, H, Lcap, units, scale, static_cast<float*>(ws),
      error_word());
  IG_CHECK_LAUNCH("attention launch");
  k5_combine<D><<<units, D, 0, st>>>(static_cast<const float*>(ws), cnt, per_seq, H, Lcap, units, G,
                                     reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(kn),
                                     reinterpret_cast<const __half*>(vn), scale, out);
  IG_CHECK_LAUNCH("attention combine launch");
  return IG_OK;
}

size_t attend_ws_bytes(int B, int H, int d) {
  return round_up((size_t)(B * H + kMaxAttCtas) * (d + 2) * sizeof(float), 256);
}

ig_status attend_common(void* stream, int B, int H, int d, int Lcap, float scale,
                        const uint16_t* q, const uint16_t* K, const uint16_t* V,
                        const int32_t* cnt, int per_seq, const uint16_t* kn, const uint16_t* vn,
                        float* out, void* ws, size_t ws_bytes) {
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128 (got %d)", d);
  IG_REQUIRE(B * H <= kMaxAttUnits, "B*H = %d exceeds %d", B * H, kMaxAttUnits);
  IG_REQUIRE((long long)B * H * Lcap < (1ll << 31), "B*H*Lcap must stay below 2^31 rows");
  IG_REQUIRE(q && K && V && cnt && out, "null pointer argument");
  IG_REQUIRE((kn == nullptr) == (vn == nullptr), "k_new and v_new go together");
  IG_REQUIRE(aligned(q, 16) && aligned(K, 16) && aligned(V, 16), "q, K, V must be 16-byte aligned");
  IG_REQUIRE(!kn || (aligned(kn, 16) && aligned(vn, 16)), "k_new, v_new must be 16-byte aligned");
  const size_t need = attend_ws_bytes(B, H, d);
  if (!ws || ws_bytes < need) return fail(IG_ERR_CAPACITY, "attention needs %zu workspace bytes", need);
  IG_REQUIRE(aligned(ws, 256), "workspace must be 256-byte aligned");
  cudaStream_t s = as_stream(stream);
  if (d == 128) return launch_attend<128>(s, B, H, Lcap, scale, q, K, V, cnt, per_seq, kn, vn, out, ws);
  return launch_attend<64>(s, B, H, Lcap, scale, q, K, V, cnt, per_seq, kn, vn, out, ws);
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" size_t ig_attend_workspace_bytes(int B, int H, int d, int Lcap) {
  if (B <= 0 || H <= 0 || d <= 0 || Lcap <= 0) return 0;
  return attend_ws_bytes(B, H, d);
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
