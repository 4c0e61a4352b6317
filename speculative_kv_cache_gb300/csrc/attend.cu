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
#include <cuda_fp8.h>
#include <math.h>

#include "ig_common.cuh"
#include "pool_impl.h"

namespace ig {
namespace {

constexpr int kAttThreads = 128;
constexpr int kAttUnroll = 4;
constexpr int kMaxAttCtas = 2048;   // upper bound of the balanced grid (sizes the workspace)
constexpr int kMaxAttUnits = 16384; // (units + 1) ints of shared memory for the scan
#ifndef IG_FA_THREADS
#define IG_FA_THREADS 256
#endif
#ifndef IG_FA_MIN_CTAS
#define IG_FA_MIN_CTAS 1
#endif
constexpr int kFaThreads = IG_FA_THREADS;  // fused fetch + attention: as the gather (host-link bound)
#ifndef IG_FA_UNROLL
#define IG_FA_UNROLL 6
#endif
#ifndef IG_FA_UNROLL_Q
#define IG_FA_UNROLL_Q IG_FA_UNROLL
#endif
// rows per batch and lane group (two batches in flight): fp16 rows, quantized rows
__host__ __device__ constexpr int fa_unroll(int bits) { return bits ? IG_FA_UNROLL_Q : IG_FA_UNROLL; }
constexpr int kMaxFaCtas = 256;     // upper bound of its grid (sizes its workspace)
// a partial in the workspace: [max, sum, -, -, unnormalised output[D]] (D + 4 floats, so
// that the output part of every partial starts on a 16-byte boundary)
constexpr int kPartHead = 4;

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
// The counts are first copied to shared memory with coalesced loads, kScanBatch of them in
// flight per thread (one round trip for up to kScanBatch * THREADS units: this prologue is on
// every CTA's critical path), then each thread sums a contiguous chunk and the chunk sums are
// scanned across the block.
constexpr int kScanBatch = 8;
template <int THREADS>
__device__ void scan_counts(const int32_t* cnt, int cnt_per_seq, int H, int units, int Lcap, int* pre,
                            int* wsum, int* err) {
  for (int base = 0; base < units; base += kScanBatch * THREADS) {
    int c[kScanBatch];
#pragma unroll
    for (int x = 0; x < kScanBatch; ++x) {
      const int u = base + x * THREADS + (int)threadIdx.x;
      c[x] = u < units ? (cnt_per_seq ? cnt[u / H] : cnt[u]) : 0;
    }
#pragma unroll
    for (int x = 0; x < kScanBatch; ++x) {
      const int u = base + x * THREADS + (int)threadIdx.x;
      if (u < units) {
        int v = c[x];
        if (v < 0 || v > Lcap) {
          raise_error(err, IG_DEVERR_INDEX);
          v = v < 0 ? 0 : Lcap;
        }
        pre[u + 1] = v;
      }
    }
  }
  __syncthreads();
  const int per = (units + THREADS - 1) / THREADS;
  const int u0 = threadIdx.x * per;
  int local = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) local += pre[u + 1];
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
    float* __restrict__ ws, int* __restrict__ gpre, int* err) {
  constexpr int VPR = D / 8;                    // lanes per row
  constexpr int RPW = 32 / VPR;                 // rows per warp step
  constexpr int NG = (kAttThreads / 32) * RPW;  // lane groups per CTA
  extern __shared__ int pre[];                  // [units + 1]
  __shared__ int wsum[kAttThreads / 32];
  __shared__ float sm_m[NG], sm_l[NG];
  __shared__ float sm_acc[NG][D];
  pdl_trigger();  // the combine may be scheduled now; it waits for this grid to complete
  scan_counts<kAttThreads>(cnt, cnt_per_seq, H, units, Lcap, pre, wsum, err);
  if (blockIdx.x == 0)  // the row prefix, for the combine
    for (int i = threadIdx.x; i <= units; i += kAttThreads) gpre[i] = pre[i];
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
    float* w = ws + ((size_t)u + blockIdx.x) * (D + kPartHead);
    for (int dd = threadIdx.x; dd < D; dd += kAttThreads) {
      float o = 0.f;
      for (int i = 0; i < NG; ++i)
        if (sm_m[i] != -INFINITY) o += sm_acc[i][dd] * __expf(sm_m[i] - M);
      w[kPartHead + dd] = o;
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

// Fused fetch + attention straight from the pinned pool.  The CTA's rows (the same balanced
// split as above) are streamed as in the gather, without stopping at head boundaries: lane
// group g takes rows start + g, start + g + NG, ..., fa_unroll(BITS) of them in flight, each with
// its head's query chunk (loaded where the head changes), and keeps one online softmax for its
// current head.  When its next
// row belongs to another head it writes its partial to ws[(head + CTA) * NG + g] and starts
// afresh, so a group writes one partial per head it touches and no CTA-wide barrier sits on
// the load path.  Every slot is range-checked; a bad one is skipped and flagged.
// BITS = 0: fp16 rows (Kp, Vp); BITS = 8 or 4: a quantized pool's code records (Rec, rec bytes
// each: K codes then V codes) and the rows' scales in device memory (Sc, [row][2]).  A lane
// loads the 8 codes of its 8 elements (8 or 4 bytes) of the key and of the value and dequantizes
// them when the row is folded in, exactly as the staged fetch does (code value x scale in fp32,
// rounded to fp16), so the attention sees the same values.
template <int BITS>
struct FaRow;  // the raw data a lane holds for one row in flight
template <>
struct FaRow<0> {
  uint4 k, v;
};
template <>
struct FaRow<8> {
  uint2 k, v;
  float2 s;
};
template <>
struct FaRow<4> {
  uint32_t k, v;
  float2 s;
};

// 8 codes (one lane's share of a row) and their scale -> 8 fp16 values packed in a uint4
__device__ __forceinline__ uint4 dq8(uint2 c, float sc) {
  const uint32_t w[2] = {c.x, c.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
    const __half2 ra = __floats2half2_rn(a.x * sc, a.y * sc);
    const __half2 rb = __floats2half2_rn(b.x * sc, b.y * sc);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&ra);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&rb);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ uint4 dq4(uint32_t c, float sc) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c0 = (int)(c << (28 - 8 * j)) >> 28;
    const int c1 = (int)(c << (24 - 8 * j)) >> 28;
    const __half2 r = __floats2half2_rn((float)c0 * sc, (float)c1 * sc);
    o[j] = *reinterpret_cast<const uint32_t*>(&r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int D, int BITS>
__global__ void __launch_bounds__(kFaThreads, IG_FA_MIN_CTAS) k5_fetch_attend(
    const __half* __restrict__ q, const uint4* __restrict__ Kp, const uint4* __restrict__ Vp,
    const uint8_t* __restrict__ Rec, int rec, const float* __restrict__ Sc,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int H, int Lcap, int units,
    int cap, float scale, float* __restrict__ ws, int* __restrict__ gpre, int* err) {
  constexpr int VPR = D / 8;                  // lanes per row
  constexpr int RPW = 32 / VPR;               // rows per warp step
  constexpr int NG = (kFaThreads / 32) * RPW; // lane groups per CTA
  extern __shared__ int pre[];                // [units + 1]
  __shared__ int wsum[kFaThreads / 32];
  scan_counts<kFaThreads>(cnt, 0, H, units, Lcap, pre, wsum, err);
  if (blockIdx.x == 0)  // the row prefix, for the combine
    for (int i = threadIdx.x; i <= units; i += kFaThreads) gpre[i] = pre[i];
  const long long R = pre[units];
  const int r0 = (int)(R * blockIdx.x / gridDim.x);
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
  int cur = -1;  // head of the running partial (and of qf)
  float m = -INFINITY, l = 0.f, acc[8], qf[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = qf[i] = 0.f;
  auto flush = [&]() {
    // 16-byte aligned: ws is 256-byte aligned and (D + kPartHead) floats is a multiple of 16 B
    float* w = ws + ((size_t)(cur + blockIdx.x) * NG + g) * (D + kPartHead);
    *reinterpret_cast<float4*>(w + kPartHead + v * 8) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(w + kPartHead + 4 + v * 8) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (v == 0) {
      w[0] = m;
      w[1] = l;
    }
  };
  constexpr int kFaU = fa_unroll(BITS);
  // Software pipeline over batches of kFaU rows per group: the loads of batch n + 1
  // (index, then pool rows and, where the head changes, the query chunk) are issued before
  // batch n is folded in, so the host link always has this group's rows in flight.
  auto prepare = [&](int rw, int (&hu)[kFaU], int (&slot)[kFaU]) {
#pragma unroll
    for (int x = 0; x < kFaU; ++x) {
      const int rr = rw + sub + x * NG;
      hu[x] = -1;
      slot[x] = -1;
      if (rr < r1) {
        while (pre[u + 1] <= rr) ++u;
        hu[x] = u;
        const int sl = idx[(size_t)u * Lcap + (rr - pre[u])];
        if (sl < 0 || sl >= cap) raise_error(err, IG_DEVERR_INDEX);
        else slot[x] = sl;
      }
    }
  };
  // the query chunk is loaded only where the head changes (a group's rows mostly share one)
  auto issue = [&](const int (&hu)[kFaU], const int (&slot)[kFaU], int prev, FaRow<BITS> (&rw_)[kFaU],
                   uint4 (&qv)[kFaU]) {
#pragma unroll
    for (int x = 0; x < kFaU; ++x) {
      rw_[x] = FaRow<BITS>{};
      qv[x] = make_uint4(0, 0, 0, 0);
      if (hu[x] >= 0 && hu[x] != (x == 0 ? prev : hu[x - 1]))
        qv[x] = *reinterpret_cast<const uint4*>(q + (size_t)hu[x] * D + v * 8);
      if (slot[x] >= 0) {
        const size_t row = (size_t)hu[x] * cap + slot[x];
        if constexpr (BITS == 0) {
          rw_[x].k = ld_nc_v4(Kp + row * VPR + v);
          rw_[x].v = ld_nc_v4(Vp + row * VPR + v);
        } else if constexpr (BITS == 8) {
          const uint8_t* rp = Rec + row * rec;
          rw_[x].k = ld_nc_v2(rp + (size_t)v * 8);
          rw_[x].v = ld_nc_v2(rp + D + (size_t)v * 8);
          rw_[x].s = __ldg(reinterpret_cast<const float2*>(Sc) + row);
        } else {
          const uint8_t* rp = Rec + row * rec;
          rw_[x].k = ld_nc_u32(rp + (size_t)v * 4);
          rw_[x].v = ld_nc_u32(rp + D / 2 + (size_t)v * 4);
          rw_[x].s = __ldg(reinterpret_cast<const float2*>(Sc) + row);
        }
      }
    }
  };
  auto key_of = [&](const FaRow<BITS>& r) -> uint4 {
    if constexpr (BITS == 0) return r.k;
    else if constexpr (BITS == 8) return dq8(r.k, r.s.x);
    else return dq4(r.k, r.s.x);
  };
  auto value_of = [&](const FaRow<BITS>& r) -> uint4 {
    if constexpr (BITS == 0) return r.v;
    else if constexpr (BITS == 8) return dq8(r.v, r.s.y);
    else return dq4(r.v, r.s.y);
  };
  int hu[kFaU], slot[kFaU], hn[kFaU], sn[kFaU];
  FaRow<BITS> cu[kFaU], nx[kFaU];
  uint4 qv[kFaU], qn[kFaU];
  int rw = r0 + warp * RPW;
  prepare(rw, hu, slot);
  issue(hu, slot, -1, cu, qv);
  // warp-uniform trip count (the shuffles take the full mask); rows past the end compute on
  // zeros and change nothing
  while (rw < r1) {
    const int rnext = rw + NG * kFaU;
    int last = cur;  // head of the last row of this batch (the query in use when the next starts)
#pragma unroll
    for (int x = 0; x < kFaU; ++x) last = hu[x] >= 0 ? hu[x] : last;
    prepare(rnext, hn, sn);
    issue(hn, sn, last, nx, qn);
#pragma unroll
    for (int x = 0; x < kFaU; ++x) {
      if (hu[x] >= 0 && hu[x] != cur) {  // a new head: hand over the previous one's partial
        if (cur >= 0) flush();
        cur = hu[x];
        m = -INFINITY;
        l = 0.f;
        float2 a = h2_to_f2(qv[x].x), b = h2_to_f2(qv[x].y), c = h2_to_f2(qv[x].z), e = h2_to_f2(qv[x].w);
        qf[0] = a.x * scale; qf[1] = a.y * scale; qf[2] = b.x * scale; qf[3] = b.y * scale;
        qf[4] = c.x * scale; qf[5] = c.y * scale; qf[6] = e.x * scale; qf[7] = e.y * scale;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      const float z = group_sum<VPR>(lane_dot(qf, key_of(cu[x])));
      if (slot[x] >= 0) online_add(z, value_of(cu[x]), m, l, acc);
    }
#pragma unroll
    for (int x = 0; x < kFaU; ++x) {
      hu[x] = hn[x];
      slot[x] = sn[x];
      cu[x] = nx[x];
      qv[x] = qn[x];
    }
    rw = rnext;
  }
  if (cur >= 0) flush();
}

// CTA of the balanced grid whose row range holds row r (the last c with start(c) <= r).
__device__ __forceinline__ int cta_of(long long r, long long R, int G) {
  int c = (int)((r * G) / R);
  while (c + 1 < G && (R * (c + 1)) / G <= r) ++c;
  while (c > 0 && (R * c) / G > r) --c;
  return c;
}

// One CTA (d threads) per head: merges the partials of the CTAs that covered its rows, adds
// the current token, normalises.  NGP partials per (head, CTA): 1 for the staged attention;
// the lane-group count for the fused fetch, where group g of CTA cc holds a partial for the
// head iff one of the head's rows in that CTA's range is g's (rows go round-robin to groups).
// The head's candidate partials are numbered t = (cc - c0) * NGP + g and taken D at a time,
// one per thread, so their loads are issued together rather than one after another; the
// sums still run over t in order.
template <int D, int NGP>
__global__ void __launch_bounds__(D) k5_combine(const float* __restrict__ ws, const int* __restrict__ gpre,
                                                int units, int G, const __half* __restrict__ q,
                                                const __half* __restrict__ k_new,
                                                const __half* __restrict__ v_new, float scale,
                                                float* __restrict__ out) {
  __shared__ float red[D / 32];
  __shared__ float sf[D], sl[D];
  __shared__ int sw[D];
  // after the attention (launched as its programmatic dependent): its partials and prefix
  pdl_wait();
  const int u = blockIdx.x, dd = threadIdx.x;
  // rows before this head, its rows and all rows (the main kernel's clamped prefix)
  const long long lo = gpre[u], R = gpre[units];
  const int c = gpre[u + 1] - gpre[u];
  float M = -INFINITY, Ls = 0.f, o = 0.f;
  if (c > 0) {
    // CTAs c0..c1 cover this head's rows; those with an empty range (fewer rows than CTAs)
    // wrote nothing, and are skipped
    const int c0 = cta_of(lo, R, G), c1 = cta_of(lo + c - 1, R, G);
    const int P = (c1 - c0 + 1) * NGP;
    // offset (in floats) of candidate t's partial, or -1 where it holds none
    auto where = [&](int t) -> long long {
      const int cc = c0 + t / NGP, gi = t % NGP;
      const long long s0 = (R * cc) / G, s1 = (R * (cc + 1)) / G;
      if (s0 == s1) return -1;
      if (NGP > 1) {
        const long long a = lo > s0 ? lo : s0, e = (lo + c) < s1 ? (lo + c) : s1;
        const long long n = e - a, off = (a - s0) % NGP;
        if (n < NGP && (gi - off + NGP) % NGP >= n) return -1;
      }
      return (((long long)u + cc) * NGP + gi) * (D + kPartHead);
    };
    for (int base = 0; base < P; base += D) {  // the head's maximum
      const int t = base + dd;
      const long long w = t < P ? where(t) : -1;
      float mt = w >= 0 ? ws[w] : -INFINITY;
      for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      if ((dd & 31) == 0) red[dd >> 5] = mt;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < D / 32; ++i) M = fmaxf(M, red[i]);
      __syncthreads();
    }
    for (int base = 0; base < P; base += D) {  // weights, then the sums in candidate order
      const int t = base + dd;
      const long long w = t < P ? where(t) : -1;
      const float mt = w >= 0 ? ws[w] : -INFINITY;
      const bool live = mt != -INFINITY;
      sf[dd] = live ? __expf(mt - M) : 0.f;
      sl[dd] = live ? ws[w + 1] : 0.f;
      sw[dd] = live ? (int)(w / (D + kPartHead)) : -1;
      __syncthreads();
      const int n = min(D, P - base);
#pragma unroll 4
      for (int i = 0; i < n; ++i) {
        const int wi = sw[i];
        if (wi >= 0) {
          const float f = sf[i];
          Ls += sl[i] * f;
          o += ws[(size_t)wi * (D + kPartHead) + kPartHead + dd] * f;
        }
      }
      __syncthreads();
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

// workspace: the partials, then the row prefix [units + 1] ints
inline size_t att_part_bytes(int B, int H, int d) {
  return round_up((size_t)(B * H + kMaxAttCtas) * (d + kPartHead) * sizeof(float), 256);
}
template <int D>
constexpr int fa_groups() { return (kFaThreads / 32) * (32 / (D / 8)); }
inline size_t fa_part_bytes(int B, int H, int d) {
  const int ng = d == 64 ? fa_groups<64>() : fa_groups<128>();
  return round_up((size_t)(B * H + kMaxFaCtas) * ng * (d + kPartHead) * sizeof(float), 256);
}
inline size_t prefix_bytes(int B, int H) { return round_up((size_t)(B * H + 1) * sizeof(int), 256); }

// 8 CTAs of 4 warps per SM (the register limit at 64 per thread): 32 warps, 8 rows in flight
// each, to cover the memory latency
#ifndef IG_ATT_CTAS_PER_SM
#define IG_ATT_CTAS_PER_SM 8
#endif
inline int att_grid(cudaStream_t st) {
  int g = IG_ATT_CTAS_PER_SM * sm_count(st);
  return g > kMaxAttCtas ? kMaxAttCtas : g;
}

template <int D>
ig_status launch_attend(cudaStream_t st, int B, int H, int Lcap, float scale, const uint16_t* q,
                        const uint16_t* K, const uint16_t* V, const int32_t* cnt, int per_seq,
                        const uint16_t* kn, const uint16_t* vn, float* out, void* ws) {
  const int units = B * H;
  const int G = att_grid(st);
  const size_t smem = (size_t)(units + 1) * sizeof(int);
  if (smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k5_attend<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "attention smem attribute");
  }
  int* gpre = reinterpret_cast<int*>(static_cast<char*>(ws) + att_part_bytes(B, H, D));
  k5_attend<D><<<G, kAttThreads, smem, st>>>(reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(K),
                                            reinterpret_cast<const __half*>(V), cnt, per_seq, H, Lcap, units,
                                            scale, static_cast<float*>(ws), gpre, error_word());
  IG_CHECK_LAUNCH("attention launch");
  {
    // a programmatic dependent launch: the combine's CTAs are scheduled as the attention's
    // finish, instead of after a full launch gap (Llama-2-7B alpha = 2 layer: 24.8 -> 21.2 us)
    cudaError_t ce = launch_pdl(k5_combine<D, 1>, dim3(units), dim3(D), 0, st, static_cast<const float*>(ws),
                                static_cast<const int*>(gpre), units, G, reinterpret_cast<const __half*>(q),
                                reinterpret_cast<const __half*>(kn), reinterpret_cast<const __half*>(vn), scale, out);
    if (ce != cudaSuccess) return cuda_fail(ce, "attention combine launch");
    IG_CHECK_LAUNCH("attention combine launch");
  }
  return IG_OK;
}

template <int D, int BITS>
ig_status launch_fetch_partials(cudaStream_t st, int B, int H, int Lcap, int cap, float scale, const uint16_t* q,
                                const uint16_t* Kp, const uint16_t* Vp, const uint8_t* Rec, int rec, const float* Sc,
                                const int32_t* idx, const int32_t* cnt, void* ws, int grid) {
  const int units = B * H;
  const size_t smem = (size_t)(units + 1) * sizeof(int);
  if (smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k5_fetch_attend<D, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "fetch-attention smem attribute");
  }
  int* gpre = reinterpret_cast<int*>(static_cast<char*>(ws) + fa_part_bytes(B, H, D));
  k5_fetch_attend<D, BITS><<<grid, kFaThreads, smem, st>>>(
      reinterpret_cast<const __half*>(q), reinterpret_cast<const uint4*>(Kp), reinterpret_cast<const uint4*>(Vp), Rec,
      rec, Sc, idx, cnt, H, Lcap, units, cap, scale, static_cast<float*>(ws), gpre, error_word());
  IG_CHECK_LAUNCH("fetch-attention launch");
  return IG_OK;
}

template <int D>
ig_status launch_fetch_combine(cudaStream_t st, int B, int H, float scale, const uint16_t* q, const uint16_t* kn,
                               const uint16_t* vn, float* out, const void* ws, int grid) {
  const int units = B * H;
  const int* gpre = reinterpret_cast<const int*>(static_cast<const char*>(ws) + fa_part_bytes(B, H, D));
  k5_combine<D, fa_groups<D>()><<<units, D, 0, st>>>(
      static_cast<const float*>(ws), gpre, units, grid, reinterpret_cast<const __half*>(q),
      reinterpret_cast<const __half*>(kn), reinterpret_cast<const __half*>(vn), scale, out);
  IG_CHECK_LAUNCH("fetch-attention combine launch");
  return IG_OK;
}

size_t fetch_attend_ws_bytes(int B, int H, int d) { return fa_part_bytes(B, H, d) + prefix_bytes(B, H); }

size_t attend_ws_bytes(int B, int H, int d) { return att_part_bytes(B, H, d) + prefix_bytes(B, H); }

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
ig_status check_pool_device(const ig_pool* pool);
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

extern "C" size_t ig_gather_attend_workspace_bytes(int B, int H, int d, int Lcap) {
  if (B <= 0 || H <= 0 || (d != 64 && d != 128) || Lcap <= 0) return 0;
  return fetch_attend_ws_bytes(B, H, d);
}

namespace ig {

// The fused fetch + attention in its two launches: the partials (the pool read over the host
// link, on `st`) and the combine (a CTA per head merges them, adds the current token and
// normalises).  The decode step puts the combine on its compute stream so that the fetch
// stream moves straight on to the next layer's rows; *grid_out is the partials' grid, which
// the combine needs.
ig_status fetch_attend_partials(cudaStream_t s, const ig_pool* pool, int layer, int B, int H, int d, int Lcap,
                                float scale, const uint16_t* q, const int32_t* idx, const int32_t* cnt,
                                const uint16_t* k_new, const uint16_t* v_new, const float* out, void* workspace,
                                size_t workspace_bytes, int max_ctas, int* grid_out) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(pool->storage, "the pool was created without storage");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  if (ig_status dst = check_pool_device(pool); dst != IG_OK) return dst;
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  IG_REQUIRE(B > 0 && H > 0 && Lcap > 0, "B, H, Lcap must be positive");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128 (got %d)", d);
  IG_REQUIRE(B * H <= kMaxAttUnits, "B*H = %d exceeds %d", B * H, kMaxAttUnits);
  IG_REQUIRE((long long)B * H * Lcap < (1ll << 31), "B*H*Lcap must stay below 2^31 rows");
  IG_REQUIRE(q && idx && cnt && out, "null pointer argument");
  IG_REQUIRE((k_new == nullptr) == (v_new == nullptr), "k_new and v_new go together");
  IG_REQUIRE(aligned(q, 16), "q must be 16-byte aligned");
  IG_REQUIRE(!k_new || (aligned(k_new, 16) && aligned(v_new, 16)), "k_new, v_new must be 16-byte aligned");
  IG_REQUIRE(max_ctas >= 0 && max_ctas <= kMaxFaCtas, "max_ctas must be in [0, %d]", kMaxFaCtas);
  const size_t need = fetch_attend_ws_bytes(B, H, d);
  if (!workspace || workspace_bytes < need)
    return fail(IG_ERR_CAPACITY, "fused fetch + attention needs %zu workspace bytes", need);
  IG_REQUIRE(aligned(workspace, 256), "workspace must be 256-byte aligned");
  // the same default as the gather (twice it for a quantized pool, whose rows need dequantizing)
  int grid = max_ctas > 0 ? max_ctas : (pool->qbits ? 2 : 1) * (256 / kFaThreads) * fetch_grid(s);
  if (grid < 1) grid = 1;
  if (grid > kMaxFaCtas) grid = kMaxFaCtas;
  *grid_out = grid;
  const size_t rows = (size_t)B * H * pool->cap;
  if (pool->qbits) {
    const uint8_t* Rec = pool->R + (size_t)layer * rows * pool->rec;
    const float* Sc = pool->S + (size_t)layer * rows * 2;
#define IG_FA_Q(DD, BB)                                                                                      \
  return launch_fetch_partials<DD, BB>(s, B, H, Lcap, pool->cap, scale, q, nullptr, nullptr, Rec, pool->rec, Sc, \
                                       idx, cnt, workspace, grid)
    if (pool->qbits == 8) {
      if (d == 128) IG_FA_Q(128, 8);
      IG_FA_Q(64, 8);
    }
    if (d == 128) IG_FA_Q(128, 4);
    IG_FA_Q(64, 4);
#undef IG_FA_Q
  }
  const uint16_t* Kp = pool->Kdev + (size_t)layer * rows * d;
  const uint16_t* Vp = pool->Vdev + (size_t)layer * rows * d;
  if (d == 128)
    return launch_fetch_partials<128, 0>(s, B, H, Lcap, pool->cap, scale, q, Kp, Vp, nullptr, 0, nullptr, idx, cnt,
                                         workspace, grid);
  return launch_fetch_partials<64, 0>(s, B, H, Lcap, pool->cap, scale, q, Kp, Vp, nullptr, 0, nullptr, idx, cnt,
                                      workspace, grid);
}

// The combine of fetch_attend_partials' launch (same B, H, d, workspace and grid); the caller
// orders it after the partials.
ig_status fetch_attend_combine(cudaStream_t s, int B, int H, int d, float scale, const uint16_t* q,
                               const uint16_t* k_new, const uint16_t* v_new, float* out, const void* workspace,
                               int grid) {
  if (d == 128) return launch_fetch_combine<128>(s, B, H, scale, q, k_new, v_new, out, workspace, grid);
  return launch_fetch_combine<64>(s, B, H, scale, q, k_new, v_new, out, workspace, grid);
}

}  // namespace ig

extern "C" ig_status ig_gather_attend(void* stream, const ig_pool* pool, int layer, int B, int H,
                                      int d, int Lcap, float scale, const uint16_t* q,
                                      const int32_t* idx, const int32_t* cnt,
                                      const uint16_t* k_new, const uint16_t* v_new, float* out,
                                      void* workspace, size_t workspace_bytes, int max_ctas) {
  cudaStream_t s = as_stream(stream);
  int grid = 0;
  ig_status st = fetch_attend_partials(s, pool, layer, B, H, d, Lcap, scale, q, idx, cnt, k_new, v_new, out,
                                       workspace, workspace_bytes, max_ctas, &grid);
  if (st != IG_OK) return st;
  return fetch_attend_combine(s, B, H, d, scale, q, k_new, v_new, out, workspace, grid);
}
