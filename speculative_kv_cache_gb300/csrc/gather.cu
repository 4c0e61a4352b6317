// Gather of the chosen full key/value rows from the pinned host pool into HBM
// (InfiniGen paper-graph summary, section 3.4, "Decoding Stage", Step 5).
//
// The pool is mapped pinned host memory, readable by the GPU over the host link, so the
// fetch is a kernel of zero-copy 16-byte loads rather than one copy call per row: for d = 128
// a row is 256 B and 16 lanes fetch it together; each lane keeps 2 x kUnroll loads in flight
// (keys and values).  The grid is kept small (a fraction of the SMs): the host link saturates
// with a few dozen CTAs, and the rest of the GPU stays free for the compute stream.
//
// Balance: the rows to fetch, over all (b, h) units, are numbered 0..R-1 in unit order (an
// exclusive scan of the per-unit counts, which every CTA computes in shared memory), and CTA c
// fetches rows [c R / G, (c + 1) R / G).  Every CTA therefore moves the same number of bytes,
// whatever the spread of the per-head counts, without atomics or scratch memory.
#include <cuda_fp8.h>

#include "ig_common.cuh"
#include "pool_impl.h"

namespace ig {
namespace {

constexpr int kGatherThreads = 256;
// 4 rows x (K, V) in flight per lane at 64 registers (4 CTAs' worth per SM): a gather CTA then
// fits beside the compute stream's kernels, which leave it 16 K registers but not the 27 K it
// took at 8 rows and 106 registers.  Live, Llama-2-7B alpha = 2: 5.2-5.4 -> 4.93 ms per step (the
// fetch no longer waits for SMs to drain before it starts); OPT-30B unchanged at 195 GB/s.
#ifndef IG_G_UNROLL
#define IG_G_UNROLL 4
#endif
#ifndef IG_G_MIN_CTAS
#define IG_G_MIN_CTAS 4
#endif
constexpr int kUnroll = IG_G_UNROLL;  // rows x (K, V) in flight per lane
#ifndef IG_GQ_UNROLL
#define IG_GQ_UNROLL 4
#endif
#ifndef IG_GQ_MIN_CTAS
#define IG_GQ_MIN_CTAS 4
#endif
constexpr int kUnroll8 = IG_GQ_UNROLL;  // quantized records: one 16-byte load per lane and row, so more rows
constexpr int kMaxGatherUnits = 32768;  // (units + 1) ints of shared memory: 128 KB

__global__ void __launch_bounds__(kGatherThreads, IG_G_MIN_CTAS) k4_gather(
    const uint4* __restrict__ Kp, const uint4* __restrict__ Vp, int units, int cap, int vpr,
    int Lcap, const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
    uint4* __restrict__ Kg, uint4* __restrict__ Vg, int* err) {
  extern __shared__ int pre[];  // pre[u] = rows of units < u; pre[units] = R
  __shared__ int wsum[kGatherThreads / 32];
  // --- exclusive scan of the clamped counts, in chunks of `per` units per thread
  const int per = (units + kGatherThreads - 1) / kGatherThreads;
  const int u0 = threadIdx.x * per;
  int local = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) {
    int c = cnt[u];
    if (c < 0 || c > Lcap) {
      raise_error(err, IG_DEVERR_INDEX);
      c = c < 0 ? 0 : Lcap;
    }
    pre[u + 1] = c;  // temporarily the count
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
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  int run = base + incl - local;  // rows before this thread's chunk
  if (threadIdx.x == 0) pre[0] = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) {
    const int c = pre[u + 1];
    run += c;
    pre[u + 1] = run;
  }
  __syncthreads();
  const long long R = pre[units];
  const int r0 = (int)(R * blockIdx.x / gridDim.x);
  const int r1 = (int)(R * (blockIdx.x + 1) / gridDim.x);

  // --- fetch rows [r0, r1): row-group rg takes rows r0 + rg, r0 + rg + rpp, ...
  const int rpp = kGatherThreads / vpr;
  const int v = threadIdx.x % vpr, rg = threadIdx.x / vpr;
  int u = 0;  // unit of the row-group's current row; rows only grow, so u only advances
  {
    int lo = 0, hi = units;  // first unit whose end is past r0 (upper bound of r0 in pre)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid + 1] <= r0) lo = mid + 1; else hi = mid;
    }
    u = lo;
  }
  for (int r = r0 + rg; r < r1; r += rpp * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
    int unit[kUnroll], row[kUnroll], slot[kUnroll];
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      const int rr = r + q * rpp;
      slot[q] = -1;
      unit[q] = 0;
      row[q] = 0;
      if (rr < r1) {
        while (pre[u + 1] <= rr) ++u;
        unit[q] = u;
        row[q] = rr - pre[u];
        const int sl = idx[(size_t)u * Lcap + row[q]];
        if (sl < 0 || sl >= cap) {
          raise_error(err, IG_DEVERR_INDEX);
        } else {
          slot[q] = sl;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      if (slot[q] >= 0) {
        const size_t src = ((size_t)unit[q] * cap + slot[q]) * vpr + v;
        kv[q] = ld_nc_v4(Kp + src);
        vv[q] = ld_nc_v4(Vp + src);
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      if (slot[q] >= 0) {
        const size_t dst = ((size_t)unit[q] * Lcap + row[q]) * vpr + v;
        Kg[dst] = kv[q];
        Vg[dst] = vv[q];
      }
    }
  }
}

// Quantized pool (one record of codes per (token, head) in the pinned pool: K codes, then V
// codes; the two fp32 scales of the row in device memory): the same balanced row split; a row
// is one contiguous record of 2 d BITS / 8 bytes (whole 128-byte lines at d = 128), read by
// vpr = 2 d BITS / 128 lanes (16 bytes of codes each: the first half of the lanes the key, the
// rest the value) plus each lane's scale from the device-resident scale array, and
// dequantized to fp16 (code value x scale in fp32, rounded to nearest) into the usual staging
// layout.  BITS = 8: 16 e4m3 codes per lane; BITS = 4: 32 signed 4-bit codes per lane
// (element 2j in the low nibble of byte j).
template <int BITS>
__global__ void __launch_bounds__(kGatherThreads, IG_GQ_MIN_CTAS) k4_gather_q(
    const uint8_t* __restrict__ Rec, int rec, const float* __restrict__ Sc, int units, int cap, int vpr, int Lcap,
    const int32_t* __restrict__ idx,
    const int32_t* __restrict__ cnt, uint4* __restrict__ Kg, uint4* __restrict__ Vg, int* err) {
  extern __shared__ int pre[];
  __shared__ int wsum[kGatherThreads / 32];
  const int per = (units + kGatherThreads - 1) / kGatherThreads;
  const int u0 = threadIdx.x * per;
  int local = 0;
  for (int u = u0; u < min(units, u0 + per); ++u) {
    int c = cnt[u];
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
  const long long R = pre[units];
  const int r0 = (int)(R * blockIdx.x / gridDim.x);
  const int r1 = (int)(R * (blockIdx.x + 1) / gridDim.x);
  const int rpp = kGatherThreads / vpr;
  const int v = threadIdx.x % vpr, rg = threadIdx.x / vpr;
  int u = 0;
  {
    int lo = 0, hi = units;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid + 1] <= r0) lo = mid + 1; else hi = mid;
    }
    u = lo;
  }
  constexpr int OUT = BITS == 8 ? 2 : 4;  // 16-byte fp16 pieces a lane writes
  const int half = vpr / 2;            // lanes of the key codes
  const bool is_v = v >= half;
  const int cv = is_v ? v - half : v;   // 16-byte chunk of codes within K or V
  uint4* out = is_v ? Vg : Kg;
  for (int r = r0 + rg; r < r1; r += rpp * kUnroll8) {
    uint4 cd[kUnroll8];
    float sc[kUnroll8];
    int unit[kUnroll8], row[kUnroll8], slot[kUnroll8];
#pragma unroll
    for (int q = 0; q < kUnroll8; ++q) {
      const int rr = r + q * rpp;
      slot[q] = -1;
      unit[q] = 0;
      row[q] = 0;
      if (rr < r1) {
        while (pre[u + 1] <= rr) ++u;
        unit[q] = u;
        row[q] = rr - pre[u];
        const int sl = idx[(size_t)u * Lcap + row[q]];
        if (sl < 0 || sl >= cap) raise_error(err, IG_DEVERR_INDEX);
        else slot[q] = sl;
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll8; ++q) {
      if (slot[q] >= 0) {
        const size_t rw = (size_t)unit[q] * cap + slot[q];
        cd[q] = ld_nc_v4(Rec + rw * rec + (size_t)v * 16);
        sc[q] = __ldg(Sc + 2 * rw + (is_v ? 1 : 0));
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll8; ++q) {
      if (slot[q] < 0) continue;
      const size_t dst = ((size_t)unit[q] * Lcap + row[q]) * (OUT * half) + OUT * cv;
      const uint32_t w4[4] = {cd[q].x, cd[q].y, cd[q].z, cd[q].w};
      uint32_t o[4 * OUT];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (BITS == 8) {
          // two codes at a time: exact fp16 values of the codes, then x scale in fp32
          const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[i] & 0xffffu), __NV_E4M3);
          const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[i] >> 16), __NV_E4M3);
          const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
          const __half2 ra = __floats2half2_rn(a.x * sc[q], a.y * sc[q]);
          const __half2 rb = __floats2half2_rn(b.x * sc[q], b.y * sc[q]);
          o[2 * i] = *reinterpret_cast<const uint32_t*>(&ra);
          o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&rb);
        } else {
          // eight signed nibbles: shift each to the top and back, sign-extending
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c0 = (int)(w4[i] << (28 - 8 * j)) >> 28;
            const int c1 = (int)(w4[i] << (24 - 8 * j)) >> 28;
            const __half2 r = __floats2half2_rn((float)c0 * sc[q], (float)c1 * sc[q]);
            o[4 * i + j] = *reinterpret_cast<const uint32_t*>(&r);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < OUT; ++i) out[dst + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
  }
}

}  // namespace
}  // namespace ig

namespace ig {
ig_status check_pool_device(const ig_pool* pool);
}

using namespace ig;

extern "C" ig_status ig_gather_kv(void* stream, const ig_pool* pool, int layer, int B, int H,
                                  int d, int Lcap, const int32_t* idx, const int32_t* cnt,
                                  uint16_t* Kg, uint16_t* Vg, int max_ctas) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(pool->storage, "the pool was created without storage");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  IG_REQUIRE(Lcap > 0 && idx && cnt && Kg && Vg, "bad Lcap or null pointer");
  IG_REQUIRE((d * 2) % 16 == 0 && (d * 2) / 16 <= kGatherThreads, "d*2 must be a multiple of 16 bytes");
  IG_REQUIRE(aligned(Kg, 16) && aligned(Vg, 16), "Kg, Vg must be 16-byte aligned");
  const int vpr = d * 2 / 16;
  IG_REQUIRE(kGatherThreads % vpr == 0, "unsupported d %d", d);
  const int units = B * H;
  IG_REQUIRE(units <= kMaxGatherUnits, "B*H = %d exceeds %d", units, kMaxGatherUnits);
  IG_REQUIRE((long long)units * Lcap < (1ll << 31), "B*H*Lcap must stay below 2^31 rows");
  // a quantized fetch also dequantizes every row: by default it takes twice the CTAs of the
  // fp16 fetch (OPT-30B, int4 pool: 76 CTAs move 138 GB/s live against 116 for 38)
  int grid = max_ctas > 0 ? max_ctas : (pool->qbits ? 2 : 1) * fetch_grid(as_stream(stream));
  if (grid < 1) grid = 1;
  const size_t smem = (size_t)(units + 1) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k4_gather, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "gather smem attribute");
  }
  if (pool->qbits) {
    if (ig_status dst = check_pool_device(pool); dst != IG_OK) return dst;
    const int vprq = 2 * (d * pool->qbits / 8) / 16;  // lanes per record (16 bytes of codes each: K, then V)
    auto kern = pool->qbits == 8 ? k4_gather_q<8> : k4_gather_q<4>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "gather smem attribute");
    }
    const size_t rows = (size_t)B * H * pool->cap, r0 = (size_t)layer * rows;
    kern<<<grid, kGatherThreads, smem, as_stream(stream)>>>(
        pool->R + r0 * pool->rec, pool->rec, pool->S + r0 * 2, units, pool->cap, vprq, Lcap, idx, cnt,
        reinterpret_cast<uint4*>(Kg), reinterpret_cast<uint4*>(Vg), error_word());
    IG_CHECK_LAUNCH("quantized gather launch");
    return IG_OK;
  }
  const size_t layer_elems = (size_t)B * H * pool->cap * d;
  const uint4* Kp = reinterpret_cast<const uint4*>(pool->Kdev + (size_t)layer * layer_elems);
  const uint4* Vp = reinterpret_cast<const uint4*>(pool->Vdev + (size_t)layer * layer_elems);
  k4_gather<<<grid, kGatherThreads, smem, as_stream(stream)>>>(
      Kp, Vp, units, pool->cap, vpr, Lcap, idx, cnt, reinterpret_cast<uint4*>(Kg),
      reinterpret_cast<uint4*>(Vg), error_word());
  IG_CHECK_LAUNCH("gather launch");
  return IG_OK;
}
