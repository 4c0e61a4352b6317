// Gather of the chosen full key/value rows from the pinned host pool into HBM
// (InfiniGen paper-graph summary, section 3.4, "Decoding Stage", Step 5).
//
// The pool is mapped pinned host memory, readable by the GPU over the host link, so the
// fetch is a kernel of zero-copy 16-byte loads rather than one copy call per row: for d = 128
// a row is 256 B and 16 lanes fetch it together; each lane keeps 2 x kUnroll loads in flight
// (keys and values).  The grid is kept small (a fraction of the SMs): the host link saturates
// with a few dozen CTAs, and the rest of the GPU stays free for the compute stream.
#include "ig_common.cuh"
#include "pool_impl.h"

namespace ig {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kGatherThreads) k4_gather(
    const uint4* __restrict__ Kp, const uint4* __restrict__ Vp, int units, int cap, int vpr,
    int Lcap, const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
    uint4* __restrict__ Kg, uint4* __restrict__ Vg, int* err) {
  const int rpp = kGatherThreads / vpr;  // rows fetched in parallel per CTA
  const int v = threadIdx.x % vpr, rg = threadIdx.x / vpr;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    int c = cnt[u];
    if (c < 0 || c > Lcap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      c = c < 0 ? 0 : Lcap;
    }
    const int32_t* ii = idx + (size_t)u * Lcap;
    const uint4* ksrc = Kp + (size_t)u * cap * vpr;
    const uint4* vsrc = Vp + (size_t)u * cap * vpr;
    uint4* kdst = Kg + (size_t)u * Lcap * vpr;
    uint4* vdst = Vg + (size_t)u * Lcap * vpr;
    for (int j = rg; j < c; j += rpp * kUnroll) {
      uint4 kv[kUnroll], vv[kUnroll];
      int slot[kUnroll];
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int jj = j + q * rpp;
        slot[q] = (jj < c) ? ii[jj] : -1;
        if (jj < c && (slot[q] < 0 || slot[q] >= cap)) {
          raise_error(err, IG_DEVERR_INDEX);
          slot[q] = -1;
        }
      }
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        if (slot[q] >= 0) {
          kv[q] = ld_nc_v4(ksrc + (size_t)slot[q] * vpr + v);
          vv[q] = ld_nc_v4(vsrc + (size_t)slot[q] * vpr + v);
        }
      }
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int jj = j + q * rpp;
        if (slot[q] >= 0) {
          kdst[(size_t)jj * vpr + v] = kv[q];
          vdst[(size_t)jj * vpr + v] = vv[q];
        }
      }
    }
  }
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" ig_status ig_gather_kv(void* stream, const ig_pool* pool, int layer, int B, int H,
                                  int d, int Lcap, const int32_t* idx, const int32_t* cnt,
                                  uint16_t* Kg, uint16_t* Vg, int max_ctas) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  IG_REQUIRE(Lcap > 0 && idx && cnt && Kg && Vg, "bad Lcap or null pointer");
  IG_REQUIRE((d * 2) % 16 == 0 && (d * 2) / 16 <= kGatherThreads, "d*2 must be a multiple of 16 bytes");
  IG_REQUIRE(aligned(Kg, 16) && aligned(Vg, 16), "Kg, Vg must be 16-byte aligned");
  const int vpr = d * 2 / 16;
  IG_REQUIRE(kGatherThreads % vpr == 0, "unsupported d %d", d);
  const int units = B * H;
  int grid = max_ctas > 0 ? max_ctas : sm_count() / 2;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  const size_t layer_elems = (size_t)B * H * pool->cap * d;
  const uint4* Kp = reinterpret_cast<const uint4*>(pool->Kdev + (size_t)layer * layer_elems);
  const uint4* Vp = reinterpret_cast<const uint4*>(pool->Vdev + (size_t)layer * layer_elems);
  k4_gather<<<grid, kGatherThreads, 0, as_stream(stream)>>>(
      Kp, Vp, units, pool->cap, vpr, Lcap, idx, cnt, reinterpret_cast<uint4*>(Kg),
      reinterpret_cast<uint4*>(Vg), error_word());
  IG_CHECK_LAUNCH("gather launch");
  return IG_OK;
}
