// Host-link probes: how fast the GPU can read mapped, pinned host memory over its host link,
// as a plain stream and as a gather of fixed-size rows at random positions.  They measure the
// ceiling against which the fetch of the selected K/V rows is judged; they are not steps of
// the method.
#include "ig_common.cuh"

namespace ig {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 8;  // 16-byte loads in flight per thread

// Streams `n16` 16-byte words of src (grid-stride, kProbeUnroll loads issued before any is
// used).  The loads are volatile, and their XOR feeds a store that only a pattern no real
// buffer produces would trigger, so nothing is optimised away and nothing is written.
__global__ void __launch_bounds__(kProbeThreads) k_link_read(const uint4* __restrict__ src, size_t n16,
                                                             uint4* __restrict__ sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_nc_v4(src + i + (size_t)u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) {
      acc.x ^= v[u].x;
      acc.y ^= v[u].y;
      acc.z ^= v[u].z;
      acc.w ^= v[u].w;
    }
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_nc_v4(src + i);
    acc.x ^= v.x;
    acc.y ^= v.y;
    acc.z ^= v.z;
    acc.w ^= v.w;
  }
  if (acc.x == 0x9e3779b9u && acc.y == 0x7f4a7c15u && acc.z == 0xf39cc060u && acc.w == 0x5ced1e3bu)
    *sink = acc;
}

// Copies row idx[j] of src (rows of `lanes` 16-byte words) to row j of dst for j < n: `lanes`
// consecutive threads per row, kProbeUnroll rows in flight per thread group.  An index outside
// [0, rows) is reported and its row skipped.
__global__ void __launch_bounds__(kProbeThreads) k_link_gather(const uint4* __restrict__ src, size_t rows,
                                                               int lanes, const int32_t* __restrict__ idx,
                                                               size_t n, uint4* __restrict__ dst, int* err) {
  const int groups_per_cta = kProbeThreads / lanes;
  const int g = threadIdx.x / lanes, lane = threadIdx.x % lanes;
  if (g >= groups_per_cta) return;
  const size_t gstride = (size_t)gridDim.x * groups_per_cta;
  size_t j = (size_t)blockIdx.x * groups_per_cta + g;
  for (; j < n; j += kProbeUnroll * gstride) {
    uint4 v[kProbeUnroll];
    bool ok[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) {
      const size_t jj = j + (size_t)u * gstride;
      ok[u] = false;
      if (jj < n) {
        const int32_t r = __ldg(idx + jj);
        if (r >= 0 && (size_t)r < rows) {
          ok[u] = true;
          v[u] = ld_nc_v4(src + (size_t)r * lanes + lane);
        } else if (lane == 0) {
          raise_error(err, IG_DEVERR_INDEX);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u)
      if (ok[u]) dst[(j + (size_t)u * gstride) * lanes + lane] = v[u];
  }
}

int probe_grid(int ctas) { return ctas > 0 ? ctas : 4 * sm_count(); }

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" ig_status ig_link_read(void* stream, const void* src, size_t bytes, void* sink, int ctas) {
  IG_REQUIRE(src && sink, "null src or sink");
  IG_REQUIRE(bytes > 0 && bytes % 16 == 0, "bytes must be a positive multiple of 16");
  IG_REQUIRE(aligned(src, 16) && aligned(sink, 16), "src and sink must be 16-byte aligned");
  IG_REQUIRE(ctas >= 0 && ctas <= 65535, "ctas out of range");
  k_link_read<<<probe_grid(ctas), kProbeThreads, 0, as_stream(stream)>>>(
      static_cast<const uint4*>(src), bytes / 16, static_cast<uint4*>(sink));
  IG_CHECK_LAUNCH("link read probe launch");
  return IG_OK;
}

extern "C" ig_status ig_link_gather(void* stream, const void* src, size_t rows, int row_bytes,
                                    const int32_t* idx, size_t n, void* dst, int ctas) {
  IG_REQUIRE(src && idx && dst, "null pointer argument");
  IG_REQUIRE(row_bytes >= 16 && row_bytes <= 16 * kProbeThreads && row_bytes % 16 == 0 &&
                 kProbeThreads % (row_bytes / 16) == 0,
             "row_bytes must be 16 times a divisor of %d", kProbeThreads);
  IG_REQUIRE(rows > 0 && rows <= 0x7fffffffu, "rows must be in [1, 2^31)");
  IG_REQUIRE(aligned(src, 16) && aligned(dst, 16), "src and dst must be 16-byte aligned");
  IG_REQUIRE(ctas >= 0 && ctas <= 65535, "ctas out of range");
  if (n == 0) return IG_OK;
  k_link_gather<<<probe_grid(ctas), kProbeThreads, 0, as_stream(stream)>>>(
      static_cast<const uint4*>(src), rows, row_bytes / 16, idx, n, static_cast<uint4*>(dst), error_word());
  IG_CHECK_LAUNCH("link gather probe launch");
  return IG_OK;
}
