// Prefill stage on the GPU (InfiniGen paper-graph summary, section 3.4, "Prefill Stage:
// Partial Weight Index Generation", Steps 1-3; RoPE models rotate each key before the skew, so
// for them K = X W_K is followed by a kernel computing K~_h = RoPE_t(K_h) A_h):
//   Step 1  K~ = X W~_K and V = X W_V for every prompt token (a tcgen05 GEMM), the rows of the
//           tokens the pool keeps written to the pinned pool, token t at slot t mod cap;
//   Step 2  column score = column sums of |W~_Q| plus column sums of |K~| over every prompt
//           token, top-k per head;
//   Step 3  the partial query weight (the chosen rows of W~_Q^T) and the partial key cache.
//
// The GEMM C[M][N] = A[M][K] . Bt[N][K]^T (both K-major, fp16 in, fp32 accumulate, fp16 out):
// a persistent kernel, one CTA per SM, each taking 128 x 256 output tiles in turn.  One thread
// issues the TMA loads into a ring of 4 stages of 64-wide K (48 KB each), another the tcgen05
// MMAs (128x256x16) into one of two 256-column accumulators in tensor memory, each stage
// released by a tcgen05.commit onto its "empty" mbarrier and each finished accumulator
// announced on its "full" one; four epilogue warps read it with tcgen05.ld (warp w owns TMEM
// lanes 32 (w % 4) .. + 31 = rows), hand it back, store fp16 rows, and, when asked, reduce |C|
// down each column of the tile (a shuffle transpose-reduce in each warp, then the four row
// quarters in a fixed order) into per-tile partial sums, so the column score is deterministic.
// The MMAs of the next tile run while the epilogue drains the last one.
#include <cuda.h>

#include <mutex>

#include "ig_common.cuh"
#include "pool_impl.h"
#include "tc_common.cuh"

namespace ig {
namespace {

constexpr int kGM = 128;        // tile rows (tcgen05 M = TMEM lanes)
constexpr int kGN = 256;        // tile columns (tcgen05 N = TMEM columns of one accumulator)
constexpr int kGK = 64;         // K per stage: one 128-byte swizzle atom of fp16
constexpr int kGStages = 4;
constexpr int kGThreads = 192;  // warp 0: TMA loads, warp 1: MMAs, warps 2-5: epilogue
constexpr uint32_t kGStageA = kGM * kGK * 2;  // 16 KB
constexpr uint32_t kGStageB = kGN * kGK * 2;  // 32 KB
constexpr uint32_t kGTmemCols = 2 * kGN;      // two accumulators: one fills while one drains
constexpr int kGGroup = 16;     // row tiles per group of the tile order
// kind::f16, D fp32, A/B fp16 K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28
constexpr uint32_t kGIdesc = (1u << 4) | ((uint32_t)(kGN >> 3) << 17) | ((uint32_t)(kGM >> 4) << 24);

constexpr int kGStageRow = 64 + 8;  // halves per row of an epilogue warp's staging (+8: banks)

// barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain; then the tensor-memory slot,
// flags, the column sums [4][kGN] and the epilogue warps' staging [4][32][kGStageRow] fp16
size_t gemm_smem_bytes() {
  return 1024 + kGStages * (kGStageA + kGStageB) + (2 * kGStages + 5) * 8 + 32 + 4 * kGN * sizeof(float) + 16 +
         4 * 32 * kGStageRow * 2;
}

// Rows of the output that also go to a pinned pool, as the pool keeps them: output row
// b * N + t (t >= N - cap) to slot t mod cap of [B][H][cap][d], column h * d + j to (h, j).
struct PoolOut {
  uint16_t* base;  // NULL: no pool output
  int N, H, d, cap;
};

// Tile t of the grouped order: runs of kGGroup row tiles take each column tile in turn, so a B
// tile is reused by the CTAs working on neighbouring t and the group's A tiles stay in L2.
__device__ __forceinline__ void gemm_tile(int t, int tiles_m, int tiles_n, int& mt, int& ntile) {
  const int per_group = kGGroup * tiles_n;
  const int gi = t / per_group, within = t % per_group;
  const int first_m = gi * kGGroup;
  const int gsize = min(tiles_m - first_m, kGGroup);
  mt = first_m + within % gsize;
  ntile = within / gsize;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Persistent: CTA b takes tiles b, b + G, b + 2G, ... of the grouped order.  The load ring
// and the MMAs run on across tiles, and the accumulator alternates between two 256-column
// halves of tensor memory, so the epilogue of one tile overlaps the MMAs of the next.
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_tn(const __grid_constant__ CUtensorMap map_a,
                                                           const __grid_constant__ CUtensorMap map_b,
                                                           __half* __restrict__ C, int M, int N, int K,
                                                           float* __restrict__ colpart, const PoolOut po, int* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sA = smem;
  unsigned char* sB = smem + kGStages * kGStageA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kGStages * kGStageB);
  uint64_t* empty = full + kGStages;
  uint64_t* acc_full = empty + kGStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* epi_ok = reinterpret_cast<int*>(tmem_slot + 2);   // [2]: the epilogue warps' joint verdict
  float* csum = reinterpret_cast<float*>(tmem_slot + 4);  // [4][kGN] (scalar accesses only)
  // [4][32][kGStageRow], on a 16-byte boundary (rows of 144 bytes keep every piece aligned)
  __half* stage_all = reinterpret_cast<__half*>((reinterpret_cast<uintptr_t>(csum + 4 * kGN) + 15) &
                                                ~static_cast<uintptr_t>(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = (N + kGN - 1) / kGN, tiles_m = (M + kGM - 1) / kGM;
  const int T = tiles_m * tiles_n;
  const int nk = (K + kGK - 1) / kGK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kGTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // producer: stage it % S of round it / S is free once the MMAs of the previous round on it
      // have completed (their commit arrives on empty[stage])
      uint32_t it = 0;
      for (int t = blockIdx.x; t < T && !*abort_flag; t += gridDim.x) {
        int mt, ntile;
        gemm_tile(t, tiles_m, tiles_n, mt, ntile);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t st = it % kGStages, r = it / kGStages;
          if (r > 0 && !mbar_wait_bounded(&empty[st], (r - 1) & 1)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[st], kGStageA + kGStageB);
          tma_load_2d(sA + st * kGStageA, &map_a, kb * kGK, mt * kGM, &full[st]);
          tma_load_2d(sB + st * kGStageB, &map_b, kb * kGK, ntile * kGN, &full[st]);
        }
      }
      if (*abort_flag) {
        // let the loads already issued land before the shared memory is released
        for (uint32_t st = 0; st < kGStages && st < it; ++st)
          mbar_wait_bounded(&full[st], ((it - 1 - st) / kGStages) & 1, 1u << 16);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, j = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok && !*abort_flag; t += gridDim.x, ++j) {
        const uint32_t buf = j & 1, u = j >> 1;
        // the epilogue has drained this accumulator's previous tile
        if (u > 0 && !mbar_wait_bounded(&acc_empty[buf], (u - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc_tm = tmem + buf * kGN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t st = it % kGStages, r = it / kGStages;
          if (!mbar_wait_bounded(&full[st], r & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(sA + st * kGStageA), b0 = smem_addr(sB + st * kGStageB);
#pragma unroll
          for (int kk = 0; kk < kGK / 16; ++kk) {
            const uint64_t ad = sw128_desc(a0 + kk * 32), bd = sw128_desc(b0 + kk * 32);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(acc_tm),
                "l"(ad), "l"(bd), "r"(kGIdesc), "r"(acc));
          }
          mma_commit(&empty[st]);
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      if (!ok || *abort_flag) {
        *abort_flag = 1;
        // the MMAs already issued finish before tensor memory is released
        mma_commit(drain);
        mbar_wait_bounded(drain, 0, 1u << 16);
      }
    }
  } else {
    // epilogue, warps 2-5: warp w reads TMEM lanes 32 (w % 4) .. + 31 = rows of that quarter
    const int q = warp & 3, et = threadIdx.x - 64;
    uint32_t j = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++j) {
      const uint32_t buf = j & 1, u = j >> 1;
      const bool mine = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], u & 1) ? 1 : 0) != 0;
      // one verdict for the four warps (the TMEM loads are warp-collective and the warps meet
      // at named barriers below): all four saw the tile, and nothing aborted
      // (the abort flag is read before the barrier, so no warp can see a later value than another)
      if (lane == 0) epi_ok[(j & 1)] = 1;
      epi_sync();
      if (lane == 0 && (!mine || *abort_flag)) epi_ok[(j & 1)] = 0;
      epi_sync();
      const bool go = epi_ok[(j & 1)] != 0;
      if (!go) {
        if (et == 0) {
          *abort_flag = 1;
          raise_error(err, IG_DEVERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      int mt, ntile;
      gemm_tile(t, tiles_m, tiles_n, mt, ntile);
      const int m0 = mt * kGM, n0 = ntile * kGN;
      const int row = m0 + q * 32 + lane;
      __half* stage = stage_all + (size_t)q * 32 * kGStageRow;
      const int first = po.N > po.cap ? po.N - po.cap : 0;
      for (int ch = 0; ch < kGN / 32; ++ch) {
        const int c0 = n0 + ch * 32;
        uint32_t r[32];
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + buf * kGN + (uint32_t)(ch * 32);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (c0 >= N) continue;  // warp-uniform: N is a multiple of 32
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
          h[i] = *reinterpret_cast<const uint32_t*>(&p);
        }
        if (C && row < M) {
          uint4* dst = reinterpret_cast<uint4*>(C + (size_t)row * N + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        }
        if (po.base) {
          // 64 columns at a time through shared memory, so that the pool rows (far apart in
          // host memory) go out as whole 128-byte pieces, eight lanes to a row
          uint4* srow = reinterpret_cast<uint4*>(stage + (size_t)lane * kGStageRow + (ch & 1) * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) srow[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          if ((ch & 1) || ch == kGN / 32 - 1 || c0 + 32 >= N) {
            __syncwarp();
            const int cb = c0 - (ch & 1) * 32;           // first column of the staged block
            const int ncols = min(64, N - cb);           // 32 or 64 (N is a multiple of 32)
            const int part = lane & 7;                   // 16-byte piece of a row
            const int col = cb + part * 8;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int rl = it * 4 + (lane >> 3);
              const int grow = m0 + q * 32 + rl;
              if (grow < M && part * 8 < ncols) {
                const int t = grow % po.N, b = grow / po.N;
                if (t >= first) {
                  const int hh = col / po.d, j = col % po.d;
                  uint4* dst = reinterpret_cast<uint4*>(
                      po.base + ((((size_t)b * po.H + hh) * po.cap + t % po.cap) * po.d + j));
                  *dst = *reinterpret_cast<const uint4*>(stage + (size_t)rl * kGStageRow + part * 8);
                }
              }
            }
            __syncwarp();
          }
        }
        if (colpart) {
          // |C| of the stored fp16 values (rows past M are zero: the A tile is zero-filled
          // there); transpose-reduce: after the steps 16, 8, 4, 2, 1 lane j holds column j's sum
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = row < M ? fabsf(__half2float(__float2half_rn(v[i]))) : 0.f;
#pragma unroll
          for (int s2 = 16; s2 >= 1; s2 >>= 1) {
            const bool up = (lane & s2) != 0;
#pragma unroll
            for (int i = 0; i < s2; ++i) {
              const float send = up ? v[i] : v[i + s2];
              const float keep = up ? v[i + s2] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s2);
            }
          }
          csum[q * kGN + ch * 32 + lane] = v[0];
        }
      }
      // this warp's reads of the accumulator are done: the MMAs may refill it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      if (colpart) {
        epi_sync();
        for (int c = et; c < kGN; c += 128) {
          if (n0 + c >= N) continue;
          colpart[(size_t)mt * N + n0 + c] = ((csum[c] + csum[kGN + c]) + csum[2 * kGN + c]) + csum[3 * kGN + c];
        }
        epi_sync();  // csum is refilled by the next tile
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kGTmemCols));
  }
}

// Step 2: one CTA (d threads) per head: score[c] = sum_r |Wq_t[h d + c][r]| (float64) + the
// key column partials summed over the row tiles in order; the k best (ties to the lower
// column) written ascending.
__global__ void k_choose_cols(const __half* __restrict__ Wq_t, int D, int H, int d, int k,
                              const float* __restrict__ colpart, int mtiles, int32_t* __restrict__ cols,
                              double* __restrict__ score_out) {
  extern __shared__ double sc[];  // [d]
  const int h = blockIdx.x, c = threadIdx.x;
  const int n = h * d + c;
  // the weight row sum: one warp per row would be faster; this runs once per prompt
  const __half* w = Wq_t + (size_t)n * D;
  double a = 0.0;
  for (int r = 0; r < D; ++r) a += fabs((double)__half2float(w[r]));
  double kc = 0.0;
  for (int t = 0; t < mtiles; ++t) kc += (double)colpart[(size_t)t * H * d + n];
  sc[c] = a + kc;
  if (score_out) score_out[n] = a + kc;
  __syncthreads();
  int rank = 0;
  for (int o = 0; o < d; ++o) rank += (sc[o] > sc[c] || (sc[o] == sc[c] && o < c)) ? 1 : 0;
  const bool keep = rank < k;
  __syncthreads();
  // ascending compaction of the kept columns
  int* flag = reinterpret_cast<int*>(sc);
  flag[c] = keep ? 1 : 0;
  __syncthreads();
  if (keep) {
    int pos = 0;
    for (int o = 0; o < c; ++o) pos += flag[o];
    cols[h * k + pos] = c;
  }
}

// Step 3a: the partial query weight, rows h k + j = Wq_t[h d + cols[h][j]] (16-byte copies).
__global__ void k_extract_rows(const uint4* __restrict__ Wq_t, int D, int d, int k, const int32_t* __restrict__ cols,
                               uint4* __restrict__ out, int* err) {
  const int hk = blockIdx.x, h = hk / k;
  const int c = cols[hk];
  if (c < 0 || c >= d) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    return;
  }
  const int v16 = D / 8;
  const uint4* src = Wq_t + (size_t)(h * d + c) * v16;
  for (int i = threadIdx.x; i < v16; i += blockDim.x) out[(size_t)hk * v16 + i] = src[i];
}

// Step 1 (store): rows of the tokens the pool keeps (t >= N - cap) to slot t mod cap of the
// pinned pool, 16-byte zero-copy stores; src [B][N][H][d], one warp per (b, t, h) row.  It needs
// no shared memory, so it runs beside the projection GEMM (on a side stream).
__global__ void __launch_bounds__(256) k_pool_rows(const uint4* __restrict__ src, int B, int N, int H, int d, int cap,
                                                  uint4* __restrict__ pool) {
  const int vpr = d / 8;
  const int first = N > cap ? N - cap : 0;
  const long long keep = (long long)B * (N - first) * H;
  const long long w0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  const int lane = threadIdx.x & 31;
  for (long long r = w0; r < keep; r += nw) {
    const int h = (int)(r % H);
    const long long bt = r / H;
    const int t = first + (int)(bt % (N - first));
    const int b = (int)(bt / (N - first));
    const uint4* s = src + (((size_t)b * N + t) * H + h) * vpr;
    uint4* dst = pool + (((size_t)b * H + h) * cap + t % cap) * vpr;
    for (int v = lane; v < vpr; v += 32) dst[v] = s[v];
  }
}

// Step 3b: for (b, h) and a tile of 64 prompt tokens, the chosen columns of the keys the pool
// keeps go to the partial key cache at their slots (rows staged in shared memory, coalesced
// writes along the token axis).
constexpr int kScTok = 64;
__global__ void k_partial_keys(const __half* __restrict__ Kt, int N, int H, int d, int k, int cap, int Lcap,
                               const int32_t* __restrict__ cols, __half* __restrict__ Kpart, int* err) {
  extern __shared__ __align__(16) unsigned char sraw[];
  __half* sk = reinterpret_cast<__half*>(sraw);  // [kScTok][d]
  const int t0 = blockIdx.x * kScTok, h = blockIdx.y, b = blockIdx.z;
  const int first = N > cap ? N - cap : 0;
  const int vpr = d / 8;
  const size_t bh = (size_t)b * H + h;
  for (int i = threadIdx.x; i < kScTok * vpr; i += blockDim.x) {
    const int tt = i / vpr, v = i % vpr, t = t0 + tt;
    if (t >= N || t < first) continue;
    const size_t src = ((size_t)b * N + t) * H * d + (size_t)h * d;  // halves
    reinterpret_cast<uint4*>(sk)[tt * vpr + v] = *reinterpret_cast<const uint4*>(Kt + src + v * 8);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k * kScTok; i += blockDim.x) {
    const int c = i / kScTok, tt = i % kScTok, t = t0 + tt;
    if (t >= N || t < first) continue;
    const int col = cols[h * k + c];
    if (col < 0 || col >= d) {
      raise_error(err, IG_DEVERR_INDEX);
      continue;
    }
    Kpart[(bh * k + c) * Lcap + t % cap] = sk[tt * d + col];
  }
}

// RoPE: cos and sin of t * theta^(-2j/d) for t < N, j < d/2 (angles in float64).
__global__ void k_rope_table(int N, int half, int d, double theta, float* __restrict__ cs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N * half) return;
  const int t = i / half, j = i % half;
  double sn, c;
  sincos((double)t * pow(theta, -2.0 * (double)j / (double)d), &sn, &c);
  cs[2 * (size_t)i] = (float)c;
  cs[2 * (size_t)i + 1] = (float)sn;
}

// K~ rows of a RoPE model, in place: row m (token t = m mod N) of head h becomes
// RoPE_t(K_h) A_h, rounded to fp16.  One CTA per (64 rows, head): A_h and the rotated rows in
// shared memory (fp32), thread (j, r0) computes column j of rows r0, r0 + 2, ...; the column
// sums of |K~| of the tile go to colpart[tile][h d + j] (two row halves added in order).
constexpr int kRsRows = 64;
template <int D>
__global__ void __launch_bounds__(256) k_rope_skew(__half* __restrict__ K, int M, int N, int H,
                                                  const float* __restrict__ A, const float* __restrict__ cs,
                                                  float* __restrict__ colpart) {
  extern __shared__ float smf[];
  float* sA = smf;                 // [D][D]
  float* sR = smf + D * D;         // [kRsRows][D]
  float* sC = sR + kRsRows * D;    // [2][D]
  const int h = blockIdx.y, m0 = blockIdx.x * kRsRows;
  const int Hd = H * D, half = D / 2;
  for (int i = threadIdx.x; i < D * D; i += 256) sA[i] = A[(size_t)h * D * D + i];
  for (int i = threadIdx.x; i < kRsRows * half; i += 256) {
    const int r = i / half, j = i % half, m = m0 + r;
    float lo = 0.f, hi = 0.f, c = 1.f, sn = 0.f;
    if (m < M) {
      const int t = m % N;
      lo = __half2float(K[(size_t)m * Hd + h * D + j]);
      hi = __half2float(K[(size_t)m * Hd + h * D + j + half]);
      c = cs[2 * ((size_t)t * half + j)];
      sn = cs[2 * ((size_t)t * half + j) + 1];
    }
    sR[r * D + j] = lo * c - hi * sn;
    sR[r * D + j + half] = lo * sn + hi * c;
  }
  __syncthreads();
  constexpr int TPC = 256 / D;  // threads per column (2 for D = 128, 4 for D = 64)
  const int j = threadIdx.x % D, r0 = threadIdx.x / D;
  float csum = 0.f;
  for (int r = r0; r < kRsRows; r += TPC) {
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc = fmaf(sR[r * D + i], sA[i * D + j], acc);
    const int m = m0 + r;
    const __half o = __float2half_rn(acc);
    if (m < M) {
      K[(size_t)m * Hd + h * D + j] = o;
      csum += fabsf(__half2float(o));
    }
  }
  if (TPC == 2) {
    sC[r0 * D + j] = csum;
    __syncthreads();
    if (r0 == 0) colpart[(size_t)blockIdx.x * Hd + h * D + j] = sC[j] + sC[D + j];
  } else {
    __shared__ float sc4[4][D];
    sc4[r0][j] = csum;
    __syncthreads();
    if (r0 == 0) colpart[(size_t)blockIdx.x * Hd + h * D + j] = ((sc4[0][j] + sc4[1][j]) + sc4[2][j]) + sc4[3][j];
  }
}

// A_cols[h][i][j] = A[h][i][cols[h][j]] (the decode stage's partial skew for RoPE models).
__global__ void k_extract_acols(const float* __restrict__ A, int d, int k, const int32_t* __restrict__ cols,
                                float* __restrict__ out, int* err) {
  const int h = blockIdx.x;
  for (int e = threadIdx.x; e < d * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    const int c = cols[h * k + j];
    if (c < 0 || c >= d) {
      raise_error(err, IG_DEVERR_INDEX);
      continue;
    }
    out[((size_t)h * d + i) * k + j] = A[((size_t)h * d + i) * d + c];
  }
}

}  // namespace
}  // namespace ig

using namespace ig;

namespace {

size_t rup(size_t x) { return round_up(x, 256); }

constexpr int kPrefillFreeSms = 16;  // SMs the V projection leaves to the column choice and partial keys

// The side stream and events that let the pool writes run beside the projections (one set per
// device, created on first use; creation and the enqueue sequence of a call are serialised by
// g_side_mu, which callers of side_stream hold).  The side stream belongs to the device's
// primary context, so it runs on the whole device whatever SM partition the caller's stream has.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};
std::mutex g_side_mu;
SideStream g_side[64];

ig_status side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "current device");
  if (dev < 0 || dev >= 64) return fail(IG_ERR_INVALID, "device %d out of range", dev);
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    int lo = 0, hi = 0;
    e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, hi);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ss.ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "prefill side stream");
  }
  *out = &ss;
  return IG_OK;
}

// Writes the kept rows of src to the pool on the side stream once `st`'s work so far is done.
ig_status fork_pool_rows(cudaStream_t st, SideStream* ss, int which, const uint16_t* src, int B, int N, int H,
                         int d, int cap, uint16_t* pool) {
  cudaError_t e = cudaEventRecord(ss->ev[which], st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->ev[which], 0);
  if (e != cudaSuccess) return cuda_fail(e, "prefill fork");
  k_pool_rows<<<2 * sm_count(), 256, 0, ss->s>>>(reinterpret_cast<const uint4*>(src), B, N, H, d, cap,
                                                 reinterpret_cast<uint4*>(pool));
  IG_CHECK_LAUNCH("pool rows launch");
  return IG_OK;
}

// `st` continues after everything the side stream was given.
ig_status join_side(cudaStream_t st, SideStream* ss) {
  cudaError_t e = cudaEventRecord(ss->ev[2], ss->s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->ev[2], 0);
  return e == cudaSuccess ? IG_OK : cuda_fail(e, "prefill join");
}

// workspace: K~ [B N][H d] fp16, column partials [ceil(B N / 64)][H d] fp32 (128-row tiles
// use the first half), the RoPE cos/sin table [N][d/2][2] fp32 (V needs none: its rows go from
// the GEMM's epilogue to the pool)
void prefill_layout(int B, int N, int H, int d, size_t* off_cp, size_t* off_tab, size_t* total) {
  const size_t M = (size_t)B * N, Nn = (size_t)H * d;
  const size_t mt = (M + kRsRows - 1) / kRsRows;
  *off_cp = rup(M * Nn * 2);
  *off_tab = *off_cp + rup(mt * Nn * sizeof(float));
  *total = *off_tab + rup((size_t)N * d * sizeof(float));
}

// max_ctas: at most this many persistent CTAs (0: one per SM), so that kernels on another
// stream find SMs free
ig_status gemm(cudaStream_t st, const uint16_t* A, const uint16_t* Bt, uint16_t* C, int M, int N, int K,
               float* colpart, PoolOut po = PoolOut{nullptr, 1, 1, 1, 1}, int max_ctas = 0) {
  CUtensorMap ma, mb;
  ig_status r = make_map(&ma, A, M, K, kGM);
  if (r != IG_OK) return r;
  r = make_map(&mb, Bt, N, K, kGN);
  if (r != IG_OK) return r;
  const size_t smem = gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "prefill GEMM smem attribute");
  const long long tiles = (long long)((N + kGN - 1) / kGN) * ((M + kGM - 1) / kGM);
  IG_REQUIRE(tiles < (1ll << 31), "GEMM too large for one launch");
  // persistent: one CTA per SM (its 197 KB of shared memory admit no second one)
  const int slots = max_ctas > 0 && max_ctas < sm_count(st) ? max_ctas : sm_count(st);
  const int grid = (int)(tiles < slots ? tiles : slots);
  k_gemm_tn<<<grid, kGThreads, smem, st>>>(ma, mb, reinterpret_cast<__half*>(C), M, N, K, colpart, po,
                                           error_word());
  IG_CHECK_LAUNCH("prefill GEMM launch");
  return IG_OK;
}

}  // namespace

extern "C" ig_status ig_gemm_tn(void* stream, int M, int N, int K, const uint16_t* A, const uint16_t* Bt,
                                uint16_t* C, float* colpart) {
  IG_REQUIRE(M > 0 && N > 0 && K > 0, "M, N, K must be positive");
  IG_REQUIRE(N % 32 == 0 && K % 8 == 0, "N must be a multiple of 32 and K of 8");
  IG_REQUIRE((long long)(M + kGM - 1) / kGM <= 65535, "M too large for one launch");
  IG_REQUIRE(A && Bt && C, "null pointer argument");
  IG_REQUIRE(aligned(A, 16) && aligned(Bt, 16) && aligned(C, 16), "A, Bt, C must be 16-byte aligned");
  return gemm(as_stream(stream), A, Bt, C, M, N, K, colpart);
}

extern "C" size_t ig_prefill_workspace_bytes(int B, int N, int H, int d) {
  if (B <= 0 || N <= 0 || H <= 0 || d <= 0) return 0;
  size_t oc, ot, tot;
  prefill_layout(B, N, H, d, &oc, &ot, &tot);
  return tot;
}

extern "C" ig_status ig_prefill_layer(void* stream, ig_pool* pool, int layer, int B, int N, int D, int H, int d,
                                      int k, int Lcap, const uint16_t* X, const uint16_t* Wq_t, const uint16_t* Wk_t,
                                      const uint16_t* Wv_t, int32_t* cols, uint16_t* Wq_part_t, uint16_t* Kpart,
                                      void* workspace, size_t workspace_bytes) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(pool->storage && !pool->qbits, "the prefill writes an fp16 pool with storage");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  IG_REQUIRE(N > 0 && D > 0 && D % 8 == 0, "N > 0 and D a positive multiple of 8");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128");
  IG_REQUIRE(k > 0 && k <= d, "0 < k <= d");
  IG_REQUIRE(Lcap >= pool->cap && Lcap % 8 == 0, "Lcap must cover the pool and be a multiple of 8");
  IG_REQUIRE(X && Wq_t && Wk_t && Wv_t && cols && Wq_part_t && Kpart, "null pointer argument");
  IG_REQUIRE(aligned(X, 16) && aligned(Wq_t, 16) && aligned(Wk_t, 16) && aligned(Wv_t, 16) &&
                 aligned(Wq_part_t, 16),
             "X and the weights must be 16-byte aligned");
  size_t oc, ot, tot;
  prefill_layout(B, N, H, d, &oc, &ot, &tot);
  if (!workspace || workspace_bytes < tot)
    return fail(IG_ERR_CAPACITY, "the prefill needs %zu workspace bytes", tot);
  IG_REQUIRE(aligned(workspace, 256), "workspace must be 256-byte aligned");
  cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  uint16_t* Kt = reinterpret_cast<uint16_t*>(ws);
  float* colpart = reinterpret_cast<float*>(ws + oc);
  const int M = B * N, Nn = H * d;
  const int mtiles = (M + kGM - 1) / kGM;
  IG_REQUIRE(mtiles <= 65535, "B*N too large for one launch");
  const size_t le = (size_t)B * H * pool->cap * d;
  // the lock covers the side stream's creation on first use as well as the enqueue sequence
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* ss = nullptr;
  ig_status r = side_stream(&ss);
  if (r != IG_OK) return r;
  // Step 1: K~ (with the per-tile column partials of |K~|) and V; the GEMMs' epilogues write the
  // rows the pool keeps straight to it (V goes nowhere else).  V is projected on the side stream
  // with kPrefillFreeSms SMs left free, where steps 2-3 (which need only K~) run meanwhile.
  r = gemm(st, X, Wk_t, Kt, M, Nn, D, colpart, PoolOut{pool->Kdev + (size_t)layer * le, N, H, d, pool->cap});
  if (r != IG_OK) return r;
  cudaError_t fe = cudaEventRecord(ss->ev[0], st);
  if (fe == cudaSuccess) fe = cudaStreamWaitEvent(ss->s, ss->ev[0], 0);
  if (fe != cudaSuccess) return cuda_fail(fe, "prefill fork");
  // the side stream spans the whole device, so its grid is sized by the device's SM count
  r = gemm(ss->s, X, Wv_t, nullptr, M, Nn, D, nullptr, PoolOut{pool->Vdev + (size_t)layer * le, N, H, d, pool->cap},
           sm_count() - kPrefillFreeSms);
  if (r != IG_OK) return r;
  // Step 2: the columns
  k_choose_cols<<<H, d, d * sizeof(double), st>>>(reinterpret_cast<const __half*>(Wq_t), D, H, d, k, colpart, mtiles,
                                                  cols, nullptr);
  IG_CHECK_LAUNCH("column choice launch");
  // Step 3: the partial weight and the partial key cache
  k_extract_rows<<<H * k, 128, 0, st>>>(reinterpret_cast<const uint4*>(Wq_t), D, d, k, cols,
                                        reinterpret_cast<uint4*>(Wq_part_t), error_word());
  IG_CHECK_LAUNCH("partial weight launch");
  dim3 sg((N + kScTok - 1) / kScTok, H, B);
  k_partial_keys<<<sg, 256, kScTok * d * 2, st>>>(reinterpret_cast<const __half*>(Kt), N, H, d, k, pool->cap, Lcap,
                                                 cols, reinterpret_cast<__half*>(Kpart), error_word());
  IG_CHECK_LAUNCH("partial keys launch");
  return join_side(st, ss);
}

extern "C" ig_status ig_prefill_layer_rope(void* stream, ig_pool* pool, int layer, int B, int N, int D, int H,
                                           int d, int k, int Lcap, float rope_theta, const uint16_t* X,
                                           const uint16_t* Wq_t, const uint16_t* Wk_t, const uint16_t* Wv_t,
                                           const float* A, int32_t* cols, float* A_cols, uint16_t* Kpart,
                                           void* workspace, size_t workspace_bytes) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(pool->storage && !pool->qbits, "the prefill writes an fp16 pool with storage");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  IG_REQUIRE(N > 0 && D > 0 && D % 8 == 0, "N > 0 and D a positive multiple of 8");
  IG_REQUIRE(d == 64 || d == 128, "d must be 64 or 128");
  IG_REQUIRE(k > 0 && k <= d, "0 < k <= d");
  IG_REQUIRE(rope_theta > 0.f, "rope_theta must be > 0");
  IG_REQUIRE(Lcap >= pool->cap && Lcap % 8 == 0, "Lcap must cover the pool and be a multiple of 8");
  IG_REQUIRE(X && Wq_t && Wk_t && Wv_t && A && cols && A_cols && Kpart, "null pointer argument");
  IG_REQUIRE(aligned(X, 16) && aligned(Wq_t, 16) && aligned(Wk_t, 16) && aligned(Wv_t, 16),
             "X and the weights must be 16-byte aligned");
  size_t oc, ot, tot;
  prefill_layout(B, N, H, d, &oc, &ot, &tot);
  if (!workspace || workspace_bytes < tot)
    return fail(IG_ERR_CAPACITY, "the prefill needs %zu workspace bytes", tot);
  IG_REQUIRE(aligned(workspace, 256), "workspace must be 256-byte aligned");
  cudaStream_t st = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  uint16_t* Kt = reinterpret_cast<uint16_t*>(ws);
  float* colpart = reinterpret_cast<float*>(ws + oc);
  float* tab = reinterpret_cast<float*>(ws + ot);
  const int M = B * N, Nn = H * d;
  IG_REQUIRE((M + kGM - 1) / kGM <= 65535, "B*N too large for one launch");
  // the lock covers the side stream's creation on first use as well as the enqueue sequence
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* ss = nullptr;
  ig_status r = side_stream(&ss);
  if (r != IG_OK) return r;
  const size_t le = (size_t)B * H * pool->cap * d;
  // Step 1: K = X W_K, rotated and skewed row by row (with the column partials); its pool rows
  // go out on the side stream while V is projected
  r = gemm(st, X, Wk_t, Kt, M, Nn, D, nullptr);
  if (r != IG_OK) return r;
  const int half = d / 2;
  k_rope_table<<<(N * half + 255) / 256, 256, 0, st>>>(N, half, d, (double)rope_theta, tab);
  IG_CHECK_LAUNCH("RoPE table launch");
  const int mt = (M + kRsRows - 1) / kRsRows;
  const size_t smem = ((size_t)d * d + (size_t)kRsRows * d + 2 * d) * sizeof(float);
  dim3 rg(mt, H);
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(k_rope_skew<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "rope-skew smem attribute");
    k_rope_skew<128><<<rg, 256, smem, st>>>(reinterpret_cast<__half*>(Kt), M, N, H, A, tab, colpart);
  } else {
    e = cudaFuncSetAttribute(k_rope_skew<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "rope-skew smem attribute");
    k_rope_skew<64><<<rg, 256, smem, st>>>(reinterpret_cast<__half*>(Kt), M, N, H, A, tab, colpart);
  }
  IG_CHECK_LAUNCH("rope-skew launch");
  r = fork_pool_rows(st, ss, 0, Kt, B, N, H, d, pool->cap, pool->Kdev + (size_t)layer * le);
  if (r != IG_OK) return r;
  // V's pool rows come from the GEMM's epilogue
  r = gemm(st, X, Wv_t, nullptr, M, Nn, D, nullptr, PoolOut{pool->Vdev + (size_t)layer * le, N, H, d, pool->cap});
  if (r != IG_OK) return r;
  // Step 2: the columns (W~_Q from Wq_t, the keys' partials over 64-row tiles)
  k_choose_cols<<<H, d, d * sizeof(double), st>>>(reinterpret_cast<const __half*>(Wq_t), D, H, d, k, colpart, mt,
                                                  cols, nullptr);
  IG_CHECK_LAUNCH("column choice launch");
  // Step 3: A[:, S] and the partial key cache; then wait for the pool rows
  k_extract_acols<<<H, 256, 0, st>>>(A, d, k, cols, A_cols, error_word());
  IG_CHECK_LAUNCH("partial skew launch");
  dim3 sg((N + kScTok - 1) / kScTok, H, B);
  k_partial_keys<<<sg, 256, kScTok * d * 2, st>>>(reinterpret_cast<const __half*>(Kt), N, H, d, k, pool->cap, Lcap,
                                                 cols, reinterpret_cast<__half*>(Kpart), error_word());
  IG_CHECK_LAUNCH("partial keys launch");
  return join_side(st, ss);
}
