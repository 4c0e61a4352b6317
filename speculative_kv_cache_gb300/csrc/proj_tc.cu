// Partial query projection on the 5th-generation tensor cores (InfiniGen paper-graph summary,
// section 3.4, "Decoding Stage", Step 1: q~p = x_a^(i-1) W~_Q^p,(i)).
//
// part[s][b][n] = sum_{r in split s} x[b][r] * Wt[n][r], computed as D = A * B with
//   A = Wt tile  (M = 128 output components x K, K-major: row n of Wt holds its D weights)
//   B = x tile   (N = 16 batch rows x K, K-major)
// so the batch (1..16 rows) is the MMA's N and the 128 components fill its M (swap-AB).
// One CTA per (128-component tile, reduction split, 16-row batch chunk); the reduction is
// split so that the grid holds about two CTAs per SM and runs in one wave.  Thread 0 streams
// the CTA's K range through a ring of four 64-wide 128B-swizzled stages (TMA, one "full"
// mbarrier each), issues one tcgen05.mma (128x16x16, fp16 in, fp32 accumulate in tensor
// memory) per 16-wide K step as the stages land, and refills a stage once the MMAs that read
// it have completed (tcgen05.commit onto its "empty" mbarrier), one stage behind, so loads
// stay in flight; a final commit signals the accumulator.  The four warps then read the
// accumulator rows of their TMEM sub-partition with tcgen05.ld and write the fp32 partials.
// The weight stream is the whole cost (30.5 MB per layer at the OPT-30B shape).
#include <cuda.h>

#include <mutex>

#include "ig_common.cuh"
#include "tc_common.cuh"

namespace ig {

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point (no -lcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D fp16 tensor [rows][cols] (cols contiguous), boxes of 64 columns x box_rows rows, 128B swizzle
ig_status make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(IG_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IG_ERR_INVALID, "tensor map encoding failed (%d)", (int)r);
  return IG_OK;
}


namespace {

constexpr int kTcM = 128;       // output components per CTA (tcgen05 M)
constexpr int kTcN = 16;        // batch rows per CTA (tcgen05 N)
constexpr int kTcBK = 64;       // K per stage: one 128-byte swizzle atom of fp16
constexpr int kTcThreads = 128;
#ifndef IG_TC_RING
#define IG_TC_RING 4
#endif
#ifndef IG_TC_CTAS_PER_SM
#define IG_TC_CTAS_PER_SM 2
#endif
constexpr int kTcRing = IG_TC_RING;  // stages in the ring
constexpr uint32_t kStageA = kTcM * kTcBK * 2;  // 16 KB
constexpr uint32_t kStageB = kTcN * kTcBK * 2;  // 2 KB
constexpr uint32_t kTmemCols = 32;              // minimum allocation; 16 columns used

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16 (formats 0), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);

__global__ void __launch_bounds__(kTcThreads) k1_partial_q_tc(
    const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
    float* __restrict__ part, int B, int D, int N, int split_k, int* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled stages
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int m0 = blockIdx.x * kTcM;
  const int s = blockIdx.y;
  const int b0 = blockIdx.z * kTcN;
  const int k_begin = s * split_k;
  const int k_end = min(D, k_begin + split_k);
  const int nst = (k_end - k_begin + kTcBK - 1) / kTcBK;  // stages of this CTA's K range
  const int R = nst < kTcRing ? nst : kTcRing;            // slots of the ring in use
  unsigned char* sA = smem;                               // kTcRing weight stages
  unsigned char* sB = smem + kTcRing * kStageA;           // kTcRing x stages
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kTcRing * kStageB);
  uint64_t* empty = full + kTcRing;
  uint64_t* done = empty + kTcRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the kernel after this one (the RoPE epilogue or the selection) may start now: it reads
  // this kernel's output only after its own pdl_wait()
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // the weight, read once per step, is marked first for eviction
    const uint64_t pol = l2_evict_first();
    auto load = [&](int i) {  // stage i into slot i % R
      const int slot = i % R;
      mbar_arrive_expect_tx(&full[slot], kStageA + kStageB);
      const int kx = k_begin + i * kTcBK;
      tma_load_2d_hint(sA + slot * kStageA, &map_w, kx, m0, &full[slot], pol);
      tma_load_2d(sB + slot * kStageB, &map_x, kx, b0, &full[slot]);
    };
    int issued = 0, consumed = 0;
    for (; issued < R; ++issued) load(issued);
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
      const int slot = i % R;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)(i / R) & 1u)) {
        ok = false;
        break;
      }
      consumed = i + 1;
      tc_fence_after();
      const uint32_t a0 = smem_addr(sA + slot * kStageA), bb0 = smem_addr(sB + slot * kStageB);
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk) {
        const uint64_t ad = sw128_desc(a0 + kk * 32), bd = sw128_desc(bb0 + kk * 32);
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
            "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc));
      }
      // the slot is free once these MMAs have read it
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_addr(&empty[slot]))
                   : "memory");
      // refill the previous stage's slot (its MMAs were issued one step earlier)
      if (i >= 1 && issued < nst) {
        const int ps = (i - 1) % R;
        if (!mbar_wait_bounded(&empty[ps], (uint32_t)((i - 1) / R) & 1u)) {
          ok = false;
          break;
        }
        load(issued++);
      }
    }
    if (!ok) {
      *abort_flag = 1;
      raise_error(err, IG_DEVERR_TIMEOUT);
      // let the copies in flight land before the CTA leaves
      for (int u = consumed; u < issued; ++u) mbar_wait_bounded(&full[u % R], (uint32_t)(u / R) & 1u);
    }
    // the accumulator (and every issued MMA) is complete when `done` fires
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(done))
                 : "memory");
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  // every thread must take the same branch: the TMEM load below is warp-collective
  const bool landed = __syncthreads_and(mbar_wait_bounded(done, 0) ? 1 : 0) != 0;
  if (!landed) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_TIMEOUT);
  } else if (!aborted) {
    tc_fence_after();
    // warp w reads TMEM lanes 32w..32w+31 = output components m0 + 32w + lane, 16 batch columns
    uint32_t r[16];
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const int n = m0 + warp * 32 + lane;
    if (n < N) {
#pragma unroll
      for (int j = 0; j < kTcN; ++j)
        if (b0 + j < B) part[((size_t)s * B + b0 + j) * N + n] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// shared memory of the ring: 4 stages of 18 KB (three CTAs share an SM)
size_t tc_smem_bytes() { return 1024 + kTcRing * (kStageA + kStageB) + (2 * kTcRing + 1) * 8 + 16; }

}  // namespace

// Split of the reduction axis: about two CTAs per SM over the (component tile, batch chunk)
// grid, at most S splits (the workspace's), each a multiple of 64 wide.
int tc_split_k(int D, int S, int tiles, int sms) {
  int want = (IG_TC_CTAS_PER_SM * sms + tiles / 2) / (tiles > 0 ? tiles : 1);
  if (want < 1) want = 1;
  if (want > S) want = S;
  int per = (D + want - 1) / want;
  return (per + kTcBK - 1) / kTcBK * kTcBK;
}

// part[s][b][n] for s < S_eff = ceil(D / split_k); returns S_eff through *s_eff.
ig_status launch_partial_q_tc(cudaStream_t st, const __half* x, const __half* Wt, float* part, int B, int D,
                              int N, int S, int* s_eff) {
  IG_REQUIRE(D % 8 == 0, "D must be a multiple of 8 (16-byte rows for the tensor maps)");
  IG_REQUIRE(aligned(x, 16) && aligned(Wt, 16), "x and the weight must be 16-byte aligned");
  const int tiles = ((N + kTcM - 1) / kTcM) * ((B + kTcN - 1) / kTcN);
  const int split_k = tc_split_k(D, S, tiles, sm_count(st));
  const int se = (D + split_k - 1) / split_k;
  IG_REQUIRE(se <= S, "reduction split exceeds the workspace");
  CUtensorMap mw, mx;
  ig_status r = make_map(&mw, Wt, N, D, kTcM);
  if (r != IG_OK) return r;
  r = make_map(&mx, x, B, D, kTcN);
  if (r != IG_OK) return r;
  const size_t smem = tc_smem_bytes();
  cudaError_t ae = cudaFuncSetAttribute(k1_partial_q_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (ae != cudaSuccess) return cuda_fail(ae, "tensor-core projection smem attribute");
  dim3 grid((N + kTcM - 1) / kTcM, se, (B + kTcN - 1) / kTcN);
  k1_partial_q_tc<<<grid, kTcThreads, smem, st>>>(mw, mx, part, B, D, N, split_k, error_word());
  IG_CHECK_LAUNCH("tensor-core projection launch");
  *s_eff = se;
  return IG_OK;
}

}  // namespace ig
