// Fused speculated scores + threshold selection (InfiniGen paper-graph summary, section 3.4,
// "Decoding Stage", Steps 2-3), with the scores kept on chip.
//
// Persistent CTAs, each streaming whole heads (sequence, head) one after another: CTA i takes
// heads i, i + grid, i + 2 grid, ...  A head's partial keys are k rows of Lcap tokens, adjacent
// in memory (the cache is [B][H][k][Lcap]).  The warps have two roles.  A producer warp stages
// the rows R at a time (its lanes issue one bulk copy per row, of the head's L resident tokens)
// into a ring of stages, running ahead into the next head, so that loads stay in flight
// while the consumers reduce and compact.  Eight consumer warps each own a fixed set of the
// head's tokens (runs of eight, 8 p .. 8 p + 7 for p = thread + 256 m) and keep their scores in
// registers (one 16-byte shared-memory load per run and row):
// every stage adds its R rows' terms q_c K_ct in row order, so each score is the same fp32 fmaf
// chain over c = 0..k-1 as in the separate score kernel; a consumer warp hands a stage back
// through an "empty" mbarrier.  The next head's split partials of the projection are fetched
// with cp.async meanwhile.  At the head's end the scores go to an on-chip score row, the
// consumers reduce the maximum m, and each warp compacts a contiguous run of tokens with
// (m - s) < alpha in token order (ballot + popc: a count pass, then a write pass at the warp's
// offset), so the result is identical to the separate score and select kernels'.
#include <math.h>

#include "ig_common.cuh"

namespace ig {

ig_status launch_partial_q_tc(cudaStream_t st, const __half* x, const __half* Wt, float* part, int B,
                              int D, int N, int S, int* s_eff);
ig_status launch_rope_project(cudaStream_t st, const float* part, int S, int B, int H, int d, int k,
                              const float* A_cols, const int* pos, float theta, float* qp);
int projection_splits(int D);

namespace {

constexpr int kSConsumerWarps = 8;
constexpr int kSConsumers = kSConsumerWarps * 32;
constexpr int kSThreads = kSConsumers + 32;         // + the producer warp
#ifndef IG_K23_STAGES
#define IG_K23_STAGES 3
#endif
#ifndef IG_K23_STAGE_KB
#define IG_K23_STAGE_KB 32
#endif
#ifndef IG_K23_MIN_CTAS
#define IG_K23_MIN_CTAS 2
#endif
constexpr int kSMaxStages = IG_K23_STAGES;          // ring of staged row groups
constexpr int kSRun = 8;                            // consecutive tokens a consumer thread owns
constexpr int kSBlock = kSRun * kSConsumers;        // 2048 tokens: one run per thread
constexpr int kSMaxLcap = 4 * kSBlock;              // 8192 tokens: four runs per thread
constexpr int kSStageTarget = IG_K23_STAGE_KB * 1024;  // bytes of rows per stage (at least one row)

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// barrier 1 among the consumer warps only (the producer never joins it)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSConsumers) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Shared-memory layout of one CTA (all offsets 128-byte aligned).
struct SelLayout {
  int R;   // rows per stage
  int NS;  // stages in the ring
  size_t qs, qbuf, sc, stage, stage_bytes, total;
};

__host__ __device__ inline size_t al128(size_t x) { return (x + 127) / 128 * 128; }

__host__ __device__ inline SelLayout sel_layout(int S, int k, int Lcap, int NS) {
  SelLayout l;
  l.NS = NS;
  l.R = kSStageTarget / (Lcap * 2);
  if (l.R < 1) l.R = 1;
  if (l.R > k) l.R = k;
  if (l.R > 32) l.R = 32;                          // one row per producer lane
  l.qs = 256;                                      // [0, 256): full[] and empty[] mbarriers, flags
  l.qbuf = l.qs + al128((size_t)k * 4);            // scaled query, k floats
  l.sc = l.qbuf + al128((size_t)2 * S * k * 4);    // split partials of two heads
  l.stage = l.sc + al128((size_t)Lcap * 4);        // the head's scores
  l.stage_bytes = al128((size_t)l.R * Lcap * 2);
  l.total = l.stage + (size_t)NS * l.stage_bytes;
  return l;
}


// MAXB runs of kSRun tokens per consumer thread: Lcap <= kSBlock * MAXB.
template <int MAXB>
__global__ void __launch_bounds__(kSThreads, IG_K23_MIN_CTAS) k23_score_select(
    const float* __restrict__ qsrc, int S, int B, int H, int k, const __half* __restrict__ Kpart,
    const int* __restrict__ L_valid, int Lcap, float scale, float alpha, int32_t* __restrict__ idx,
    int32_t* __restrict__ cnt, uint8_t* __restrict__ used, float* __restrict__ scores_out,
    float* __restrict__ q_out, int NS, int* err) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red_f[kSConsumerWarps];
  __shared__ int red_i[kSConsumerWarps];
  const SelLayout lay = sel_layout(S, k, Lcap, NS);
  const int R = lay.R;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kSMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kSMaxStages);
  float* qs = reinterpret_cast<float*>(smem + lay.qs);
  float* qbuf = reinterpret_cast<float*>(smem + lay.qbuf);
  float* sc = reinterpret_cast<float*>(smem + lay.sc);
  const int BH = B * H, N = H * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto head_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };
  auto len_of = [&](int bh) {
    const int L = L_valid[bh / H];
    return L < 0 ? 0 : (L > Lcap ? Lcap : L);
  };
  auto stage_ptr = [&](int st) { return reinterpret_cast<__half*>(smem + lay.stage + (size_t)st * lay.stage_bytes); };

  if (head_of(0) >= BH) return;
  if (tid == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kSConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSConsumerWarps) {
    // ---------------- producer warp ----------------
    const uint64_t pol = l2_evict_first();
    int issued = 0;
    for (int i = 0; head_of(i) < BH; ++i) {
      const int bh = head_of(i);
      const int L = len_of(bh);
      if (L == 0) continue;
      const int n_copy = (L + 7) & ~7;  // within Lcap: L <= Lcap, Lcap % 8 == 0
      const __half* head_rows = Kpart + (size_t)bh * k * Lcap;
      for (int c0 = 0; c0 < k; c0 += R) {
        const int rows = min(R, k - c0);
        const int st = issued % NS, use = issued / NS;
        if (use > 0 && !mbar_wait_bounded(&empty[st], (uint32_t)(use - 1) & 1u)) {
          // the consumers never released the stage: stop staging (their bounded waits end too)
          if (lane == 0) {
            raise_error(err, IG_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          return;
        }
        __half* dst = stage_ptr(st);
        if (lane == 0) {
          // the stage was last read through the generic proxy; order that before the async writes
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive_expect_tx(&full[st], (uint32_t)(rows * n_copy * 2));
        }
        __syncwarp();
        if (lane < rows)
          bulk_g2s_hint(dst + (size_t)lane * Lcap, head_rows + (size_t)(c0 + lane) * Lcap, n_copy * 2, &full[st], pol);
        ++issued;
      }
    }
    // stay until the consumers have released every stage that was filled
    for (int u = issued > NS ? issued - NS : 0; u < issued; ++u)
      mbar_wait_bounded(&empty[u % NS], (uint32_t)(u / NS) & 1u);
    return;
  }

  // ---------------- consumer warps ----------------
  const uint32_t lim = wait_limit(err);
  auto prefetch_q = [&](int bh, int half) {
    const int b = bh / H, h = bh % H;
    float* dst = qbuf + (size_t)half * S * k;
    for (int e = tid; e < S * k; e += kSConsumers) {
      const int sp = e / k, c = e - sp * k;
      cp_async4(dst + e, qsrc + ((size_t)sp * B + b) * N + (size_t)h * k + c);
    }
    cp_async_commit();
  };
  // the kernel may start while the projection (or the RoPE epilogue) still runs: the producer's
  // partial-key copies do not depend on it, the query does
  pdl_wait();
  prefetch_q(head_of(0), 0);
  int g = 0;                          // stages consumed so far
  for (int i = 0; head_of(i) < BH; ++i) {
    const int bh = head_of(i), b = bh / H;
    int L = L_valid[b];
    if (L < 0 || L > Lcap) {
      if (tid == 0) raise_error(err, IG_DEVERR_INDEX);
      L = L < 0 ? 0 : Lcap;
    }
    // this head's query: the split partials summed in order, scaled once
    cp_async_wait_all();
    consumer_sync();
    const float* qb = qbuf + (size_t)(i & 1) * S * k;
    for (int c = tid; c < k; c += kSConsumers) {
      float a = 0.f;
      for (int sp = 0; sp < S; ++sp) a += qb[(size_t)sp * k + c];
      qs[c] = a * scale;
      if (q_out) q_out[(size_t)bh * k + c] = a;
    }
    consumer_sync();
    if (head_of(i + 1) < BH) prefetch_q(head_of(i + 1), (i + 1) & 1);

    // scores of this thread's token runs, row group by row group
    float acc[kSRun * MAXB];
#pragma unroll
    for (int m = 0; m < kSRun * MAXB; ++m) acc[m] = 0.f;
    bool ok = L > 0;
    for (int c0 = 0; L > 0 && c0 < k; c0 += R, ++g) {
      const int st = g % NS;
      const uint32_t par = (uint32_t)(g / NS) & 1u;
      bool landed = ok && !*abort_flag;
      if (landed && !mbar_wait_bounded(&full[st], par, lim)) {
        if (lane == 0) raise_error(err, IG_DEVERR_TIMEOUT);
        landed = mbar_wait_bounded(&full[st], par);  // the default limit: copies land long before it
        if (!landed) *abort_flag = 1;               // nothing more is waited for or released
      }
      ok = ok && landed;
      if (landed) {
        const __half* Ks = stage_ptr(st) + kSRun * tid;
        const int rows = min(R, k - c0);
        for (int r = 0; r < rows; ++r) {
          const float qc = qs[c0 + r];
          const __half* row = Ks + (size_t)r * Lcap;
#pragma unroll
          for (int m = 0; m < MAXB; ++m) {
            // a run that starts below L lies within the copied ceil8(L) tokens
            if (kSRun * tid + kSBlock * m < L) {
              const uint4 v = *reinterpret_cast<const uint4*>(row + kSBlock * m);
              const float2 f0 = h2_to_f2(v.x), f1 = h2_to_f2(v.y), f2 = h2_to_f2(v.z), f3 = h2_to_f2(v.w);
              float* a = acc + kSRun * m;
              a[0] = fmaf(qc, f0.x, a[0]);
              a[1] = fmaf(qc, f0.y, a[1]);
              a[2] = fmaf(qc, f1.x, a[2]);
              a[3] = fmaf(qc, f1.y, a[3]);
              a[4] = fmaf(qc, f2.x, a[4]);
              a[5] = fmaf(qc, f2.y, a[5]);
              a[6] = fmaf(qc, f3.x, a[6]);
              a[7] = fmaf(qc, f3.y, a[7]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
      }
    }
    // the scores to the score row (and out, when asked for), with the running maximum
    float mx = -INFINITY;
#pragma unroll
    for (int m = 0; m < MAXB; ++m) {
      const int t0 = kSRun * tid + kSBlock * m;
      if (t0 < L) {
#pragma unroll
        for (int j = 0; j < kSRun; ++j) {
          const float sj = (ok && t0 + j < L) ? acc[kSRun * m + j] : -INFINITY;
          mx = fmaxf(mx, sj);  // fmaxf ignores NaN
          if (t0 + j < L) {
            sc[t0 + j] = sj;
            if (scores_out) scores_out[(size_t)bh * Lcap + t0 + j] = sj;
          }
        }
      }
    }
    // the head's maximum
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_f[warp] = mx;
    consumer_sync();
    float m = -INFINITY;
    for (int w = 0; w < kSConsumerWarps; ++w) m = fmaxf(m, red_f[w]);
    // ordered compaction: warp w owns tokens [w seg, (w + 1) seg); a count pass, the warps'
    // offsets, then a write pass.  With no valid token m is -inf and m - s is NaN: nothing kept.
    const int seg = ((L + kSConsumerWarps - 1) / kSConsumerWarps + 31) / 32 * 32;
    const int wa = min(L, warp * seg), we = min(L, wa + seg);
    int wcount = 0;
    for (int t0 = wa; t0 < we; t0 += 32) {
      const int t = t0 + lane;
      const bool f = t < we && !isnan(sc[t]) && (m - sc[t]) < alpha;
      wcount += __popc(__ballot_sync(0xffffffffu, f));
    }
    if (lane == 0) red_i[warp] = wcount;
    consumer_sync();
    int pos = 0, total = 0;
    for (int w = 0; w < kSConsumerWarps; ++w) {
      if (w < warp) pos += red_i[w];
      total += red_i[w];
    }
    int32_t* io = idx + (size_t)bh * Lcap;
    const uint32_t lt = (1u << lane) - 1u;
    for (int t0 = wa; t0 < we; t0 += 32) {
      const int t = t0 + lane;
      const bool f = t < we && !isnan(sc[t]) && (m - sc[t]) < alpha;
      const uint32_t bal = __ballot_sync(0xffffffffu, f);
      if (f) {
        io[pos + __popc(bal & lt)] = t;
        if (used) used[(size_t)b * Lcap + t] = 1;
      }
      pos += __popc(bal);
    }
    if (tid == 0) cnt[bh] = total;
    if (scores_out)
      for (int t = L + tid; t < Lcap; t += kSConsumers) scores_out[(size_t)bh * Lcap + t] = -INFINITY;
    consumer_sync();  // the score row and the reduction slots are reused by the next head
  }
  cp_async_wait_all();
}

}  // namespace

// Fused score + select on the split partials qsrc [S][B][H*k] (the projection's output, or the
// RoPE epilogue's [1][B][H*k]).  Requires Lcap <= kSMaxLcap.
template <int MAXB>
ig_status launch_k23(cudaStream_t st, const float* qsrc, int S, int B, int H, int k, const uint16_t* Kpart,
                     const int32_t* L_valid, int Lcap, float scale, float alpha, int32_t* idx, int32_t* cnt,
                     uint8_t* used, float* scores, float* q_part) {
  const long long heads = (long long)B * H;
  const int sms = sm_count(st);
  const int NS = kSMaxStages;
  const SelLayout lay = sel_layout(S, k, Lcap, NS);
  IG_REQUIRE(lay.total <= 220 * 1024, "k or Lcap too large for the fused selection (%zu bytes of shared memory)",
             lay.total);
  cudaError_t e = cudaFuncSetAttribute(k23_score_select<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)lay.total);
  if (e != cudaSuccess) return cuda_fail(e, "fused select smem attribute");
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k23_score_select<MAXB>, kSThreads, lay.total);
  if (e != cudaSuccess) return cuda_fail(e, "fused select occupancy");
  if (per_sm < 1) per_sm = 1;
  const long long slots = (long long)per_sm * sms;
  const int grid = (int)(heads < slots ? heads : slots);
  // programmatic launch: the partial keys stream while the query's producer finishes
  e = launch_pdl(k23_score_select<MAXB>, dim3(grid), dim3(kSThreads), lay.total, st, qsrc, S, B, H, k,
                 reinterpret_cast<const __half*>(Kpart), L_valid, Lcap, scale, alpha, idx, cnt, used, scores, q_part,
                 NS, error_word());
  if (e != cudaSuccess) return cuda_fail(e, "fused select launch");
  IG_CHECK_LAUNCH("fused select launch");
  return IG_OK;
}

ig_status launch_score_select(cudaStream_t st, const float* qsrc, int S, int B, int H, int k,
                              const uint16_t* Kpart, const int32_t* L_valid, int Lcap, float scale,
                              float alpha, int32_t* idx, int32_t* cnt, uint8_t* used, float* scores,
                              float* q_part) {
  IG_REQUIRE(Lcap <= kSMaxLcap, "fused selection needs Lcap <= %d (got %d)", kSMaxLcap, Lcap);
  if (Lcap <= kSBlock)
    return launch_k23<1>(st, qsrc, S, B, H, k, Kpart, L_valid, Lcap, scale, alpha, idx, cnt, used, scores, q_part);
  if (Lcap <= 2 * kSBlock)
    return launch_k23<2>(st, qsrc, S, B, H, k, Kpart, L_valid, Lcap, scale, alpha, idx, cnt, used, scores, q_part);
  return launch_k23<4>(st, qsrc, S, B, H, k, Kpart, L_valid, Lcap, scale, alpha, idx, cnt, used, scores, q_part);
}

}  // namespace ig

using namespace ig;

extern "C" size_t ig_speculate_select_workspace_bytes(int B, int D, int H, int d, int k, int rope) {
  if (B <= 0 || D <= 0 || H <= 0 || d <= 0 || k <= 0) return 0;
  return rope ? ig_speculate_rope_workspace_bytes(B, D, H, d, k) : ig_speculate_workspace_bytes(B, D, H, k);
}

extern "C" ig_status ig_speculate_select(void* stream, int B, int D, int H, int d, int k, int Lcap,
                                         const uint16_t* x, const uint16_t* Wq, const float* A_cols,
                                         const int32_t* positions, float rope_theta,
                                         const uint16_t* Kpart, const int32_t* L_valid,
                                         float score_scale, float alpha, int32_t* idx, int32_t* cnt,
                                         uint8_t* used, float* scores, float* q_part,
                                         void* workspace, size_t workspace_bytes) {
  IG_REQUIRE(B > 0 && D > 0 && H > 0 && d > 0 && k > 0 && k <= d, "bad sizes");
  IG_REQUIRE(Lcap > 0 && Lcap % 8 == 0, "Lcap must be a positive multiple of 8 (got %d)", Lcap);
  IG_REQUIRE(x && Wq && Kpart && L_valid && idx && cnt && workspace, "null pointer argument");
  IG_REQUIRE(aligned(Kpart, 16) && aligned(workspace, 256), "Kpart 16-byte, workspace 256-byte aligned");
  IG_REQUIRE(!scores || aligned(scores, 16), "scores must be 16-byte aligned");
  IG_REQUIRE(alpha > 0.f, "alpha must be > 0 (got %g)", (double)alpha);
  const bool rope = rope_theta > 0.f;
  IG_REQUIRE(!rope || (A_cols && positions && d % 2 == 0), "RoPE needs A_cols, positions and an even d");
  const size_t need = ig_speculate_select_workspace_bytes(B, D, H, d, k, rope ? 1 : 0);
  if (workspace_bytes < need) return fail(IG_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  IG_REQUIRE(Lcap <= kSMaxLcap, "fused selection needs Lcap <= %d (got %d)", kSMaxLcap, Lcap);
  cudaStream_t s = as_stream(stream);
  // the use flags are cleared before the projection, so that the selection follows the
  // projection (or the RoPE epilogue) directly and may overlap it
  if (used) {
    cudaError_t e = cudaMemsetAsync(used, 0, (size_t)B * Lcap, s);
    if (e != cudaSuccess) return cuda_fail(e, "clear used flags");
  }
  int S = projection_splits(D);
  float* part = static_cast<float*>(workspace);
  const int N = rope ? H * d : H * k;
  ig_status st = launch_partial_q_tc(s, reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(Wq),
                                     part, B, D, N, S, &S);
  if (st != IG_OK) return st;
  const float* qsrc = part;
  if (rope) {
    float* qp = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         round_up((size_t)projection_splits(D) * B * H * d * sizeof(float), 256));
    st = launch_rope_project(s, part, S, B, H, d, k, A_cols, positions, rope_theta, qp);
    if (st != IG_OK) return st;
    qsrc = qp;
    S = 1;
  }
  return launch_score_select(s, qsrc, S, B, H, k, Kpart, L_valid, Lcap, score_scale, alpha, idx, cnt, used,
                             scores, q_part);
}
