// Fused speculated scores + threshold selection (InfiniGen paper-graph summary, section 3.4,
// "Decoding Stage", Steps 2-3), with the scores kept on chip.
//
// One thread-block cluster per (sequence, head), one CTA per chunk of 512 tokens (at most 8
// chunks: Lcap <= 4096).  Each CTA stages its chunk of the partial key cache with bulk (TMA)
// copies, scores 4 tokens per thread into registers, and reduces its chunk maximum, which it
// writes into every CTA of the cluster (distributed shared memory); after one cluster barrier
// every CTA knows the head's maximum m.  Each thread then flags its tokens with (m - s) < alpha,
// the CTA scans its flags in token order and pushes its count the same way; after a second
// barrier each CTA sums the counts of the lower-ranked chunks and writes its indices at that
// offset.  No CTA touches another's shared memory after that barrier, so none waits for the
// others to finish.  The comparisons are the
// same fp32 operations as in the separate score and select kernels, so the result is
// identical to theirs.
#include <cooperative_groups.h>
#include <math.h>

#include "ig_common.cuh"

namespace cg = cooperative_groups;

namespace ig {

ig_status launch_partial_q_tc(cudaStream_t st, const __half* x, const __half* Wt, float* part, int B,
                              int D, int N, int S, int* s_eff);
ig_status launch_rope_project(cudaStream_t st, const float* part, int S, int B, int H, int d, int k,
                              const float* A_cols, const int* pos, float theta, float* qp);
int projection_splits(int D);

namespace {

constexpr int kFT = 512;             // tokens per CTA
constexpr int kFThreads = kFT / 4;   // 4 tokens per thread
constexpr int kFMaxChunks = 8;       // portable cluster size

__global__ void __launch_bounds__(kFThreads) k23_score_select(
    const float* __restrict__ qsrc, int S, int B, int H, int k, const __half* __restrict__ Kpart,
    const int* __restrict__ L_valid, int Lcap, float scale, float alpha, int32_t* __restrict__ idx,
    int32_t* __restrict__ cnt, uint8_t* __restrict__ used, float* __restrict__ scores_out,
    float* __restrict__ q_out, int* err) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red_f[kFThreads / 32];
  __shared__ int red_i[kFThreads / 32];
  // every CTA's chunk maximum and count, pushed here by their CTAs through distributed shared
  // memory, so that after each exchange every CTA reads only its own shared memory
  __shared__ float chunk_max[kFMaxChunks];
  __shared__ int chunk_cnt[kFMaxChunks];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float* qs = reinterpret_cast<float*>(smem + 16);
  __half* Ks = reinterpret_cast<__half*>(smem + 16 + ((k * 4 + 127) & ~127));
  const int rank = (int)cluster.block_rank();
  const int nranks = (int)cluster.num_blocks();
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int t0 = rank * kFT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int L = L_valid[b];
  if (L < 0 || L > Lcap) {
    if (threadIdx.x == 0 && rank == 0) raise_error(err, IG_DEVERR_INDEX);
    L = L < 0 ? 0 : Lcap;
  }
  // no CTA writes into another's shared memory before all of the cluster's CTAs run: arrive
  // now, wait just before the first push (by then the wait is long satisfied)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int n_tok = max(0, min(kFT, L - t0));
  const int n_copy = (n_tok + 7) & ~7;
  const __half* rows = Kpart + ((size_t)bh * k) * Lcap + t0;
  if (threadIdx.x == 0 && n_copy > 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)(k * n_copy * 2));
    const uint64_t pol = l2_evict_first();
    for (int c = 0; c < k; ++c) bulk_g2s_hint(Ks + (size_t)c * kFT, rows + (size_t)c * Lcap, n_copy * 2, bar, pol);
  }
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    const int N = H * k;
    const float a = sum_splits(qsrc + (size_t)b * N + h * k + c, (size_t)B * N, S);
    qs[c] = a * scale;
    if (q_out && rank == 0) q_out[(size_t)bh * k + c] = a;
  }
  __syncthreads();
  const int tl = threadIdx.x * 4;
  float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  bool landed = true;
  if (n_copy > 0) {
    // a copy that does not land is reported and its chunk selects nothing; the CTA still
    // takes part in every cluster barrier below
    landed = mbar_wait_bounded(bar, 0, wait_limit(err));
    if (!landed) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_TIMEOUT);
      landed = mbar_wait_bounded(bar, 0);  // the default limit: copies land long before it
    }
    if (landed && tl < n_tok) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < k; ++c) {
        uint2 v = *reinterpret_cast<const uint2*>(Ks + (size_t)c * kFT + tl);
        float2 f0 = h2_to_f2(v.x), f1 = h2_to_f2(v.y);
        const float qc = qs[c];
        acc[0] = fmaf(qc, f0.x, acc[0]);
        acc[1] = fmaf(qc, f0.y, acc[1]);
        acc[2] = fmaf(qc, f1.x, acc[2]);
        acc[3] = fmaf(qc, f1.y, acc[3]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[j] = (t0 + tl + j < L) ? acc[j] : -INFINITY;
    }
  }
  if (scores_out) {
    const int t = t0 + tl;
    if (t < Lcap) {
      float4 o = make_float4(sc[0], sc[1], sc[2], sc[3]);
      *reinterpret_cast<float4*>(scores_out + (size_t)bh * Lcap + t) = o;
    }
  }
  // chunk maximum (fmaxf ignores NaN), then the head's maximum across the cluster
  float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_f[warp] = mx;
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (threadIdx.x < nranks) {
    float cm = -INFINITY;
    for (int w = 0; w < kFThreads / 32; ++w) cm = fmaxf(cm, red_f[w]);
    *cluster.map_shared_rank(&chunk_max[rank], (unsigned)threadIdx.x) = cm;
  }
  cluster.sync();
  float m = -INFINITY;
  for (int r = 0; r < nranks; ++r) m = fmaxf(m, chunk_max[r]);
  // flags in token order; a token past L_valid scored -inf and is never kept (for alpha = inf,
  // (m - (-inf)) < inf is false, and with no valid token m - s is NaN)
  bool f[4];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = t0 + tl + j;
    f[j] = (t < L) && !isnan(sc[j]) && ((m - sc[j]) < alpha);
    mine += f[j] ? 1 : 0;
  }
  int incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red_i[warp] = incl;
  __syncthreads();
  int before = incl - mine;
  for (int w = 0; w < warp; ++w) before += red_i[w];
  if (threadIdx.x < nranks) {
    int tot = 0;
    for (int w = 0; w < kFThreads / 32; ++w) tot += red_i[w];
    *cluster.map_shared_rank(&chunk_cnt[rank], (unsigned)threadIdx.x) = tot;
  }
  cluster.sync();  // the last access to another CTA's shared memory is before this barrier
  int offset = 0, total = 0;
  for (int r = 0; r < nranks; ++r) {
    const int c = chunk_cnt[r];
    if (r < rank) offset += c;
    total += c;
  }
  int pos = offset + before;
  int32_t* io = idx + (size_t)bh * Lcap;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (f[j]) {
      const int t = t0 + tl + j;
      io[pos++] = t;
      if (used) used[(size_t)b * Lcap + t] = 1;
    }
  }
  if (rank == 0 && threadIdx.x == 0) cnt[bh] = total;
  // a CTA whose copies never landed waits for them once more (bounded) before it leaves
  if (!landed) mbar_wait_bounded(bar, 0);
}

size_t fused_smem(int k) { return 16 + round_up((size_t)k * 4, 128) + (size_t)k * kFT * 2; }

}  // namespace

// Fused score + select on the split partials qsrc [S][B][H*k] (the projection's output, or the
// RoPE epilogue's [1][B][H*k]).  Requires Lcap <= 8 * 512.
ig_status launch_score_select(cudaStream_t st, const float* qsrc, int S, int B, int H, int k,
                              const uint16_t* Kpart, const int32_t* L_valid, int Lcap, float scale,
                              float alpha, int32_t* idx, int32_t* cnt, uint8_t* used, float* scores,
                              float* q_part) {
  const int nch = (Lcap + kFT - 1) / kFT;
  IG_REQUIRE(nch <= kFMaxChunks, "fused selection needs Lcap <= %d (got %d)", kFMaxChunks * kFT, Lcap);
  const size_t sm = fused_smem(k);
  IG_REQUIRE(sm <= 200 * 1024, "k too large for the fused selection");
  cudaError_t e = cudaFuncSetAttribute(k23_score_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return cuda_fail(e, "fused select smem attribute");
  if (used) {
    e = cudaMemsetAsync(used, 0, (size_t)B * Lcap, st);
    if (e != cudaSuccess) return cuda_fail(e, "clear used flags");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nch, B * H, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nch;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k23_score_select, qsrc, S, B, H, k, reinterpret_cast<const __half*>(Kpart),
                         L_valid, Lcap, scale, alpha, idx, cnt, used, scores, q_part, error_word());
  if (e != cudaSuccess) return cuda_fail(e, "fused select launch");
  IG_CHECK_LAUNCH("fused select launch");
  return IG_OK;
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
  cudaStream_t s = as_stream(stream);
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
