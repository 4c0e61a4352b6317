// Speculation for layer i from layer i-1's attention input (InfiniGen paper-graph summary,
// section 3.4, "Decoding Stage", Steps 1-2):
//   K1  partial query projection  q~p = x W~_Q^p       tcgen05 tensor cores (proj_tc.cu), split-K,
//                                                       fp32 partial sums in workspace
//   K1b RoPE epilogue (Llama)     q~p = RoPE(x W_Q) A[:, S]
//   K2  speculated scores         s = scale q~p (K~p)^T, partial-key rows staged by bulk TMA
#include <math.h>

#include <mutex>

#include "ig_common.cuh"

namespace ig {
ig_status launch_partial_q_tc(cudaStream_t st, const __half* x, const __half* Wt, float* part, int B,
                              int D, int N, int S, int* s_eff);
namespace {

constexpr int kMaxSplits = 32;

// Number of K-splits of the projection for a given reduction length: 256-wide pieces (four
// 64-wide tensor-core stages each), at most 32.
inline int proj_splits(int D) {
  int s = (D + 255) / 256;
  return s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
}

// K1: the partial query projection runs on the tensor cores (proj_tc.cu); part holds S_eff
// split partials [S_eff][B][N] of x W (W given transposed, [N][D]).
ig_status launch_k1(cudaStream_t st, const __half* x, const __half* Wt, float* part, int B, int D,
                    int N, int S, int* s_eff) {
  return launch_partial_q_tc(st, x, Wt, part, B, D, N, S, s_eff);
}


// K1b: RoPE epilogue for one (b, h) (launched so that it may start during the projection: the
// copy of A[:, S] is issued first, the partials are read after pdl_wait): q = sum of the split
// partials of x W_Q,h; rotate the
// pairs (j, j + d/2) by the angle p * theta^(-2j/d) (the inverse frequencies come from the host
// in float64; the angle is formed and reduced to [-pi, pi] in float64, then rotated in
// float64); then q~p[c] = sum_j q_rot[j] A[h][j][c] with A[h][:, S_h] (a contiguous d x k
// block) staged in shared memory by one bulk copy that overlaps the split sums, and one warp
// per output c.
constexpr int kRopeMaxHalf = 128;  // d <= 256
struct InvFreq {
  double v[kRopeMaxHalf];
};

__global__ void k1b_rope_project(const float* __restrict__ part, int S, int B, int H, int d, int k,
                                 const float* __restrict__ A_cols, const int* __restrict__ pos,
                                 const __grid_constant__ InvFreq inv, float* __restrict__ qp, int* err) {
  extern __shared__ __align__(16) float sh[];
  const int dk = d * k;
  float* As = sh;                                    // d * k (16-byte aligned: first)
  float* q = sh + ((dk + 3) & ~3);                   // d
  float* qr = q + d;                                 // d
  uint64_t* bar = reinterpret_cast<uint64_t*>(qr + ((d + 1) & ~1));
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  const int N = H * d;
  const float* Ah = A_cols + (size_t)h * dk;
  // one bulk copy when the block is 16-byte aligned and a multiple of 16 bytes, else plain loads
  const bool bulk = (reinterpret_cast<uintptr_t>(Ah) % 16) == 0 && (dk % 4) == 0;
  if (bulk && threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)(dk * 4));
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(As)),
        "l"(Ah), "r"(dk * 4), "r"(smem_addr(bar))
        : "memory");
  }
  pdl_trigger();
  pdl_wait();  // the projection's partials are complete and visible from here on
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    q[j] = sum_splits(part + (size_t)b * N + h * d + j, (size_t)B * N, S);
  }
  if (!bulk) {
    for (int i0 = threadIdx.x; i0 < dk; i0 += 8 * blockDim.x) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = i0 + u * (int)blockDim.x < dk ? __ldg(Ah + i0 + u * blockDim.x) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * (int)blockDim.x < dk) As[i0 + u * blockDim.x] = v[u];
    }
  }
  __syncthreads();
  const int half = d / 2;
  const double p = (double)pos[b];
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const double a = p * inv.v[j];
    const double r = a - two_pi * rint(a / two_pi);
    double sn, cs;
    sincos(r, &sn, &cs);
    const float lo = q[j], hi = q[j + half];
    qr[j] = (float)((double)lo * cs - (double)hi * sn);
    qr[j + half] = (float)((double)lo * sn + (double)hi * cs);
  }
  bool landed = true;
  if (bulk) {
    landed = mbar_wait_bounded(bar, 0);
    if (!landed && threadIdx.x == 0) raise_error(err, IG_DEVERR_TIMEOUT);
  }
  landed = __syncthreads_and(landed ? 1 : 0) != 0;
  if (!landed) {
    mbar_wait_bounded(bar, 0);  // let the copy land (bounded) before the CTA leaves
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int c = warp; c < k; c += nw) {
    float a = 0.f;
    for (int j = lane; j < d; j += 32) a = fmaf(qr[j], As[j * k + c], a);
    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) qp[((size_t)b * H + h) * k + c] = a;
  }
}

// K2: speculated scores for one (b, h) and a chunk of T tokens.  Thread 0 stages the k
// partial-key rows of the chunk (T fp16 each, contiguous in the column-major cache) with k
// bulk copies completing on one mbarrier; each thread then scores 4 tokens out of shared
// memory.  The partial query is the sum of the S split partials, scaled once.
__global__ void k2_scores(const float* __restrict__ qsrc, int S, int B, int H, int k,
                          const __half* __restrict__ Kpart, const int* __restrict__ L_valid,
                          int Lcap, int T, float scale, float* __restrict__ scores,
                          float* __restrict__ q_out, int* err) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float* qs = reinterpret_cast<float*>(smem + 16);
  __half* Ks = reinterpret_cast<__half*>(smem + 16 + ((k * 4 + 127) & ~127));
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int t0 = blockIdx.x * T;
  int L = L_valid[b];
  if (L < 0 || L > Lcap) {
    if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
    L = L < 0 ? 0 : Lcap;
  }
  const int n_tok = max(0, min(T, L - t0));
  const int n_copy = (n_tok + 7) & ~7;
  const __half* rows = Kpart + ((size_t)bh * k) * Lcap + t0;
  if (threadIdx.x == 0 && n_copy > 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)(k * n_copy * 2));
    const uint64_t pol = l2_evict_first();
    for (int c = 0; c < k; ++c) bulk_g2s_hint(Ks + (size_t)c * T, rows + (size_t)c * Lcap, n_copy * 2, bar, pol);
  }
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    const int N = H * k;
    const float a = sum_splits(qsrc + (size_t)b * N + h * k + c, (size_t)B * N, S);
    qs[c] = a * scale;
    if (q_out && blockIdx.x == 0) q_out[(size_t)bh * k + c] = a;
  }
  __syncthreads();
  const int tl = threadIdx.x * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (n_copy > 0) {
    if (!mbar_wait_bounded(bar, 0, wait_limit(err))) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_TIMEOUT);
      mbar_wait_bounded(bar, 0);  // let the copies in flight land (default limit) before leaving
      return;
    }
    if (tl < n_tok) {
      for (int c = 0; c < k; ++c) {
        uint2 v = *reinterpret_cast<const uint2*>(Ks + (size_t)c * T + tl);
        float2 f0 = h2_to_f2(v.x), f1 = h2_to_f2(v.y);
        const float qc = qs[c];
        acc[0] = fmaf(qc, f0.x, acc[0]);
        acc[1] = fmaf(qc, f0.y, acc[1]);
        acc[2] = fmaf(qc, f1.x, acc[2]);
        acc[3] = fmaf(qc, f1.y, acc[3]);
      }
    }
  }
  const int t = t0 + tl;
  if (tl < T && t < Lcap) {
    float4 o;
    o.x = (t + 0 < L) ? acc[0] : -INFINITY;
    o.y = (t + 1 < L) ? acc[1] : -INFINITY;
    o.z = (t + 2 < L) ? acc[2] : -INFINITY;
    o.w = (t + 3 < L) ? acc[3] : -INFINITY;
    *reinterpret_cast<float4*>(scores + (size_t)bh * Lcap + t) = o;
  }
}

// Tokens per score CTA: as many as keep the staged rows within 80 KB (two or more CTAs per SM).
inline int score_chunk(int k) {
  int T = 512;
  while (T > 64 && (size_t)k * T * 2 > 80 * 1024) T >>= 1;
  return T;
}

inline size_t score_smem(int k, int T) { return 16 + round_up((size_t)k * 4, 128) + (size_t)k * T * 2; }

ig_status launch_k2(cudaStream_t st, const float* qsrc, int S, int B, int H, int k,
                    const uint16_t* Kpart, const int32_t* L_valid, int Lcap, float scale,
                    float* scores, float* q_part) {
  const int T = score_chunk(k);
  const size_t sm = score_smem(k, T);
  cudaError_t e = cudaFuncSetAttribute(k2_scores, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return cuda_fail(e, "score kernel smem attribute");
  dim3 grid((Lcap + T - 1) / T, B * H);
  k2_scores<<<grid, T / 4, sm, st>>>(qsrc, S, B, H, k, reinterpret_cast<const __half*>(Kpart),
                                     L_valid, Lcap, T, scale, scores, q_part, error_word());
  IG_CHECK_LAUNCH("score kernel launch");
  return IG_OK;
}

ig_status check_common(int B, int D, int H, int k, int Lcap, const void* x, const void* Kpart,
                       const void* L_valid, const void* scores, const void* ws) {
  IG_REQUIRE(B > 0 && D > 0 && H > 0 && k > 0, "B, D, H, k must be positive (got %d %d %d %d)", B, D, H, k);
  IG_REQUIRE(Lcap > 0 && Lcap % 8 == 0, "Lcap must be a positive multiple of 8 (got %d)", Lcap);
  IG_REQUIRE(x && Kpart && L_valid && scores && ws, "null pointer argument");
  IG_REQUIRE(aligned(Kpart, 16), "Kpart must be 16-byte aligned");
  IG_REQUIRE(aligned(scores, 16), "scores must be 16-byte aligned");
  IG_REQUIRE(aligned(ws, 256), "workspace must be 256-byte aligned");
  IG_REQUIRE((size_t)k * 4 <= 64 * 1024, "k too large");
  return IG_OK;
}

}  // namespace

int projection_splits(int D) { return proj_splits(D); }

ig_status launch_rope_project(cudaStream_t st, const float* part, int S, int B, int H, int d, int k,
                              const float* A_cols, const int* pos, float theta, float* qp) {
  IG_REQUIRE(d / 2 <= kRopeMaxHalf, "RoPE head width d must be <= %d", 2 * kRopeMaxHalf);
  InvFreq inv = {};
  for (int j = 0; j < d / 2; ++j) inv.v[j] = pow((double)theta, -2.0 * (double)j / (double)d);
  const size_t rope_smem = (size_t)(((d * k + 3) & ~3) + 2 * ((d + 1) & ~1)) * sizeof(float) + 16;
  if (rope_smem > 48 * 1024) {
    cudaError_t ae = cudaFuncSetAttribute(k1b_rope_project, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)rope_smem);
    if (ae != cudaSuccess) return cuda_fail(ae, "rope epilogue smem attribute");
  }
  // may start during the projection: A's copy overlaps it, the partials are read after pdl_wait
  cudaError_t le = launch_pdl(k1b_rope_project, dim3(B * H), dim3(128), rope_smem, st, part, S, B, H, d, k, A_cols,
                              pos, inv, qp, error_word());
  if (le != cudaSuccess) return cuda_fail(le, "rope epilogue launch");
  IG_CHECK_LAUNCH("rope epilogue launch");
  return IG_OK;
}

}  // namespace ig

using namespace ig;

extern "C" size_t ig_speculate_workspace_bytes(int B, int D, int H, int k) {
  if (B <= 0 || D <= 0 || H <= 0 || k <= 0) return 0;
  return round_up((size_t)proj_splits(D) * B * H * k * sizeof(float), 256);
}

extern "C" ig_status ig_speculate(void* stream, int B, int D, int H, int k, int Lcap,
                                  const uint16_t* x, const uint16_t* Wq_part,
                                  const uint16_t* Kpart, const int32_t* L_valid,
                                  float score_scale, float* scores, float* q_part,
                                  void* workspace, size_t workspace_bytes) {
  ig_status st = check_common(B, D, H, k, Lcap, x, Kpart, L_valid, scores, workspace);
  if (st != IG_OK) return st;
  IG_REQUIRE(Wq_part, "null Wq_part");
  const size_t need = ig_speculate_workspace_bytes(B, D, H, k);
  if (workspace_bytes < need)
    return fail(IG_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  cudaStream_t s = as_stream(stream);
  int S = proj_splits(D);
  float* part = static_cast<float*>(workspace);
  st = launch_k1(s, reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(Wq_part),
                 part, B, D, H * k, S, &S);
  if (st != IG_OK) return st;
  return launch_k2(s, part, S, B, H, k, Kpart, L_valid, Lcap, score_scale, scores, q_part);
}

extern "C" size_t ig_speculate_rope_workspace_bytes(int B, int D, int H, int d, int k) {
  if (B <= 0 || D <= 0 || H <= 0 || d <= 0 || k <= 0) return 0;
  return round_up((size_t)proj_splits(D) * B * H * d * sizeof(float), 256) +
         round_up((size_t)B * H * k * sizeof(float), 256);
}

extern "C" ig_status ig_speculate_rope(void* stream, int B, int D, int H, int d, int k, int Lcap,
                                       const uint16_t* x, const uint16_t* Wq,
                                       const float* A_cols, const int32_t* positions,
                                       float rope_theta, const uint16_t* Kpart,
                                       const int32_t* L_valid, float score_scale,
                                       float* scores, float* q_part, void* workspace,
                                       size_t workspace_bytes) {
  ig_status st = check_common(B, D, H, k, Lcap, x, Kpart, L_valid, scores, workspace);
  if (st != IG_OK) return st;
  IG_REQUIRE(Wq && A_cols && positions, "null Wq, A_cols or positions");
  IG_REQUIRE(d > 0 && d % 2 == 0 && k <= d, "d must be even and k <= d (d=%d k=%d)", d, k);
  IG_REQUIRE(rope_theta > 0.f, "rope_theta must be positive");
  const size_t need = ig_speculate_rope_workspace_bytes(B, D, H, d, k);
  if (workspace_bytes < need)
    return fail(IG_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  cudaStream_t s = as_stream(stream);
  int S = proj_splits(D);
  float* part = static_cast<float*>(workspace);
  float* qp = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       round_up((size_t)S * B * H * d * sizeof(float), 256));
  st = launch_k1(s, reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(Wq), part,
                 B, D, H * d, S, &S);
  if (st != IG_OK) return st;
  st = launch_rope_project(s, part, S, B, H, d, k, A_cols, positions, rope_theta, qp);
  if (st != IG_OK) return st;
  return launch_k2(s, qp, 1, B, H, k, Kpart, L_valid, Lcap, score_scale, scores, q_part);
}

// ---------------------------------------------------------------------------------------
// ig_speculate_static: ig_speculate for callers that must not allocate device memory.
// The split-K partial sums live in this file-scope array instead of a caller workspace.
// The array's name is only a host-side stand-in in host code: its device address is looked
// up once per device with cudaGetSymbolAddress and handed to the kernels.
// ---------------------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB on every device that loads the library
static __device__ __align__(256) float g_speculate_scratch[kStaticScratchBytes / sizeof(float)];

std::mutex g_static_mu;
float* g_static_ptr[64] = {};

// Device address of the scratch array on the current device (looked up on first use).
ig_status static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "ig_speculate_static: current device");
  if (dev < 0 || dev >= 64) return fail(IG_ERR_INVALID, "ig_speculate_static: device %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_speculate_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "ig_speculate_static: scratch address");
    g_static_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_static_ptr[dev];
  return IG_OK;
}

}  // namespace

extern "C" ig_status ig_speculate_static(void* stream, int B, int D, int H, int k, int Lcap,
                                         const uint16_t* x, const uint16_t* Wq_part,
                                         const uint16_t* Kpart, const int32_t* L_valid,
                                         float score_scale, float* scores, float* q_part) {
  float* part = nullptr;
  ig_status st = static_scratch(&part);
  if (st != IG_OK) return st;
  st = check_common(B, D, H, k, Lcap, x, Kpart, L_valid, scores, part);
  if (st != IG_OK) return st;
  IG_REQUIRE(Wq_part, "null Wq_part");
  const size_t need = ig_speculate_workspace_bytes(B, D, H, k);
  if (need > kStaticScratchBytes)
    return fail(IG_ERR_CAPACITY,
                "ig_speculate_static needs %zu bytes of scratch for B=%d, H*k=%d, D=%d; its static "
                "scratch holds %zu bytes (use ig_speculate with a workspace)",
                need, B, H * k, D, kStaticScratchBytes);
  cudaStream_t s = as_stream(stream);
  int S = proj_splits(D);
  st = launch_k1(s, reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(Wq_part),
                 part, B, D, H * k, S, &S);
  if (st != IG_OK) return st;
  return launch_k2(s, part, S, B, H, k, Kpart, L_valid, Lcap, score_scale, scores, q_part);
}
