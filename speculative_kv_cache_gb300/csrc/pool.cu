// KV cache pool in pinned, mapped host memory and its slot manager (InfiniGen paper-graph
// summary, section 3.4, "KV Cache Pool Management Under Memory Pressure"): the counter policy
// InfiniGen uses and the FIFO and LRU policies it is compared with in Table 2, plus the
// append of the current token ("Partial Key Cache Updates During Decoding").
#include <stdlib.h>
#include <string.h>

#include <cuda_fp8.h>

#include <new>

#include "ig_common.cuh"
#include "pool_impl.h"

namespace ig {
namespace {

// Host-side fault injection for tests: IG_FAULT=pool_alloc makes pool creation fail as if
// the pinned allocation had been refused.
bool fault_injected(const char* what) {
  const char* f = getenv("IG_FAULT");
  return f && strstr(f, what) != nullptr;
}

// K6: the current token of every (b, h): full key/value row to the pool slot (16-byte
// zero-copy stores over the host link), the k chosen columns of the key to the partial key
// cache, and optionally the full row to an HBM-resident KV.
__global__ void k6_append(uint4* __restrict__ Kp, uint4* __restrict__ Vp, int cap, int H, int d,
                          int k, int Lcap, const int32_t* __restrict__ slot,
                          const int32_t* __restrict__ cols, const __half* __restrict__ k_new,
                          const __half* __restrict__ v_new, __half* __restrict__ Kpart,
                          uint4* __restrict__ Kd, uint4* __restrict__ Vd, int* err) {
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  const int sl = slot[b];
  if (sl < 0) return;
  const int vpr = d / 8;
  const uint4* kn = reinterpret_cast<const uint4*>(k_new + (size_t)bh * d);
  const uint4* vn = reinterpret_cast<const uint4*>(v_new + (size_t)bh * d);
  if (Kp) {
    if (sl >= cap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      return;
    }
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
      Kp[((size_t)bh * cap + sl) * vpr + v] = kn[v];
      Vp[((size_t)bh * cap + sl) * vpr + v] = vn[v];
    }
  }
  if (Kpart || Kd) {
    if (sl >= Lcap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      return;
    }
  }
  if (Kd) {
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
      Kd[((size_t)bh * Lcap + sl) * vpr + v] = kn[v];
      Vd[((size_t)bh * Lcap + sl) * vpr + v] = vn[v];
    }
  }
  if (Kpart) {
    for (int c = threadIdx.x; c < k; c += blockDim.x) {
      int col = cols[h * k + c];
      if (col < 0 || col >= d) {
        raise_error(err, IG_DEVERR_INDEX);
        continue;
      }
      Kpart[((size_t)bh * k + c) * Lcap + sl] = k_new[(size_t)bh * d + col];
    }
  }
}

// One warp quantizes one row of d fp16 values (d = 32 * PER, lane i holding elements
// PER i .. PER i + PER - 1) with one fp32 scale per row; a row of zeros gets scale 0 and zero
// codes.  BITS = 8: e4m3 codes, scale amax / 448, codes = RN-even e4m3, saturating, of
// x * (448 / amax) in fp32.  BITS = 4: signed codes in [-7, 7], scale amax / 7, codes = the
// nearest integer (ties to even) of x * (7 / amax) in fp32, two per byte, element 2j in the low
// nibble of byte j.  The codes take d * BITS / 8 bytes.
template <int BITS, int PER>
__device__ void quantize_row(const __half* __restrict__ x, uint8_t* __restrict__ codes, float* __restrict__ scale) {
  constexpr float kMax = BITS == 8 ? 448.f : 7.f;
  const int lane = threadIdx.x & 31;
  float v[PER];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    v[i] = __half2float(x[lane * PER + i]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint32_t packed = 0;
  if (amax > 0.f) {
    const float inv = kMax / amax;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if constexpr (BITS == 8) {
        packed |= (uint32_t)__nv_cvt_float_to_fp8(v[i] * inv, __NV_SATFINITE, __NV_E4M3) << (8 * i);
      } else {
        const int c = min(7, max(-7, __float2int_rn(v[i] * inv)));
        packed |= (uint32_t)(c & 0xF) << (4 * i);
      }
    }
  }
  constexpr int kBytes = PER * BITS / 8;  // per lane: 4 or 2 (fp8), 2 or 1 (int4)
  if constexpr (kBytes == 4) reinterpret_cast<uint32_t*>(codes)[lane] = packed;
  else if constexpr (kBytes == 2) reinterpret_cast<uint16_t*>(codes)[lane] = (uint16_t)packed;
  else codes[lane] = (uint8_t)packed;
  if (lane == 0) *scale = amax > 0.f ? amax / kMax : 0.f;
}

// Pool write of a quantized pool: rows [rows][d] fp16 (device-accessible) -> code records (K,
// then V codes) in the pinned pool and the two scales of each row in device memory.
template <int BITS, int PER>
__global__ void k_quantize_rows(const __half* __restrict__ K, const __half* __restrict__ V, size_t rows,
                                uint8_t* __restrict__ R, int rec, float* __restrict__ S) {
  constexpr int D = 32 * PER, CB = D * BITS / 8;
  const size_t r = (size_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  uint8_t* rr = R + r * rec;
  quantize_row<BITS, PER>(K + r * D, rr, S + 2 * r);
  quantize_row<BITS, PER>(V + r * D, rr + CB, S + 2 * r + 1);
}

// Append into a quantized pool: one warp per (b, h) quantizes the current token's key and value
// into its record.
template <int BITS, int PER>
__global__ void k6_append_q(uint8_t* __restrict__ R, int rec, float* __restrict__ S, int units, int cap, int H,
                            const int32_t* __restrict__ slot, const __half* __restrict__ k_new,
                            const __half* __restrict__ v_new, int* err) {
  constexpr int D = 32 * PER, CB = D * BITS / 8;
  const int bh = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (bh >= units) return;
  const int sl = slot[bh / H];
  if (sl < 0) return;
  if (sl >= cap) {
    if ((threadIdx.x & 31) == 0) raise_error(err, IG_DEVERR_INDEX);
    return;
  }
  const size_t row = (size_t)bh * cap + sl;
  uint8_t* rr = R + row * rec;
  quantize_row<BITS, PER>(k_new + (size_t)bh * D, rr, S + 2 * row);
  quantize_row<BITS, PER>(v_new + (size_t)bh * D, rr + CB, S + 2 * row + 1);
}

// Appends of every layer's current token in one launch (grid: (b, h) x layer), run once the
// step's fetches are done: layer 0 to the dense rows when given, other layers to the pool
// (BITS = 0: fp16 rows by 16-byte copies; BITS = 8 or 4: quantized rows, the first two warps),
// and each layer's chosen columns to its partial key cache.
constexpr int kMaxAppendLayers = 128;
struct AppendLayers {
  __half* Kpart[kMaxAppendLayers];
  const int32_t* cols[kMaxAppendLayers];
  int k[kMaxAppendLayers];
};

template <int BITS, int PER>
__global__ void __launch_bounds__(64) k6_append_layers(
    const AppendLayers P, uint4* __restrict__ Kp, uint4* __restrict__ Vp, uint8_t* __restrict__ R, int rec,
    float* __restrict__ S, int cap, int H, int d, int Lcap,
    int units, const int32_t* __restrict__ slot, const __half* __restrict__ k_new,
    const __half* __restrict__ v_new, uint4* __restrict__ Kd, uint4* __restrict__ Vd, int* err) {
  const int bh = blockIdx.x, l = blockIdx.y, b = bh / H, h = bh % H;
  const int sl = slot[l * (units / H) + b];
  if (sl < 0) return;
  const __half* kn = k_new + ((size_t)l * units + bh) * d;
  const __half* vn = v_new + ((size_t)l * units + bh) * d;
  const int vpr = d / 8;
  if (l == 0 && Kd) {
    if (sl >= Lcap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      return;
    }
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
      Kd[((size_t)bh * Lcap + sl) * vpr + v] = reinterpret_cast<const uint4*>(kn)[v];
      Vd[((size_t)bh * Lcap + sl) * vpr + v] = reinterpret_cast<const uint4*>(vn)[v];
    }
  } else {
    if (sl >= cap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      return;
    }
    const size_t row = ((size_t)l * units + bh) * cap + sl;
    if constexpr (BITS == 0) {
      for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
        Kp[row * vpr + v] = reinterpret_cast<const uint4*>(kn)[v];
        Vp[row * vpr + v] = reinterpret_cast<const uint4*>(vn)[v];
      }
    } else {
      constexpr int CB = 32 * PER * BITS / 8;
      uint8_t* rr = R + row * rec;
      if (threadIdx.x < 32) quantize_row<BITS, PER>(kn, rr, S + 2 * row);
      else quantize_row<BITS, PER>(vn, rr + CB, S + 2 * row + 1);
    }
  }
  __half* kp = P.Kpart[l];
  if (kp) {
    if (sl >= Lcap) {
      if (threadIdx.x == 0) raise_error(err, IG_DEVERR_INDEX);
      return;
    }
    const int k = P.k[l];
    const int32_t* cl = P.cols[l];
    for (int c = threadIdx.x; c < k; c += blockDim.x) {
      const int col = cl[h * k + c];
      if (col < 0 || col >= d) {
        raise_error(err, IG_DEVERR_INDEX);
        continue;
      }
      kp[((size_t)bh * k + c) * Lcap + sl] = kn[col];
    }
  }
}

}  // namespace
}  // namespace ig

using namespace ig;

extern "C" ig_status ig_pool_create_ex(int layers, int B, int H, int d, int cap, int policy,
                                        int flags, ig_pool** out) {
  IG_REQUIRE(out, "null out");
  *out = nullptr;
  IG_REQUIRE(policy == IG_POOL_COUNTER || policy == IG_POOL_FIFO || policy == IG_POOL_LRU,
             "unknown pool policy %d", policy);
  IG_REQUIRE((flags & ~(IG_POOL_NO_STORAGE | IG_POOL_FP8 | IG_POOL_INT4)) == 0, "unknown pool flags 0x%x", flags);
  IG_REQUIRE(!((flags & IG_POOL_FP8) && (flags & IG_POOL_INT4)), "IG_POOL_FP8 and IG_POOL_INT4 exclude each other");
  const bool storage = !(flags & IG_POOL_NO_STORAGE);
  const int qbits = !storage ? 0 : (flags & IG_POOL_FP8) ? 8 : (flags & IG_POOL_INT4) ? 4 : 0;
  IG_REQUIRE(!qbits || d == 64 || d == 128, "a quantized pool needs d = 64 or 128");
  IG_REQUIRE(layers > 0 && B > 0 && cap > 0, "pool sizes must be positive");
  IG_REQUIRE(!storage || (H > 0 && d > 0), "a pool with storage needs H, d > 0");
  IG_REQUIRE(!storage || d % 8 == 0, "d must be a multiple of 8 (16-byte rows)");
  if (fault_injected("pool_alloc")) return fail(IG_ERR_OOM, "injected pinned-allocation failure");
  ig_pool* p = new (std::nothrow) ig_pool();
  if (!p) return fail(IG_ERR_OOM, "host allocation of the pool header failed");
  p->layers = layers;
  p->B = B;
  p->H = storage ? H : 0;
  p->d = storage ? d : 0;
  p->cap = cap;
  p->policy = policy;
  p->storage = storage;
  if (storage) {
    const size_t elems = (size_t)layers * B * H * cap * d;
    const size_t nrows = (size_t)layers * B * H * cap;
    const unsigned hflags = cudaHostAllocMapped | cudaHostAllocPortable;
    // with mapped pinned memory on this platform the host address is also the device address;
    // it is still obtained through cudaHostGetDevicePointer below for the fp16 rows
    auto alloc = [&](void** p, size_t bytes) { return cudaHostAlloc(p, bytes, hflags); };
    cudaError_t e;
    if (qbits) {
      p->qbits = qbits;
      p->rec = 2 * (d * qbits / 8);
      e = alloc(reinterpret_cast<void**>(&p->R), nrows * (size_t)p->rec);
      if (e != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return fail(IG_ERR_OOM, "pinned allocation of the quantized pool (%zu bytes) failed: %s", nrows * (size_t)p->rec,
                    cudaGetErrorString(e));
      }
      // the scales stay in device memory, so that the link carries whole lines of codes only
      e = cudaGetDevice(&p->sdev);
      if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->S), nrows * 2 * sizeof(float));
      if (e == cudaSuccess) e = cudaMemset(p->S, 0, nrows * 2 * sizeof(float));
      if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(p->R);
        if (p->S) cudaFree(p->S);
        delete p;
        return fail(IG_ERR_OOM, "device allocation of the quantized pool's scales (%zu bytes) failed: %s",
                    nrows * 2 * sizeof(float), cudaGetErrorString(e));
      }
    } else {
      e = alloc(reinterpret_cast<void**>(&p->K), elems * 2);
      if (e == cudaSuccess) e = alloc(reinterpret_cast<void**>(&p->V), elems * 2);
      if (e != cudaSuccess) {
        cudaGetLastError();
        if (p->K) cudaFreeHost(p->K);
        delete p;
        return fail(IG_ERR_OOM, "pinned allocation of 2 x %zu bytes failed: %s", elems * 2,
                    cudaGetErrorString(e));
      }
      void* kd = nullptr;
      void* vd = nullptr;
      e = cudaHostGetDevicePointer(&kd, p->K, 0);
      if (e == cudaSuccess) e = cudaHostGetDevicePointer(&vd, p->V, 0);
      if (e != cudaSuccess) {
        cudaFreeHost(p->K);
        cudaFreeHost(p->V);
        delete p;
        return cuda_fail(e, "device pointer of the pinned pool");
      }
      p->Kdev = static_cast<uint16_t*>(kd);
      p->Vdev = static_cast<uint16_t*>(vd);
    }
  }
  try {
    const size_t npb = (size_t)layers * B;
    p->counter.assign(npb * cap, 0);
    p->seq.assign(npb * cap, 0);
    p->filled.assign(npb, 0);
    p->next_seq.assign(npb, 0);
    p->last_use.assign(npb * cap, 0);
    p->clock.assign(npb, 0);
    p->evictions.assign(npb, 0);
  } catch (...) {
    for (void* q : {(void*)p->K, (void*)p->V, (void*)p->R})
      if (q) cudaFreeHost(q);
    if (p->S) cudaFree(p->S);
    delete p;
    return fail(IG_ERR_OOM, "host allocation of the pool manager failed");
  }
  *out = p;
  return IG_OK;
}

extern "C" ig_status ig_pool_create(int layers, int B, int H, int d, int cap, ig_pool** out) {
  return ig_pool_create_ex(layers, B, H, d, cap, IG_POOL_COUNTER, 0, out);
}

extern "C" ig_status ig_pool_destroy(ig_pool* pool) {
  if (!pool) return IG_OK;
  cudaError_t first = cudaSuccess;
  for (void* q : {(void*)pool->K, (void*)pool->V, (void*)pool->R}) {
    if (!q) continue;
    const cudaError_t e = cudaFreeHost(q);
    if (first == cudaSuccess) first = e;
  }
  if (pool->S) {
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e == cudaSuccess && cur != pool->sdev) e = cudaSetDevice(pool->sdev);
    if (e == cudaSuccess) e = cudaFree(pool->S);
    if (cur != pool->sdev) cudaSetDevice(cur);
    if (first == cudaSuccess) first = e;
  }
  delete pool;
  if (first != cudaSuccess) return cuda_fail(first, "free pool memory");
  return IG_OK;
}

extern "C" ig_status ig_pool_kv(const ig_pool* pool, int layer, uint16_t** K, uint16_t** V) {
  IG_REQUIRE(pool && K && V, "null argument");
  IG_REQUIRE(pool->storage, "the pool was created without storage");
  IG_REQUIRE(!pool->qbits, "a quantized pool has no fp16 rows (use ig_pool_kv8)");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  const size_t le = (size_t)pool->B * pool->H * pool->cap * pool->d;
  *K = pool->K + (size_t)layer * le;
  *V = pool->V + (size_t)layer * le;
  return IG_OK;
}

extern "C" ig_status ig_pool_kv8(const ig_pool* pool, int layer, uint8_t** records, int* record_bytes,
                                  float** scales) {
  IG_REQUIRE(pool && records && record_bytes, "null argument");
  IG_REQUIRE(pool->qbits, "not a quantized pool");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  const size_t rows = (size_t)pool->B * pool->H * pool->cap;
  *records = pool->R + (size_t)layer * rows * pool->rec;
  *record_bytes = pool->rec;
  if (scales) *scales = pool->S + (size_t)layer * rows * 2;
  return IG_OK;
}

extern "C" ig_status ig_pool_read_scales(const ig_pool* pool, int layer, float* out) {
  IG_REQUIRE(pool && out, "null argument");
  IG_REQUIRE(pool->qbits, "not a quantized pool");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  const size_t rows = (size_t)pool->B * pool->H * pool->cap;
  cudaError_t e = cudaMemcpy(out, pool->S + (size_t)layer * rows * 2, rows * 2 * sizeof(float), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read the pool's scales");
  return IG_OK;
}

namespace ig {
// A quantized pool's scales live on one device: its kernels must run there.
ig_status check_pool_device(const ig_pool* pool) {
  if (!pool || !pool->qbits) return IG_OK;
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "current device");
  IG_REQUIRE(cur == pool->sdev, "the quantized pool's scales are on device %d, the current device is %d", pool->sdev,
             cur);
  return IG_OK;
}
}  // namespace ig

extern "C" ig_status ig_pool_write(ig_pool* pool, void* stream, int layer, const uint16_t* K,
                                   const uint16_t* V) {
  IG_REQUIRE(pool && K && V, "null argument");
  if (ig_status dst = check_pool_device(pool); dst != IG_OK) return dst;
  IG_REQUIRE(pool->storage, "the pool was created without storage");
  IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
  const size_t le = (size_t)pool->B * pool->H * pool->cap * pool->d;
  cudaStream_t s = as_stream(stream);
  if (pool->qbits) {
    // the rows are quantized by a kernel, so they must be readable by the device
    for (const void* src : {(const void*)K, (const void*)V}) {
      cudaPointerAttributes at{};
      const cudaError_t e = cudaPointerGetAttributes(&at, src);
      if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered) {
        cudaGetLastError();
        return fail(IG_ERR_INVALID, "writing a quantized pool needs device or pinned source rows");
      }
    }
    const size_t rows = (size_t)pool->B * pool->H * pool->cap;
    const size_t r0 = (size_t)layer * rows;
    const int wpb = 8;  // rows (warps) per block
    const unsigned blocks = (unsigned)((rows + wpb - 1) / wpb);
    auto Kh = reinterpret_cast<const __half*>(K);
    auto Vh = reinterpret_cast<const __half*>(V);
    uint8_t* R0 = pool->R + r0 * pool->rec;
    float* S0 = pool->S + r0 * 2;
    const bool d128 = pool->d == 128;
    if (pool->qbits == 8) {
      if (d128) k_quantize_rows<8, 4><<<blocks, 32 * wpb, 0, s>>>(Kh, Vh, rows, R0, pool->rec, S0);
      else k_quantize_rows<8, 2><<<blocks, 32 * wpb, 0, s>>>(Kh, Vh, rows, R0, pool->rec, S0);
    } else {
      if (d128) k_quantize_rows<4, 4><<<blocks, 32 * wpb, 0, s>>>(Kh, Vh, rows, R0, pool->rec, S0);
      else k_quantize_rows<4, 2><<<blocks, 32 * wpb, 0, s>>>(Kh, Vh, rows, R0, pool->rec, S0);
    }
    IG_CHECK_LAUNCH("quantized pool write launch");
    return IG_OK;
  }
  cudaError_t e = cudaMemcpyAsync(pool->K + (size_t)layer * le, K, le * 2, cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(pool->V + (size_t)layer * le, V, le * 2, cudaMemcpyDefault, s);
  if (e != cudaSuccess) return cuda_fail(e, "pool write");
  return IG_OK;
}

extern "C" ig_status ig_append_kv(void* stream, ig_pool* pool, int layer, int B, int H, int d,
                                  int k, int Lcap, const int32_t* slot, const int32_t* cols,
                                  const uint16_t* k_new, const uint16_t* v_new, uint16_t* Kpart,
                                  uint16_t* Kdense, uint16_t* Vdense) {
  IG_REQUIRE(B > 0 && H > 0 && d > 0 && d % 8 == 0 && Lcap > 0, "bad sizes");
  IG_REQUIRE(slot && k_new && v_new, "null slot, k_new or v_new");
  IG_REQUIRE(!Kpart || (cols && k > 0 && k <= d), "Kpart needs cols and 0 < k <= d");
  IG_REQUIRE((Kdense == nullptr) == (Vdense == nullptr), "Kdense and Vdense go together");
  IG_REQUIRE(aligned(k_new, 16) && aligned(v_new, 16), "k_new, v_new must be 16-byte aligned");
  IG_REQUIRE(!Kdense || (aligned(Kdense, 16) && aligned(Vdense, 16)), "dense KV must be 16-byte aligned");
  uint4* Kp = nullptr;
  uint4* Vp = nullptr;
  int cap = 0;
  if (pool) {
    IG_REQUIRE(pool->storage, "the pool was created without storage");
    IG_REQUIRE(layer >= 0 && layer < pool->layers, "layer %d out of range", layer);
    IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
    if (ig_status dst = check_pool_device(pool); dst != IG_OK) return dst;
    if (pool->qbits) {  // the quantized row goes to the pool here; the kernel below does the rest
      const size_t rows = (size_t)B * H * pool->cap, r0 = (size_t)layer * rows;
      const int units = B * H, wpb = 8;
      auto kn = reinterpret_cast<const __half*>(k_new);
      auto vn = reinterpret_cast<const __half*>(v_new);
      uint8_t* R0 = pool->R + r0 * pool->rec;
      float* S0 = pool->S + r0 * 2;
      const unsigned g = (unsigned)((units + wpb - 1) / wpb);
      cudaStream_t s = as_stream(stream);
      int* err = error_word();
      if (pool->qbits == 8) {
        if (d == 128) k6_append_q<8, 4><<<g, 32 * wpb, 0, s>>>(R0, pool->rec, S0, units, pool->cap, H, slot, kn, vn, err);
        else k6_append_q<8, 2><<<g, 32 * wpb, 0, s>>>(R0, pool->rec, S0, units, pool->cap, H, slot, kn, vn, err);
      } else {
        if (d == 128) k6_append_q<4, 4><<<g, 32 * wpb, 0, s>>>(R0, pool->rec, S0, units, pool->cap, H, slot, kn, vn, err);
        else k6_append_q<4, 2><<<g, 32 * wpb, 0, s>>>(R0, pool->rec, S0, units, pool->cap, H, slot, kn, vn, err);
      }
      IG_CHECK_LAUNCH("quantized append launch");
      if (!Kpart && !Kdense) return IG_OK;
    } else {
      const size_t le = (size_t)B * H * pool->cap * d;
      Kp = reinterpret_cast<uint4*>(pool->Kdev + (size_t)layer * le);
      Vp = reinterpret_cast<uint4*>(pool->Vdev + (size_t)layer * le);
      cap = pool->cap;
    }
  }
  k6_append<<<B * H, 64, 0, as_stream(stream)>>>(
      Kp, Vp, cap, H, d, k, Lcap, slot, cols, reinterpret_cast<const __half*>(k_new),
      reinterpret_cast<const __half*>(v_new), reinterpret_cast<__half*>(Kpart),
      reinterpret_cast<uint4*>(Kdense), reinterpret_cast<uint4*>(Vdense), error_word());
  IG_CHECK_LAUNCH("append launch");
  return IG_OK;
}

extern "C" ig_status ig_append_kv_layers(void* stream, ig_pool* pool, int layers, int B, int H, int d,
                                         const int* ks, int Lcap, const int32_t* slot,
                                         const int32_t* const* cols, const uint16_t* k_new,
                                         const uint16_t* v_new, uint16_t* const* Kpart, uint16_t* Kdense,
                                         uint16_t* Vdense) {
  IG_REQUIRE(pool && pool->storage, "a pool with storage is needed");
  IG_REQUIRE(layers >= 1 && layers <= pool->layers && layers <= kMaxAppendLayers, "bad layer count %d", layers);
  IG_REQUIRE(B == pool->B && H == pool->H && d == pool->d, "B/H/d do not match the pool");
  if (ig_status dst = check_pool_device(pool); dst != IG_OK) return dst;
  IG_REQUIRE(Lcap > 0 && slot && k_new && v_new, "bad Lcap or null pointer");
  IG_REQUIRE((Kdense == nullptr) == (Vdense == nullptr), "Kdense and Vdense go together");
  IG_REQUIRE(aligned(k_new, 16) && aligned(v_new, 16), "k_new, v_new must be 16-byte aligned");
  IG_REQUIRE(!Kdense || (aligned(Kdense, 16) && aligned(Vdense, 16)), "dense rows must be 16-byte aligned");
  AppendLayers P{};
  for (int l = 0; l < layers; ++l) {
    P.Kpart[l] = Kpart ? reinterpret_cast<__half*>(Kpart[l]) : nullptr;
    P.cols[l] = cols ? cols[l] : nullptr;
    P.k[l] = ks ? ks[l] : 0;
    IG_REQUIRE(!P.Kpart[l] || (P.cols[l] && P.k[l] > 0 && P.k[l] <= d), "layer %d: Kpart needs cols and 0 < k <= d", l);
  }
  const int units = B * H;
  dim3 grid(units, layers);
  cudaStream_t st = as_stream(stream);
  auto kn = reinterpret_cast<const __half*>(k_new);
  auto vn = reinterpret_cast<const __half*>(v_new);
  auto Kd = reinterpret_cast<uint4*>(Kdense);
  auto Vd = reinterpret_cast<uint4*>(Vdense);
  int* err = error_word();
  if (!pool->qbits) {
    k6_append_layers<0, 1><<<grid, 64, 0, st>>>(P, reinterpret_cast<uint4*>(pool->Kdev),
                                               reinterpret_cast<uint4*>(pool->Vdev), nullptr, 0, nullptr, pool->cap, H, d,
                                               Lcap,
                                               units, slot, kn, vn, Kd, Vd, err);
  } else if (pool->qbits == 8) {
    if (d == 128)
      k6_append_layers<8, 4><<<grid, 64, 0, st>>>(P, nullptr, nullptr, pool->R, pool->rec, pool->S, pool->cap, H, d, Lcap, units,
                                                 slot, kn, vn, Kd, Vd, err);
    else
      k6_append_layers<8, 2><<<grid, 64, 0, st>>>(P, nullptr, nullptr, pool->R, pool->rec, pool->S, pool->cap, H, d, Lcap, units,
                                                 slot, kn, vn, Kd, Vd, err);
  } else {
    if (d == 128)
      k6_append_layers<4, 4><<<grid, 64, 0, st>>>(P, nullptr, nullptr, pool->R, pool->rec, pool->S, pool->cap, H, d, Lcap, units,
                                                 slot, kn, vn, Kd, Vd, err);
    else
      k6_append_layers<4, 2><<<grid, 64, 0, st>>>(P, nullptr, nullptr, pool->R, pool->rec, pool->S, pool->cap, H, d, Lcap, units,
                                                 slot, kn, vn, Kd, Vd, err);
  }
  IG_CHECK_LAUNCH("batched append launch");
  return IG_OK;
}
