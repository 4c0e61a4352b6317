// Spatial split of one GPU between the fetch stream and the compute stream (green contexts).
//
// The decode step runs two streams at once: the host-link fetch of the selected rows and the
// HBM-bound speculation and attention.  Sharing every SM, the fetch's CTAs (whose loads wait
// microseconds on the host link) sit beside compute CTAs, and the compute kernels, which split
// their work evenly over their CTAs, finish only when the CTAs on those SMs do.  Two green
// contexts over disjoint SM sets keep the two apart.  The driver entry points come through the
// runtime (cudaGetDriverEntryPointByVersion), so the library does not link the driver itself.
#include <cuda.h>

#include <mutex>

#include "ig_common.cuh"

using namespace ig;

namespace {

typedef CUresult (*PFN_DeviceGet)(CUdevice*, int);
typedef CUresult (*PFN_DeviceGetDevResource)(CUdevice, CUdevResource*, CUdevResourceType);
typedef CUresult (*PFN_SmSplit)(CUdevResource*, unsigned int*, const CUdevResource*, CUdevResource*, unsigned int,
                                unsigned int);
typedef CUresult (*PFN_GenerateDesc)(CUdevResourceDesc*, CUdevResource*, unsigned int);
typedef CUresult (*PFN_GreenCtxCreate)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned int);
typedef CUresult (*PFN_GreenCtxDestroy)(CUgreenCtx);
typedef CUresult (*PFN_GreenCtxStreamCreate)(CUstream*, CUgreenCtx, unsigned int, int);
typedef CUresult (*PFN_StreamDestroy)(CUstream);

struct Driver {
  PFN_DeviceGet device_get = nullptr;
  PFN_DeviceGetDevResource get_resource = nullptr;
  PFN_SmSplit split = nullptr;
  PFN_GenerateDesc gen_desc = nullptr;
  PFN_GreenCtxCreate ctx_create = nullptr;
  PFN_GreenCtxDestroy ctx_destroy = nullptr;
  PFN_GreenCtxStreamCreate stream_create = nullptr;
  PFN_StreamDestroy stream_destroy = nullptr;
  bool ok = false;
};

std::mutex g_drv_mu;
Driver g_drv;
bool g_drv_tried = false;

const char* g_missing = "";

// the entry point of the ABI version this file was compiled against (the header's)
template <class F>
bool entry(const char* name, F* fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &p, CUDA_VERSION, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p) {
    g_missing = name;
    return false;
  }
  *fn = reinterpret_cast<F>(p);
  return true;
}

const Driver& driver() {
  std::lock_guard<std::mutex> lk(g_drv_mu);
  if (!g_drv_tried) {
    g_drv_tried = true;
    Driver d;
    d.ok = entry("cuDeviceGet", &d.device_get) && entry("cuDeviceGetDevResource", &d.get_resource) &&
           entry("cuDevSmResourceSplitByCount", &d.split) && entry("cuDevResourceGenerateDesc", &d.gen_desc) &&
           entry("cuGreenCtxCreate", &d.ctx_create) && entry("cuGreenCtxDestroy", &d.ctx_destroy) &&
           entry("cuGreenCtxStreamCreate", &d.stream_create) && entry("cuStreamDestroy", &d.stream_destroy);
    g_drv = d;
  }
  return g_drv;
}

ig_status cu_fail(CUresult r, const char* what) {
  return fail(IG_ERR_CUDA, "%s: driver error %d", what, (int)r);
}

}  // namespace

struct ig_sm_split {
  CUgreenCtx ctx[2] = {nullptr, nullptr};  // [0] compute, [1] fetch
  CUstream stream[2] = {nullptr, nullptr};
  int sms[2] = {0, 0};
};

extern "C" ig_status ig_sm_split_destroy(ig_sm_split* sp) {
  if (!sp) return IG_OK;
  const Driver& d = driver();
  for (int i = 0; i < 2; ++i) {
    if (sp->stream[i]) {
      unregister_stream_sms(reinterpret_cast<cudaStream_t>(sp->stream[i]));
      if (d.ok) d.stream_destroy(sp->stream[i]);
    }
    if (sp->ctx[i] && d.ok) d.ctx_destroy(sp->ctx[i]);
  }
  delete sp;
  return IG_OK;
}

extern "C" ig_status ig_sm_split_create(int device, int fetch_sms, ig_sm_split** out, void** compute_stream,
                                        void** fetch_stream, int* compute_sms, int* fetch_sms_out) {
  IG_REQUIRE(out && compute_stream && fetch_stream, "null argument");
  *out = nullptr;
  IG_REQUIRE(fetch_sms > 0, "fetch_sms must be positive");
  cudaError_t e = cudaSetDevice(device);
  if (e == cudaSuccess) e = cudaFree(nullptr);  // the primary context exists from here on
  if (e != cudaSuccess) return cuda_fail(e, "sm split: device");
  const Driver& d = driver();
  if (!d.ok) return fail(IG_ERR_CUDA, "sm split: the driver does not provide %s", g_missing);
  CUdevice dev;
  CUresult r = d.device_get(&dev, device);
  if (r != CUDA_SUCCESS) return cu_fail(r, "cuDeviceGet");
  CUdevResource all{}, part{}, rest{};
  r = d.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM);
  if (r != CUDA_SUCCESS) return cu_fail(r, "cuDeviceGetDevResource");
  IG_REQUIRE((unsigned)fetch_sms < all.sm.smCount, "fetch_sms %d leaves no SM for the compute stream (%u SMs)",
             fetch_sms, all.sm.smCount);
  unsigned int groups = 1;
  r = d.split(&part, &groups, &all, &rest, 0, (unsigned)fetch_sms);
  if (r != CUDA_SUCCESS) return cu_fail(r, "cuDevSmResourceSplitByCount");
  if (groups != 1 || rest.sm.smCount == 0)
    return fail(IG_ERR_INVALID, "sm split: %d SMs for the fetch stream leave no compute partition", fetch_sms);
  ig_sm_split* sp = new ig_sm_split;
  CUdevResource* res[2] = {&rest, &part};
  int lo = 0, hi = 0;
  e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
  if (e != cudaSuccess) {
    delete sp;
    return cuda_fail(e, "stream priority range");
  }
  for (int i = 0; i < 2; ++i) {
    CUdevResourceDesc desc;
    r = d.gen_desc(&desc, res[i], 1);
    if (r == CUDA_SUCCESS) r = d.ctx_create(&sp->ctx[i], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM);
    // the fetch stream at the highest priority, as without the split
    if (r == CUDA_SUCCESS) r = d.stream_create(&sp->stream[i], sp->ctx[i], CU_STREAM_NON_BLOCKING, i == 1 ? hi : 0);
    if (r != CUDA_SUCCESS) {
      ig_sm_split_destroy(sp);
      return cu_fail(r, "green context");
    }
    sp->sms[i] = (int)res[i]->sm.smCount;
    register_stream_sms(reinterpret_cast<cudaStream_t>(sp->stream[i]), sp->sms[i]);
  }
  *compute_stream = sp->stream[0];
  *fetch_stream = sp->stream[1];
  if (compute_sms) *compute_sms = sp->sms[0];
  if (fetch_sms_out) *fetch_sms_out = sp->sms[1];
  *out = sp;
  return IG_OK;
}
