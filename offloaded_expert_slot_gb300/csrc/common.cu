// Host-side helpers: last-error message, SM count, tensor-map encoding.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace oes {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return OES_ERR_CUDA;
}

int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Kernel attributes are set once per (device, kernel); calls from several
// host threads are serialised by a mutex.
namespace {
std::mutex g_attr_mu;
std::map<std::pair<int, const void*>, size_t> g_smem_set;     // largest dynamic size set
std::map<std::pair<int, const void*>, bool> g_carveout_set;
}  // namespace

int set_max_dynamic_smem(const void* func, size_t bytes, const char* name) {
  int dev = 0;
  OES_TRY_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_attr_mu);
  size_t& have = g_smem_set[{dev, func}];
  if (bytes <= have) return OES_OK;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return cuda_fail(e, name);
  have = bytes;
  return OES_OK;
}

int prefer_max_shared_carveout(const void* func, const char* name) {
  int dev = 0;
  OES_TRY_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_attr_mu);
  bool& done = g_carveout_set[{dev, func}];
  if (done) return OES_OK;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e, name);
  done = true;
  return OES_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  // the encoder is a driver call and needs a current context; a thread whose
  // first CUDA call this is has none yet, so bind the current device's
  // primary context once per thread
  static thread_local bool bound = false;
  if (!bound) {
    int dev = 0;
    OES_TRY_CUDA(cudaGetDevice(&dev));
    OES_TRY_CUDA(cudaSetDevice(dev));
    bound = true;
  }
  auto fn = get_encode();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return OES_ERR_CUDA;
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d, rank %d, dims %llu x %llu x %llu)",
              (int)r, rank, (unsigned long long)dims[0],
              (unsigned long long)(rank > 1 ? dims[1] : 1),
              (unsigned long long)(rank > 2 ? dims[2] : 1));
    return OES_ERR_CUDA;
  }
  return OES_OK;
}

}  // namespace oes

extern "C" const char* oes_last_error(void) { return oes::g_err; }
