// runtime.cu — host runtime of libfnorm: error strings, per-device cache,
// the device status word, tensor-map encoding and the wait-timeout self test.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace fnorm {

// Written by kernels that give up on a bounded wait; read and cleared by
// fnorm_check_status.  One copy per device (module-scope device variable).
__device__ uint32_t g_status_word;

namespace {
thread_local std::string t_error;

constexpr int kMaxDevices = 64;
struct DevSlot {
  std::once_flag once;
  fnorm_status_t init_status = FNORM_OK;
  int num_sms = 0;
  uint32_t* status = nullptr;
};
DevSlot g_dev[kMaxDevices];

std::atomic<uint64_t> g_wait_limit{2000000000ull};
}  // namespace

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_error = buf;
}

fnorm_status_t cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return FNORM_ERR_CUDA;
}

const char* last_error_cstr() { return t_error.c_str(); }
void clear_error() { t_error.clear(); }

fnorm_status_t current_device(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return FNORM_ERR_UNSUPPORTED;
  }
  DevSlot& s = g_dev[dev];
  std::call_once(s.once, [&] {
    int major = 0, minor = 0;
    cudaError_t e2 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e2 == cudaSuccess) e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e2 == cudaSuccess) e2 = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e2 != cudaSuccess) {
      s.init_status = cuda_fail(e2, "cudaDeviceGetAttribute");
      return;
    }
    if (major != 10 || minor != 3) {
      set_error("libfnorm is built for sm_103a (GB300); device %d is sm_%d%d", dev, major, minor);
      s.init_status = FNORM_ERR_UNSUPPORTED;
      return;
    }
    void* p = nullptr;
    e2 = cudaGetSymbolAddress(&p, g_status_word);
    if (e2 != cudaSuccess) {
      s.init_status = cuda_fail(e2, "cudaGetSymbolAddress(status word)");
      return;
    }
    s.status = static_cast<uint32_t*>(p);
  });
  if (s.init_status != FNORM_OK) {
    set_error("device %d unusable (first-use initialisation failed)", dev);
    return s.init_status;
  }
  out->id = dev;
  out->num_sms = s.num_sms;
  out->status = s.status;
  return FNORM_OK;
}

// Layout of a caller's grid-exchange workspace, the same for every call that
// uses it whatever its shape (so the counters are always where the last
// call left them, zeroed): 256 bytes holding the finish count (offset 0),
// then kGxMaxRowBlocks per-row-block arrival counters, then the per-tile row
// statistics [row blocks][tiles per row][128] float2 of the call.
size_t gx_workspace_bytes(int64_t M, int64_t N) {
  const int64_t rb = (M + 127) / 128, tiles = (N + 255) / 256;
  return kGxHeaderBytes + static_cast<size_t>(kGxMaxRowBlocks) * sizeof(uint64_t) +
         static_cast<size_t>(rb * tiles) * 128 * sizeof(float2);
}

fnorm_status_t gx_scratch_from(void* workspace, size_t bytes, int64_t M, int64_t N, GxScratch* out) {
  const size_t need = gx_workspace_bytes(M, N);
  if (workspace == nullptr || bytes < need) {
    set_error("the grid-exchange workspace of a %lld x %lld post-norm needs %zu bytes (given %zu)", (long long)M,
              (long long)N, need, workspace == nullptr ? (size_t)0 : bytes);
    return FNORM_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) {
    set_error("workspace must be 16-byte aligned");
    return FNORM_ERR_INVALID_ARG;
  }
  char* base = static_cast<char*>(workspace);
  out->finish = reinterpret_cast<uint32_t*>(base);
  out->cnt = reinterpret_cast<unsigned long long*>(base + kGxHeaderBytes);
  out->part = reinterpret_cast<float2*>(base + kGxHeaderBytes + static_cast<size_t>(kGxMaxRowBlocks) * 8);
  const size_t units = (bytes - kGxHeaderBytes - static_cast<size_t>(kGxMaxRowBlocks) * 8) / (128 * sizeof(float2));
  out->units_cap = static_cast<int>(units < 0x7fffffffu ? units : 0x7fffffffu);
  out->rowblocks_cap = kGxMaxRowBlocks;
  return FNORM_OK;
}

uint64_t wait_limit_ns() { return g_wait_limit.load(std::memory_order_relaxed); }
void set_wait_limit(uint64_t ns) { g_wait_limit.store(ns, std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("FNORM_PDL");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

bool plain_cluster_grid_exchange() {
  static const bool on = [] {
    const char* v = getenv("FNORM_PLAIN_GX_LAUNCH");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

// --------------------------------------------------------------------------
// tensor maps
// --------------------------------------------------------------------------
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

fnorm_status_t encode_tmap_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                                   uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                                   CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return FNORM_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d) for a [%llu x %llu] tensor, box %u x %u", (int)r,
              (unsigned long long)outer, (unsigned long long)inner, box_outer, box_inner);
    return FNORM_ERR_CUDA;
  }
  return FNORM_OK;
}

// --------------------------------------------------------------------------
// failure-detection self test: a bounded wait on a barrier nothing arrives on
// --------------------------------------------------------------------------
__global__ void wait_timeout_selftest_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{limit_ns, status, &abort_flag};
  if (threadIdx.x == 0) (void)mbar_wait(wc, smem_u32(&bar), 0, kSiteSelfTest);
  __syncthreads();
}

// --------------------------------------------------------------------------
// self test of the cluster-shape check: a kernel that expects clusters of two
// CTAs, launched in clusters of `cluster` CTAs; it performs no cluster
// operation of any kind, whatever the check answers
// --------------------------------------------------------------------------
__global__ void cluster_shape_selftest_kernel(uint32_t* status) {
  if (!cluster_shape_ok(2u, status)) return;
}

fnorm_status_t launch_cluster_shape_selftest(int cluster, cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(4, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cluster_shape_selftest_kernel, dev.status);
  if (e != cudaSuccess) return cuda_fail(e, "cluster_shape_selftest_kernel launch");
  return FNORM_OK;
}

fnorm_status_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(dev.status, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait_timeout_selftest_kernel launch");
  return FNORM_OK;
}

fnorm_status_t read_and_clear_status(cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, dev.status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(dev.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    if (word & kStatusClusterShape) {
      set_error("a clustered kernel ran in a cluster of another size and wrote nothing (status 0x%08x); "
                "a launch path dropped its cluster shape (profilers replay a cooperative launch of clusters "
                "without them: set FNORM_PLAIN_GX_LAUNCH=1 when profiling)", word);
      return FNORM_ERR_CUDA;
    }
    static const char* sites[] = {"?", "TMA producer", "MMA issuer", "epilogue", "norm warps",
                                  "cluster statistics exchange", "teardown drain", "self test"};
    const uint32_t site = (word >> 8) & 0xFFu;
    set_error("a kernel gave up on a bounded wait (first at: %s; status 0x%08x)",
              site < sizeof(sites) / sizeof(sites[0]) ? sites[site] : "?", word);
    return FNORM_ERR_TIMEOUT;
  }
  return FNORM_OK;
}

}  // namespace fnorm
