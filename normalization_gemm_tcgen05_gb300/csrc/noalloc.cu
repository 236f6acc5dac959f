// noalloc.cu — the fixed workspace of fnorm_gemm_postnorm_noalloc: the
// grid-exchange statistics of wide post-norm rows in a file-scope device
// array, so that entry point allocates nothing.  Its address is taken once
// per device; its counters are cleared by that first call (a failed set-up
// is retried by the next call).
#include <mutex>

#include "internal.h"

namespace fnorm {

namespace {
constexpr int kNoAllocUnits = 2048;       // (row block, 256-column tile) units: 2 MB of statistics
constexpr int kNoAllocRowBlocks = 8192;   // 128-row blocks: M up to 2^20
constexpr size_t kPartBytes = static_cast<size_t>(kNoAllocUnits) * 128 * sizeof(float2);
constexpr size_t kCntBytes = static_cast<size_t>(kNoAllocRowBlocks) * sizeof(unsigned long long);
constexpr size_t kNoAllocBytes = kPartBytes + kCntBytes + 256;
constexpr int kMaxDev = 64;

struct Slot {
  std::once_flag once;
  GxScratch gx{};
};
Slot g_slot[kMaxDev];
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {
struct SetupError {
  fnorm_status_t status;
};
}  // namespace

fnorm_status_t noalloc_scratch(cudaStream_t stream, const GxScratch** out) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);  // the device is current from here on
  if (st != FNORM_OK) return st;
  if (dev.id >= kMaxDev) {
    set_error("device ordinal %d out of range", dev.id);
    return FNORM_ERR_UNSUPPORTED;
  }
  Slot& s = g_slot[dev.id];
  try {
    // A set-up that fails throws out of call_once, which leaves the flag
    // unset: the next call on this device tries again instead of finding the
    // entry point disabled for the rest of the process.
    std::call_once(s.once, [&] {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) throw SetupError{cuda_fail(e, "cudaGetSymbolAddress(no-alloc workspace)")};
      char* base = static_cast<char*>(p);
      // counters and finish count start at zero (ordered before this call's
      // kernel on its stream); every call leaves them zero
      e = cudaMemsetAsync(base + kPartBytes, 0, kCntBytes + 256, stream);
      if (e != cudaSuccess) throw SetupError{cuda_fail(e, "clearing the no-alloc workspace")};
      s.gx.part = reinterpret_cast<float2*>(base);
      s.gx.cnt = reinterpret_cast<unsigned long long*>(base + kPartBytes);
      s.gx.finish = reinterpret_cast<uint32_t*>(base + kPartBytes + kCntBytes);
      s.gx.units_cap = kNoAllocUnits;
      s.gx.rowblocks_cap = kNoAllocRowBlocks;
    });
  } catch (const SetupError& err) {
    return err.status;
  }
  *out = &s.gx;
  return FNORM_OK;
}

}  // namespace fnorm
