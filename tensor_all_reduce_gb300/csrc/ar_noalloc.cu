// Allocation-free entry point: the staged fused kernel with its scratch in a static device
// array instead of memory allocated by ar_init.
//
// Who needs it: code that must not call cudaMalloc at the point where it wants this op.
// Typical cases are an inference engine that reserves all device memory up front for
// weights, KV cache and activations (a late allocation could fail or fragment that plan),
// a caller that is inside a stream capture (allocation calls are not allowed while a
// stream is captured in the global mode), and a latency-critical loop where an allocation
// would implicitly synchronise the device.  ar_init allocates the staged kernel's status
// word with cudaMalloc, so such callers cannot create a context; this entry point needs no
// context at all.
//
// The staged kernel's only scratch is one int: the word in which a bounded wait that ran
// out records code 1.  Here that word lives in g_noalloc_scratch, a file-scope array of
// AR_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library holds until the
// process exits.  Host code cannot use the array's name as a device address, so the
// address is fetched with cudaGetSymbolAddress once per device, with that device current.
#include <mutex>
#include <stdio.h>
#include <string.h>

#include "ar.h"
#include "ar_common.cuh"
#include "ar_launch.h"
#include "ar_staged.cuh"

namespace {

constexpr int kScratchInts = AR_NOALLOC_SCRATCH_BYTES / (int)sizeof(int);
constexpr int kMaxDevices = 64;
constexpr size_t kStatusBytes = sizeof(int);  // what one call of the staged kernel needs

static __device__ __align__(256) int g_noalloc_scratch[kScratchInts];

struct DeviceSetup {
  bool ready;
  int sm_count;
  int max_dyn_smem;
  int* scratch;  // device address of g_noalloc_scratch on this device
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// One-time set-up for the current device: SM count, shared-memory opt-in of the staged
// kernels, and the device address of the static scratch array.
ar_status setup_current_device(int dev, DeviceSetup* out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return AR_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return AR_ERR_UNSUPPORTED;
    const int max_dyn = optin - 1024;
    const void* fns[256];
    const int nf = ar::staged_kernel_list(fns, 256);
    for (int i = 0; i < nf; ++i)
      if (cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
      }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      (void)cudaGetLastError();
      return AR_ERR_CUDA;
    }
    s.sm_count = sms;
    s.max_dyn_smem = max_dyn;
    s.scratch = static_cast<int*>(ptr);
    s.ready = true;
  }
  *out = s;
  return AR_OK;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

extern "C" ar_status ar_fused_reduce_rmsnorm_noalloc(const ar_fused_args* a, void* stream) {
  // Argument rules are those of ar_fused_reduce_rmsnorm, which checks them all before it
  // looks at its context: without a context a valid call answers AR_ERR_NOT_INITIALIZED.
  const ar_status v = ar_fused_reduce_rmsnorm(nullptr, a, stream);
  if (v != AR_ERR_NOT_INITIALIZED) return v;
  if (a->m == 0) return AR_OK;

  // Only the staged kernel has this form: 16-byte-aligned rows of at most 8192 elements.
  bool vec = (a->h % 8) == 0 && a->h <= 8192 && (a->ld_in % 8) == 0 && (a->ld_out % 8) == 0;
  for (int r = 0; r < a->n; ++r) vec = vec && aligned16(a->partials[r]);
  vec = vec && aligned16(a->residual_in) && aligned16(a->residual_out) && aligned16(a->weight) &&
        aligned16(a->out) && (a->quant == AR_QUANT_NONE || (reinterpret_cast<uintptr_t>(a->q_out) % 8) == 0);
  if (!vec) return AR_ERR_UNSUPPORTED;
  // Scratch needed by this call: one status word whatever the sizes, against the array's
  // fixed capacity.
  if (kStatusBytes > (size_t)AR_NOALLOC_SCRATCH_BYTES) return AR_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return AR_ERR_UNSUPPORTED;
  DeviceSetup ds;
  const ar_status st = setup_current_device(dev, &ds);
  if (st != AR_OK) return st;

  const bool quant = a->quant != AR_QUANT_NONE;
  const int es = 2;
  const int row_packs = (int)(a->h / 8);
  const int rows_per_stage = a->n + (a->residual_in ? 1 : 0);
  const int64_t stage_bytes = (int64_t)rows_per_stage * a->h * es;
  int S = 2;  // two stages: the fastest ring with every epilogue
  if (S * stage_bytes > ds.max_dyn_smem) S = 1;
  if (S * stage_bytes > ds.max_dyn_smem) return AR_ERR_UNSUPPORTED;
  const int ppt = 2;
  int block = ((row_packs + ppt - 1) / ppt + 31) / 32 * 32;
  if (block < 32) block = 32;

  ar::FusedParams p;
  ar::fill_fused_params(p, *a, row_packs, 1);
  p.prefetch = 1;
  ar::StagedParams sp = {};
  sp.stages = S;
  sp.row_bytes = (int)(a->h * es);
  sp.err = ds.scratch;
  sp.wait_cycles = 2000000000LL;

  const void* fn = a->dtype == AR_DTYPE_BF16 ? ar::staged_kernel_bf16(a->n, ppt, quant)
                                             : ar::staged_kernel_f16(a->n, ppt, quant);
  if (!fn) return AR_ERR_UNSUPPORTED;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, (size_t)(S * stage_bytes)) != cudaSuccess ||
      per_sm < 1) {
    (void)cudaGetLastError();  // the query's error is not the caller's
    per_sm = 1;
  }
  const int64_t slots = (int64_t)ds.sm_count * per_sm;
  const int64_t grid = a->m < slots ? a->m : slots;

  // The status word must start at zero for this call; the previous call's value stays in
  // the array until this clear runs on `stream`.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ds.scratch, 0, kStatusBytes, s) != cudaSuccess) {
    (void)cudaGetLastError();  // reported by the status; not left for the caller's next check
    return AR_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.dynamicSmemBytes = (size_t)(S * stage_bytes);
  cfg.stream = s;
  void* args[2] = {&p, &sp};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    (void)cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return AR_OK;
}
