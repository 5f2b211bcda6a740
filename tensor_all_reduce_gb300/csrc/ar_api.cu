// C ABI of libar: argument validation, variant selection and the single launch per call.
//
// Validation runs before the context is consulted, so argument errors are reported the
// same way with or without a GPU.  Nothing here allocates device memory, synchronises a
// stream or blocks: every compute call is one cudaLaunchKernelExC on the caller's stream
// (or nothing), which keeps the calls capturable in CUDA graphs.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ar.h"
#include "ar_common.cuh"
#include "ar_launch.h"
#include "ar_staged.cuh"

struct ar_ctx {
  int device;
  int sm_count;
  int64_t l2_bytes;
  int max_cluster;       // largest cluster the fused kernel can be launched with
  int max_dyn_smem;      // opt-in dynamic shared memory per block (bytes)
  int* d_status;         // device status word of the staged kernel (0 = no timeout)
  // overrides (0 = automatic)
  int force_variant;
  int cluster_size;
  int ppt;
  int reduce_unroll;
  int stages;
  int pdl;               // launch with programmatic stream serialisation
  long long wait_cycles; // bound of one staged-kernel wait (0: about a second)
  int test_stall;        // test hook: make the staged kernel's first waits run out
  int prefetch;          // warm L2 with the first inputs before the grid-dependency wait
  const char* last_variant;
  char last_error[256];
};

namespace {

constexpr int kReduceBlock = 256;

// Switch to the context's device for the duration of a call, restoring the caller's.
struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

int elem_size(ar_dtype d) { return d == AR_DTYPE_F32 ? 4 : 2; }

bool dtype_ok(int d) { return d == AR_DTYPE_F32 || d == AR_DTYPE_F16 || d == AR_DTYPE_BF16; }

uintptr_t addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }

bool overlaps(const void* a, int64_t an, const void* b, int64_t bn) {
  if (an <= 0 || bn <= 0) return false;
  return addr(a) < addr(b) + (uintptr_t)bn && addr(b) < addr(a) + (uintptr_t)an;
}

bool aligned(const void* p, int bytes) { return (addr(p) % (uintptr_t)bytes) == 0; }

ar_status fail_cuda(ar_ctx* ctx, cudaError_t e, const char* what) {
  if (ctx) snprintf(ctx->last_error, sizeof(ctx->last_error), "%s: %s", what, cudaGetErrorString(e));
  return AR_ERR_CUDA;
}

ar_status launch(ar_ctx* ctx, const void* fn, unsigned grid, unsigned block, int csize, void** args,
                 size_t dyn_smem, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (csize > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)csize;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (ctx->pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return fail_cuda(ctx, e, "kernel launch");
  return AR_OK;
}

}  // namespace

namespace ar {
void fill_fused_params(FusedParams& p, const ar_fused_args& a, int chunk, int csize) {
  memset(&p, 0, sizeof(p));
  for (int r = 0; r < a.n; ++r) p.x[r] = a.partials[r];
  p.res_in = a.residual_in;
  p.res_out = a.residual_out;
  p.w = a.weight;
  p.out = a.out;
  p.q = static_cast<uint8_t*>(a.q_out);
  p.scale = a.scale_out;
  p.m = a.m;
  p.h = (int)a.h;
  p.row_packs = (int)((a.h + 7) / 8);
  p.chunk_packs = chunk;
  p.csize = csize;
  p.eps = a.eps;
  p.inv_h = (float)(1.0 / (double)a.h);
  p.gemma = a.gemma != 0;
  p.skip_norm = a.skip_norm != 0;
  p.out_f32 = a.out_fp32 != 0 && a.out != nullptr;
  const bool per_group = a.quant == AR_QUANT_FP8_E4M3_PER_GROUP;
  p.group_lanes = per_group ? a.group_size / 8 : 0;
  p.ngroups = per_group ? (int)(a.h / a.group_size) : 0;
  p.ld_in = a.ld_in ? a.ld_in : a.h;
  p.ld_out = a.ld_out ? a.ld_out : a.h;
}

int fused_kernel_list(const void** out, int cap) {
  int k = 0;
  for (int dt = 0; dt < 2; ++dt)
    for (int n = 1; n <= AR_MAX_PARTIALS; ++n)
      for (int ppt = 1; ppt <= 4; ppt *= 2)
        for (int q = 0; q < 2; ++q)
          for (int v = 0; v < 2; ++v) {
            if (!v && ppt != 1) continue;  // the scalar form has one pack per thread
            const void* fn = dt ? fused_kernel_bf16(n, ppt, q != 0, v != 0) : fused_kernel_f16(n, ppt, q != 0, v != 0);
            if (fn && k < cap) out[k++] = fn;
          }
  return k;
}

int staged_kernel_list(const void** out, int cap) {
  int k = 0;
  for (int dt = 0; dt < 2; ++dt)
    for (int n = 1; n <= AR_MAX_PARTIALS; ++n)
      for (int ppt = 1; ppt <= 4; ppt *= 2)
        for (int q = 0; q < 2; ++q) {
          const void* fn = dt ? staged_kernel_bf16(n, ppt, q != 0) : staged_kernel_f16(n, ppt, q != 0);
          if (fn && k < cap) out[k++] = fn;
        }
  for (int dt = 0; dt < 2; ++dt)
    for (int n = 1; n <= AR_MAX_PARTIALS; ++n)
      for (int q = 0; q < 2; ++q) {
        const void* fn = dt ? batch_kernel_bf16(n, q != 0) : batch_kernel_f16(n, q != 0);
        if (fn && k < cap) out[k++] = fn;
        for (int ppt = 1; ppt <= 2; ++ppt) {
          fn = dt ? staged_cluster_kernel_bf16(n, ppt, q != 0) : staged_cluster_kernel_f16(n, ppt, q != 0);
          if (fn && k < cap) out[k++] = fn;
        }
      }
  return k;
}
}  // namespace ar

extern "C" {

const char* ar_status_string(ar_status s) {
  switch (s) {
    case AR_OK: return "success";
    case AR_ERR_INVALID_ARG: return "invalid argument";
    case AR_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case AR_ERR_ALIGNMENT: return "pointer not aligned to its element size";
    case AR_ERR_CUDA: return "CUDA error";
    case AR_ERR_NOT_INITIALIZED: return "context not initialised";
    case AR_ERR_OVERLAP: return "output overlaps an input or another output";
  }
  return "unknown status";
}

const char* ar_last_error(const ar_ctx* ctx) { return ctx ? ctx->last_error : ""; }

const char* ar_last_variant(const ar_ctx* ctx) { return ctx ? ctx->last_variant : ""; }

ar_status ar_init(ar_ctx** out, int device, unsigned flags) {
  if (!out) return AR_ERR_INVALID_ARG;
  *out = nullptr;
  if (flags != 0) return AR_ERR_INVALID_ARG;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return AR_ERR_CUDA;
  if (device < 0 || device >= count) return AR_ERR_INVALID_ARG;
  int major = 0, minor = 0, sms = 0, l2 = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, device) != cudaSuccess)
    return AR_ERR_CUDA;
  if (major != 10 || minor != 3) return AR_ERR_UNSUPPORTED;  // built for sm_103a only

  ar_ctx* ctx = static_cast<ar_ctx*>(calloc(1, sizeof(ar_ctx)));
  if (!ctx) return AR_ERR_INVALID_ARG;
  ctx->device = device;
  ctx->sm_count = sms;
  ctx->l2_bytes = l2;
  ctx->last_variant = "none";
  ctx->max_cluster = 8;
  ctx->pdl = 1;
  ctx->prefetch = 1;

  DeviceGuard g(device);
  // Load every kernel now (lazy module loading would otherwise do it on first launch,
  // possibly inside a stream capture) and allow 16-CTA clusters for the fused kernels.
  const void* fns[512];
  int nf = ar::fused_kernel_list(fns, 512);
  for (int i = 0; i < nf; ++i) {
    e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      free(ctx);
      return AR_ERR_CUDA;
    }
  }
  for (int dt = 0; dt < 3; ++dt)
    for (int n = 1; n <= AR_MAX_PARTIALS; ++n)
      for (int u = 1; u <= 4; u += 3)
        for (int v = 0; v < 2; ++v)
          for (int t = 0; t < 2; ++t) {
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, ar::reduce_kernel(dt, n, u, v != 0, t != 0));
            if (e != cudaSuccess) {
              free(ctx);
              return AR_ERR_CUDA;
            }
          }
  // Staged kernels: allow the opt-in shared memory size; one status word for their
  // bounded waits (the only device memory a context owns).
  {
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
      free(ctx);
      return AR_ERR_CUDA;
    }
    ctx->max_dyn_smem = optin - 1024;  // room for the kernels' static shared memory
    nf = ar::staged_kernel_list(fns, 512);
    for (int i = 0; i < nf; ++i) {
      e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, ctx->max_dyn_smem);
      if (e != cudaSuccess) {
        free(ctx);
        return AR_ERR_CUDA;
      }
    }
    if (cudaMalloc(&ctx->d_status, 256) != cudaSuccess || cudaMemset(ctx->d_status, 0, 256) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
      if (ctx->d_status) cudaFree(ctx->d_status);
      free(ctx);
      return AR_ERR_CUDA;
    }
  }
  // Largest cluster the fused kernel supports with a small block on this device.
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int csz = 0;
    if (cudaOccupancyMaxPotentialClusterSize(&csz, ar::fused_kernel_bf16(4, 1, true, true), &cfg) ==
            cudaSuccess &&
        csz >= 1)
      ctx->max_cluster = csz >= 16 ? 16 : (csz >= 8 ? 8 : (csz >= 4 ? 4 : (csz >= 2 ? 2 : 1)));
    cudaGetLastError();
  }
  *out = ctx;
  return AR_OK;
}

ar_status ar_destroy(ar_ctx* ctx) {
  if (ctx) {
    if (ctx->d_status) {
      DeviceGuard g(ctx->device);
      cudaFree(ctx->d_status);
    }
    free(ctx);
  }
  return AR_OK;
}

ar_status ar_device_status(ar_ctx* ctx, int* code) {
  if (!code) return AR_ERR_INVALID_ARG;
  if (!ctx) return AR_ERR_NOT_INITIALIZED;
  DeviceGuard g(ctx->device);
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(ctx, e, "status read");
  if (v != 0) {
    e = cudaMemset(ctx->d_status, 0, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(ctx, e, "status reset");
  }
  *code = v;
  return AR_OK;
}

ar_status ar_set_option(ar_ctx* ctx, ar_option opt, int64_t v) {
  if (!ctx) return AR_ERR_NOT_INITIALIZED;
  switch (opt) {
    case AR_OPT_FORCE_VARIANT:
      if (v < 0 || v > 4) return AR_ERR_INVALID_ARG;
      ctx->force_variant = (int)v;
      return AR_OK;
    case AR_OPT_CLUSTER_SIZE:
      if (!(v == 0 || v == 1 || v == 2 || v == 4 || v == 8 || v == 16)) return AR_ERR_INVALID_ARG;
      ctx->cluster_size = (int)v;
      return AR_OK;
    case AR_OPT_PACKS_PER_THREAD:
      if (!(v == 0 || v == 1 || v == 2 || v == 4)) return AR_ERR_INVALID_ARG;
      ctx->ppt = (int)v;
      return AR_OK;
    case AR_OPT_REDUCE_UNROLL:
      if (!(v == 0 || v == 1 || v == 4)) return AR_ERR_INVALID_ARG;
      ctx->reduce_unroll = (int)v;
      return AR_OK;
    case AR_OPT_STAGES:
      if (!(v == 0 || (v >= 1 && v <= 4))) return AR_ERR_INVALID_ARG;
      ctx->stages = (int)v;
      return AR_OK;
    case AR_OPT_PDL:
      if (v != 0 && v != 1) return AR_ERR_INVALID_ARG;
      ctx->pdl = (int)v;
      return AR_OK;
    case AR_OPT_WAIT_CYCLES:
      if (v != 0 && (v < 1000 || v > 8000000000LL)) return AR_ERR_INVALID_ARG;
      ctx->wait_cycles = v;
      return AR_OK;
    case AR_OPT_TEST_STALL:
      if (v != 0 && v != 1) return AR_ERR_INVALID_ARG;
      ctx->test_stall = (int)v;
      return AR_OK;
    case AR_OPT_L2_PREFETCH:
      if (v != 0 && v != 1) return AR_ERR_INVALID_ARG;
      ctx->prefetch = (int)v;
      return AR_OK;
  }
  return AR_ERR_INVALID_ARG;
}

ar_status ar_get_info(const ar_ctx* ctx, ar_info key, int64_t* value) {
  if (!value) return AR_ERR_INVALID_ARG;
  if (!ctx) return AR_ERR_NOT_INITIALIZED;
  switch (key) {
    case AR_INFO_SM_COUNT: *value = ctx->sm_count; return AR_OK;
    case AR_INFO_L2_BYTES: *value = ctx->l2_bytes; return AR_OK;
    case AR_INFO_REDUCE_TILE_PACKS:
      *value = (int64_t)kReduceBlock * (ctx->reduce_unroll ? ctx->reduce_unroll : 4);
      return AR_OK;
    case AR_INFO_DEVICE: *value = ctx->device; return AR_OK;
  }
  return AR_ERR_INVALID_ARG;
}

// ---------------------------------------------------------------------------
// plain reduce
// ---------------------------------------------------------------------------

static ar_status fused_impl(ar_ctx* ctx, const ar_fused_args* a, void* stream, bool host);

// Smallest 16-bit array reduced through the staged kernel, in elements per SM: sixteen rows
// of the longest row length per SM (with fewer rows per CTA its pipeline fill and drain
// cost more than the bulk copies gain).
constexpr int64_t kStagedReduceMinElemsPerSm = 8192LL * 16;

ar_status ar_reduce_sum(ar_ctx* ctx, void* out, const void* const* partials, int n, int64_t numel,
                        ar_dtype dtype, void* stream) {
  if (!partials || n < 1 || n > AR_MAX_PARTIALS || numel < 0 || !dtype_ok(dtype)) return AR_ERR_INVALID_ARG;
  if (numel == 0) {  // nothing is touched: any pointer (NULL included) is acceptable
    if (!ctx) return AR_ERR_NOT_INITIALIZED;
    ctx->last_variant = "none";
    return AR_OK;
  }
  if (!out) return AR_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  if (numel > INT64_MAX / 16) return AR_ERR_INVALID_ARG;
  const int64_t bytes = numel * es;
  if (!aligned(out, es)) return AR_ERR_ALIGNMENT;
  for (int r = 0; r < n; ++r) {
    if (!partials[r]) return AR_ERR_INVALID_ARG;
    if (!aligned(partials[r], es)) return AR_ERR_ALIGNMENT;
    if (partials[r] != out && overlaps(out, bytes, partials[r], bytes)) return AR_ERR_OVERLAP;
  }
  if (!ctx) return AR_ERR_NOT_INITIALIZED;

  ar::ReduceParams p;
  memset(&p, 0, sizeof(p));
  for (int r = 0; r < n; ++r) p.x[r] = partials[r];
  p.out = out;
  p.numel = numel;
  p.prefetch = ctx->prefetch;
  bool vec = aligned(out, 16);
  for (int r = 0; r < n; ++r) vec = vec && aligned(partials[r], 16);
  if (ctx->force_variant == 4) vec = false;

  // Large 16-bit arrays of 4 to 6 partials: the same sum through the staged fused kernel on
  // the array viewed as rows (no residual, no norm; the rounded sum is stored as the output,
  // bit for bit the value below).  Same-GPU A/B on GB300 at 25M elements: N = 4 at 95.7 %
  // of the measured copy bandwidth against 88.0 % for the per-thread kernel, N = 6 99.1 %
  // against 96.0 %; with fewer partials they tie, with eight the per-thread kernel wins.
  if (es == 2 && vec && n >= 4 && n <= 6 && ctx->force_variant == 0 && ctx->reduce_unroll == 0 &&
      numel >= kStagedReduceMinElemsPerSm * ctx->sm_count) {
    // the longest row that divides the array and leaves room for two stages of N rows
    int64_t h = 0;
    for (int64_t c : {8192, 7168, 6144, 5120, 4096, 3072, 2048})
      if (numel % c == 0 && 2 * n * c * es <= ctx->max_dyn_smem) {
        h = c;
        break;
      }
    if (h) {
      ar_fused_args fa;
      memset(&fa, 0, sizeof(fa));
      fa.n = n;
      for (int r = 0; r < n; ++r) fa.partials[r] = partials[r];
      fa.out = out;
      fa.m = numel / h;
      fa.h = h;
      fa.dtype = dtype;
      fa.skip_norm = 1;
      fa.quant = AR_QUANT_NONE;
      const ar_status st = fused_impl(ctx, &fa, stream, false);
      if (st == AR_OK) ctx->last_variant = strcmp(ctx->last_variant, "fused_staged") == 0 ? "reduce_staged" : "reduce_rows";
      return st;
    }
  }

  DeviceGuard g(ctx->device);
  const int max_grid = ctx->sm_count * (2048 / kReduceBlock);
  unsigned grid;
  const void* fn;
  const char* name;
  if (vec) {
    const int epp = 16 / es;
    p.npacks = numel / epp;
    // Four packs per thread per tile only for 16-bit sums of one to three partials that fill
    // at least one wave of single-pack tiles; one pack otherwise.  Same-GPU A/B on GB300 with
    // the L2 prefetch (us/call, HBM-cold, four packs against one): bf16 N = 2, 6.3M elements
    // 6.39 / 7.17, 25M 24.21 / 23.88; N = 3, 25M 34.01 / 34.21; N = 8, 25M 90.89 / 68.33;
    // fp16 N = 4, 3.1M 8.30 / 6.16; fp32 N = 2 / 4 / 8, 25M 47.24 / 46.66, 78.91 / 77.41,
    // 140.08 / 138.20; fp32 N = 4, 6.3M 23.77 / 20.94.
    int unroll = ctx->reduce_unroll;
    if (unroll == 0)
      unroll = (es == 2 && n <= 3 && p.npacks >= (int64_t)max_grid * kReduceBlock) ? 4 : 1;
    const int64_t tile = (int64_t)kReduceBlock * unroll;
    p.full_tiles = p.npacks / tile;
    const bool has_tail = (p.npacks % tile) != 0 || (numel % epp) != 0;
    // with room in the grid the tail gets a block of its own (block full_tiles owns it), so
    // it runs beside the full tiles instead of after one of them
    const int64_t want = p.full_tiles + (has_tail ? 1 : 0);
    int64_t gr = want < max_grid ? want : max_grid;
    if (gr < 1) gr = 1;
    grid = (unsigned)gr;
    fn = ar::reduce_kernel(dtype, n, unroll, true, has_tail);
    name = has_tail ? "reduce_vec_tail" : "reduce_vec";
  } else {
    int64_t gr = (numel + kReduceBlock - 1) / kReduceBlock;
    if (gr > max_grid) gr = max_grid;
    grid = (unsigned)gr;
    fn = ar::reduce_kernel(dtype, n, 1, false, false);
    name = "reduce_scalar";
  }
  if (!fn) return AR_ERR_UNSUPPORTED;
  void* args[1] = {&p};
  ar_status st = launch(ctx, fn, grid, kReduceBlock, 1, args, 0, stream);
  if (st == AR_OK) ctx->last_variant = name;
  return st;
}

// ---------------------------------------------------------------------------
// fused reduce + residual + RMSNorm (+ FP8)
// ---------------------------------------------------------------------------

// The fused call.  `host`: some buffers are page-locked host memory (already resolved to
// their device addresses), so only kernels that reach memory through plain loads and
// stores run (bulk asynchronous copies are used on device memory only).
static ar_status fused_impl(ar_ctx* ctx, const ar_fused_args* a, void* stream, bool host) {
  if (!a) return AR_ERR_INVALID_ARG;
  if (a->n < 1 || a->n > AR_MAX_PARTIALS || a->m < 0 || a->h < 1 || (!a->weight && !a->skip_norm))
    return AR_ERR_INVALID_ARG;
  if (a->dtype != AR_DTYPE_BF16 && a->dtype != AR_DTYPE_F16) return AR_ERR_INVALID_ARG;
  if (a->quant != AR_QUANT_NONE && a->quant != AR_QUANT_FP8_E4M3_PER_TOKEN && a->quant != AR_QUANT_FP8_E4M3_PER_GROUP)
    return AR_ERR_INVALID_ARG;
  const bool quant = a->quant != AR_QUANT_NONE;
  const bool per_group = a->quant == AR_QUANT_FP8_E4M3_PER_GROUP;
  if (per_group) {  // groups of 8..256 (a power of two) elements, a whole number per row
    const int g = a->group_size;
    if (g < 8 || g > 256 || (g & (g - 1)) != 0 || a->h % g != 0) return AR_ERR_INVALID_ARG;
    if (a->h > 8192) return AR_ERR_UNSUPPORTED;  // one CTA holds a whole row
  }
  const int64_t scale_count = per_group ? a->m * (a->h / a->group_size) : a->m;
  if (!(a->eps >= 0.0f) || isinf(a->eps)) return AR_ERR_INVALID_ARG;  // also rejects NaN
  if (a->h > (int64_t)1 << 30 || a->ld_in < 0 || a->ld_out < 0 || (a->ld_in && a->ld_in < a->h) ||
      (a->ld_out && a->ld_out < a->h) || a->ld_in > (int64_t)1 << 31 || a->ld_out > (int64_t)1 << 31)
    return AR_ERR_INVALID_ARG;
  const int64_t li = a->ld_in ? a->ld_in : a->h, lo = a->ld_out ? a->ld_out : a->h;  // row strides
  if (a->m > ((int64_t)1 << 40) / (li > lo ? li : lo)) return AR_ERR_INVALID_ARG;
  if (a->m == 0) {  // no rows: only the weight is a real buffer; nothing is touched
    if (!ctx) return AR_ERR_NOT_INITIALIZED;
    ctx->last_variant = "none";
    return AR_OK;
  }
  if (quant && (!a->q_out || !a->scale_out)) return AR_ERR_INVALID_ARG;
  if (!quant && !a->out) return AR_ERR_INVALID_ARG;
  for (int r = 0; r < a->n; ++r)
    if (!a->partials[r]) return AR_ERR_INVALID_ARG;

  const int es = elem_size(a->dtype);
  const int oes = a->out_fp32 ? 4 : es;  // element size of `out`
  const int64_t ext_in = (a->m - 1) * li + a->h;   // elements an input spans (padding included)
  const int64_t ext_out = (a->m - 1) * lo + a->h;  // elements an output spans
  const int64_t tb = ext_in * es;                  // bytes of one input [m, h] tensor
  // element alignment
  for (int r = 0; r < a->n; ++r)
    if (!aligned(a->partials[r], es)) return AR_ERR_ALIGNMENT;
  if ((a->residual_in && !aligned(a->residual_in, es)) || (a->residual_out && !aligned(a->residual_out, es)) ||
      !aligned(a->weight, es) || (a->out && !aligned(a->out, oes)) || (quant && !aligned(a->scale_out, 4)))
    return AR_ERR_ALIGNMENT;
  // overlap: outputs may equal an [m, h] input of the same type and row stride exactly
  // (every element is read before the same thread writes it), never partially overlap an
  // input, and never overlap one another
  struct Range { const void* p; int64_t n; bool same_shape; };
  Range ins[AR_MAX_PARTIALS + 2];
  int ni = 0;
  for (int r = 0; r < a->n; ++r) ins[ni++] = {a->partials[r], tb, true};
  if (a->residual_in) ins[ni++] = {a->residual_in, tb, true};
  if (a->weight) ins[ni++] = {a->weight, (int64_t)a->h * es, false};
  Range outs[4];
  int no = 0;
  if (a->residual_out) outs[no++] = {a->residual_out, ext_out * es, li == lo};
  if (a->out) outs[no++] = {a->out, ext_out * oes, !a->out_fp32 && li == lo};
  if (quant) {
    outs[no++] = {a->q_out, ext_out, false};
    outs[no++] = {a->scale_out, scale_count * 4, false};
  }
  for (int o = 0; o < no; ++o) {
    for (int i = 0; i < ni; ++i) {
      if (outs[o].same_shape && ins[i].same_shape && outs[o].p == ins[i].p) continue;
      if (overlaps(outs[o].p, outs[o].n, ins[i].p, ins[i].n)) return AR_ERR_OVERLAP;
    }
    for (int o2 = o + 1; o2 < no; ++o2)
      if (overlaps(outs[o].p, outs[o].n, outs[o2].p, outs[o2].n)) return AR_ERR_OVERLAP;
  }
  if (!ctx) return AR_ERR_NOT_INITIALIZED;

  // ---- variant selection ----
  // the vector kernels need 16-byte-aligned rows: h, and both row strides, multiples of 8
  bool vec = (a->h % 8) == 0 && (li % 8) == 0 && (lo % 8) == 0;
  for (int r = 0; r < a->n; ++r) vec = vec && aligned(a->partials[r], 16);
  vec = vec && (!a->residual_in || aligned(a->residual_in, 16)) && (!a->residual_out || aligned(a->residual_out, 16)) &&
        aligned(a->weight, 16) && (!a->out || aligned(a->out, 16)) && (!quant || aligned(a->q_out, 8));
  if (ctx->force_variant == 4) vec = false;

  const int row_packs = (int)((a->h + 7) / 8);
  const int max_cl = ctx->max_cluster;

  // ---- staged (bulk-copy pipelined, persistent) variants ----
  const int rows_per_stage = a->n + (a->residual_in ? 1 : 0);
  // kernel parameters of the staged forms: `chunk` packs of each row per CTA, `cl` CTAs per row
  auto staged_params = [&](ar::FusedParams& p, ar::StagedParams& sp, int chunk, int cl, int stages) {
    ar::fill_fused_params(p, *a, chunk, cl);
    p.prefetch = ctx->prefetch;
    sp = ar::StagedParams{};
    sp.stages = stages;
    sp.row_bytes = chunk * 16;  // bytes of a row's chunk (a whole row without a cluster)
    sp.err = ctx->d_status;
    sp.wait_cycles = ctx->wait_cycles ? ctx->wait_cycles : 2000000000LL;  // about a second at 2 GHz
    sp.stall_first = ctx->test_stall;
  };

  // Cluster form: rows longer than one CTA holds (more than 1024 packs) are split over 2 or
  // 4 CTAs of a cluster, each staging its slice; forced with AR_OPT_FORCE_VARIANT = 3 and
  // a cluster size.
  if (!host && vec) {
    DeviceGuard dg(ctx->device);
    int cl = 0;
    if (ctx->force_variant == 3 && ctx->cluster_size > 1) {
      cl = ctx->cluster_size;
    } else if (ctx->force_variant == 0 && ctx->cluster_size == 0 && ctx->ppt == 0 && row_packs > 1024) {
      // 2 or 4 CTAs per row: of the sizes whose slices fit one CTA with two stages, the one
      // that keeps the most threads resident per SM, then the smaller (same-GPU A/B on GB300:
      // N = 4, h = 12288 at 90 % of the measured copy bandwidth with 4 CTAs, three per SM,
      // against 88 % with 2; h = 16384 95 % with 2 against 90 % with 4; N = 8, h = 16384
      // 96 % with 4; 8 CTAs per row was never faster where fewer fit, and is used only where
      // they do not).  With few rows (at most a quarter as many as SMs) the larger size that
      // fits, to engage more SMs (m = 16, h = 16384: 4.1 us with 4 CTAs, 4.8 with 2).
      const bool few_rows = a->m * 4 <= ctx->sm_count;
      int best = 0;
      for (int c = 2; c <= 8; c *= 2) {
        if (c == 8 && cl) break;
        const int ch = row_packs / c;
        const int64_t st2 = 2 * (int64_t)rows_per_stage * ch * 16;
        if (row_packs % c || ch > 1024 || st2 > ctx->max_dyn_smem) continue;
        const int thr = ((ch + 1) / 2 + 31) / 32 * 32;
        const void* f = a->dtype == AR_DTYPE_BF16 ? ar::staged_cluster_kernel_bf16(a->n, 2, quant)
                                                  : ar::staged_cluster_kernel_f16(a->n, 2, quant);
        int per_sm = 1;
        if (!f || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, thr, (size_t)st2) != cudaSuccess) {
          (void)cudaGetLastError();
          per_sm = 1;
        }
        if (per_sm * thr > best || (few_rows && cl)) {
          best = per_sm * thr;
          cl = c;
        }
      }
    }
    if (cl > 1) {
      const int chunk = row_packs / cl;
      const int64_t cstage = (int64_t)rows_per_stage * chunk * 16;
      int CS = ctx->stages ? ctx->stages : 2;
      if (!ctx->stages && CS * cstage > ctx->max_dyn_smem) CS = 1;
      // two packs per thread (one pack was 10-25 % slower in this form)
      const int cppt = ctx->ppt ? ctx->ppt : 2;
      const bool ok = cl <= 8 && row_packs % cl == 0 && chunk <= 1024 && (cppt == 1 || cppt == 2) &&
                      CS * cstage <= ctx->max_dyn_smem && (!per_group || chunk % (a->group_size / 8) == 0);
      if (ok) {
        ar::FusedParams p;
        ar::StagedParams sp;
        staged_params(p, sp, chunk, cl, CS);
        int block = ((chunk + cppt - 1) / cppt + 31) / 32 * 32;
        if (block < 32) block = 32;
        const void* fn = a->dtype == AR_DTYPE_BF16 ? ar::staged_cluster_kernel_bf16(a->n, cppt, quant)
                                                   : ar::staged_cluster_kernel_f16(a->n, cppt, quant);
        if (!fn) return AR_ERR_UNSUPPORTED;
        DeviceGuard g(ctx->device);
        // persistent grid: as many clusters as fit at once
        cudaLaunchConfig_t oc = {};
        oc.gridDim = dim3((unsigned)(cl * ctx->sm_count), 1, 1);
        oc.blockDim = dim3((unsigned)block, 1, 1);
        oc.dynamicSmemBytes = (size_t)(CS * cstage);
        cudaLaunchAttribute at;
        at.id = cudaLaunchAttributeClusterDimension;
        at.val.clusterDim.x = (unsigned)cl;
        at.val.clusterDim.y = 1;
        at.val.clusterDim.z = 1;
        oc.attrs = &at;
        oc.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, fn, &oc) != cudaSuccess || nclusters < 1) {
          (void)cudaGetLastError();
          nclusters = ctx->sm_count / cl;
        }
        const int64_t clusters = a->m < nclusters ? a->m : nclusters;
        void* args[2] = {&p, &sp};
        ar_status st = launch(ctx, fn, (unsigned)(clusters * cl), (unsigned)block, cl, args, (size_t)(CS * cstage),
                              stream);
        if (st == AR_OK) ctx->last_variant = "fused_staged_cluster";
        return st;
      }
      if (ctx->force_variant == 3) return AR_ERR_UNSUPPORTED;
    }
  }

  // One CTA per row.
  const int64_t stage_bytes = (int64_t)rows_per_stage * a->h * es;
  // Stages per CTA: two stages in one CTA per SM stream best with every epilogue (three
  // stages, or one stage and two CTAs per SM, were slower in same-GPU A/B runs on GB300 at
  // N = 4 and 8, h = 6144 and 7168, m = 1024 .. 4096).  With one to two rows per SM a
  // single stage lets every row have its own resident CTA.
  const bool one_row_per_cta = a->m >= ctx->sm_count && a->m <= 2LL * ctx->sm_count;
  int S = ctx->stages ? ctx->stages : (one_row_per_cta ? 1 : 2);
  if (!ctx->stages && S * stage_bytes > ctx->max_dyn_smem) S = 1;
  const bool staged_ok = vec && row_packs <= 1024 && S * stage_bytes <= ctx->max_dyn_smem;
  // Automatic choice: the staged kernel for every batch of 16-byte-aligned rows of at most
  // 8192 elements; up to two rows per SM with one CTA per row, all resident at once, else
  // persistent.  Same-GPU sweeps on GB300 (N = 4, h = 6144 and 8192, m = 1 .. 4096, with
  // the L2 prefetch ahead of the grid-dependency wait): the per-thread-load row kernel was
  // slower at every size, also at three to four rows per SM where it once led (m = 600:
  // 10.1 against 11.2 us; 512 x 8192: 11.1 against 14.1 us).
  const bool staged_auto = ctx->force_variant == 0 && ctx->cluster_size == 0 && ctx->ppt == 0;
  if (host && ctx->force_variant == 3) return AR_ERR_UNSUPPORTED;
  if (!host && (ctx->force_variant == 3 || (staged_auto && staged_ok))) {
    if (!staged_ok) return AR_ERR_UNSUPPORTED;
    // packs per thread: 1 (768 threads for h = 6144) when each CTA runs through many rows
    // with the norm and at most 4 partials, else 2 (same A/B runs: 1 pack was 0.5-1 % faster
    // on N = 4, 2800 x 6144 with per-token and per-group FP8, without FP8 and with fp32
    // output; 2 packs on 1024 rows, on N = 8 and without the norm)
    const bool one_pack = a->n <= 4 && !a->skip_norm && a->m >= 8LL * ctx->sm_count && row_packs <= 1024;
    int sppt = ctx->ppt ? ctx->ppt : (one_pack ? 1 : 2);
    // One CTA per row with some SMs holding two rows, without FP8: one pack per thread when two
    // such CTAs still fit on an SM (same-GPU A/B on GB300, us/call HBM-cold, one pack against
    // two: N = 4, h = 6144, m = 200 / 256 / 300: 4.13 / 4.70, 4.59 / 4.77, 5.15 / 5.34;
    // h = 4096, m = 256: 3.78 / 4.43; with FP8 one pack was 2-6 % slower, at m = 152 2 %
    // slower, and at N = 8 its 54 registers a thread leave room for one CTA per SM: 28 % slower).
    if (!ctx->ppt && !one_pack && !quant && !a->skip_norm && a->m > ctx->sm_count && a->m <= 2LL * ctx->sm_count) {
      const void* f1 = a->dtype == AR_DTYPE_BF16 ? ar::staged_kernel_bf16(a->n, 1, false)
                                                 : ar::staged_kernel_f16(a->n, 1, false);
      const int b1 = (row_packs + 31) / 32 * 32;
      DeviceGuard og(ctx->device);
      int fit = 0;
      if (f1 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, f1, b1, (size_t)(S * stage_bytes)) != cudaSuccess) {
        (void)cudaGetLastError();
        fit = 0;
      }
      if (fit >= 2) sppt = 1;
    }
    int sblock = ((row_packs + sppt - 1) / sppt + 31) / 32 * 32;
    if (sblock < 32) sblock = 32;
    ar::FusedParams p;
    ar::StagedParams sp;
    staged_params(p, sp, row_packs, 1, S);
    const void* fn = a->dtype == AR_DTYPE_BF16 ? ar::staged_kernel_bf16(a->n, sppt, quant)
                                               : ar::staged_kernel_f16(a->n, sppt, quant);
    if (!fn) return AR_ERR_UNSUPPORTED;
    DeviceGuard g(ctx->device);
    // persistent grid: as many CTAs as fit on the SMs at once (shared memory bound)
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, sblock, (size_t)(S * stage_bytes)) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int64_t slots = (int64_t)ctx->sm_count * per_sm;
    const int64_t grid = a->m < slots ? a->m : slots;
    void* args[2] = {&p, &sp};
    ar_status st = launch(ctx, fn, (unsigned)grid, (unsigned)sblock, 1, args, (size_t)(S * stage_bytes), stream);
    if (st == AR_OK) ctx->last_variant = "fused_staged";
    return st;
  }
  int csize;
  if (ctx->cluster_size) {
    csize = ctx->cluster_size;
  } else if (ctx->force_variant == 1) {
    csize = 1;
  } else {
    // spread small batches over the SMs: grow the cluster while fewer CTAs than SMs would
    // be launched and every CTA keeps at least 32 packs (256 elements)
    csize = 1;
    const int64_t target = ctx->sm_count;
    while (csize < max_cl && a->m * csize < target && row_packs / (csize * 2) >= 32) csize *= 2;
    if (ctx->force_variant == 2 && csize == 1) csize = 2;
  }
  if (per_group) csize = 1;  // a group's lanes must sit in one CTA with packs from column 0
  // a CTA holds at most 1024 packs (1024 / ppt threads of ppt packs, the kernels' launch
  // bound): widen the cluster for very long rows
  constexpr int kMaxPacksPerCta = 1024;
  while (csize < max_cl && (row_packs + csize - 1) / csize > kMaxPacksPerCta) csize *= 2;
  if (csize > max_cl) csize = max_cl;
  const int chunk = (row_packs + csize - 1) / csize;
  if (chunk > kMaxPacksPerCta) return AR_ERR_UNSUPPORTED;  // h > 8192 * max cluster size
  int ppt = vec ? ctx->ppt : 1;
  // one pack per thread for short rows, and over host memory (the most loads in flight
  // per SM: measured fastest across the C2C link), else two
  if (ppt == 0) ppt = (chunk <= 256 || host) ? 1 : 2;
  int block = ((chunk + ppt - 1) / ppt + 31) / 32 * 32;
  if (block < 32) block = 32;
  const int64_t grid = a->m * csize;
  if (grid > 0x7FFFFFFFLL) return AR_ERR_UNSUPPORTED;

  ar::FusedParams p;
  ar::fill_fused_params(p, *a, chunk, csize);
  p.prefetch = host ? 0 : ctx->prefetch;  // bulk prefetches are used on device memory only

  const void* fn = a->dtype == AR_DTYPE_BF16 ? ar::fused_kernel_bf16(a->n, ppt, quant, vec)
                                             : ar::fused_kernel_f16(a->n, ppt, quant, vec);
  if (!fn) return AR_ERR_UNSUPPORTED;
  DeviceGuard g(ctx->device);
  void* args[1] = {&p};
  ar_status st = launch(ctx, fn, (unsigned)grid, (unsigned)block, csize, args, 0, stream);
  if (st == AR_OK) {
    if (vec)
      ctx->last_variant = csize > 1 ? "fused_cluster_vec" : "fused_row_vec";
    else
      ctx->last_variant = csize > 1 ? "fused_cluster_scalar" : "fused_scalar";
  }
  return st;
}

ar_status ar_fused_reduce_rmsnorm(ar_ctx* ctx, const ar_fused_args* a, void* stream) {
  return fused_impl(ctx, a, stream, false);
}

// Device address of a buffer that is device memory of the context's device or page-locked
// host memory mapped into the device's address space; anything else is refused.
static ar_status resolve_buffer(const ar_ctx* ctx, const void* p, const void** out) {
  *out = nullptr;
  if (!p) return AR_OK;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return AR_ERR_INVALID_ARG;
  }
  if (at.type == cudaMemoryTypeHost) {
    if (!at.devicePointer) return AR_ERR_INVALID_ARG;
    *out = at.devicePointer;
    return AR_OK;
  }
  if (at.type == cudaMemoryTypeDevice && at.device == ctx->device) {
    *out = p;
    return AR_OK;
  }
  return AR_ERR_INVALID_ARG;  // pageable host memory, or another device's memory
}

ar_status ar_fused_reduce_rmsnorm_host(ar_ctx* ctx, const ar_fused_args* a, void* stream) {
  // the argument rules of the device entry (they compare addresses only)
  const ar_status v = fused_impl(nullptr, a, nullptr, true);
  if (v != AR_ERR_NOT_INITIALIZED) return v;
  if (!ctx) return AR_ERR_NOT_INITIALIZED;
  DeviceGuard g(ctx->device);
  ar_fused_args d = *a;
  ar_status st = AR_OK;
  for (int r = 0; r < a->n && st == AR_OK; ++r) st = resolve_buffer(ctx, a->partials[r], &d.partials[r]);
  const void* t = nullptr;
  if (st == AR_OK) st = resolve_buffer(ctx, a->residual_in, &d.residual_in);
  if (st == AR_OK && (st = resolve_buffer(ctx, a->residual_out, &t)) == AR_OK) d.residual_out = const_cast<void*>(t);
  if (st == AR_OK) st = resolve_buffer(ctx, a->weight, &d.weight);
  if (st == AR_OK && (st = resolve_buffer(ctx, a->out, &t)) == AR_OK) d.out = const_cast<void*>(t);
  if (st == AR_OK && (st = resolve_buffer(ctx, a->q_out, &t)) == AR_OK) d.q_out = const_cast<void*>(t);
  if (st == AR_OK && (st = resolve_buffer(ctx, a->scale_out, &t)) == AR_OK)
    d.scale_out = static_cast<float*>(const_cast<void*>(t));
  if (st != AR_OK) {
    snprintf(ctx->last_error, sizeof(ctx->last_error),
             "a buffer is neither device memory of this device nor page-locked host memory");
    return st;
  }
  return fused_impl(ctx, &d, stream, true);
}

// ---------------------------------------------------------------------------
// batched fused calls
// ---------------------------------------------------------------------------

namespace {

struct CallRanges {
  int nin = 0, nout = 0;
  const void* in[AR_MAX_PARTIALS + 2];
  int64_t in_n[AR_MAX_PARTIALS + 2];
  const void* out[4];
  int64_t out_n[4];
};

CallRanges ranges_of(const ar_fused_args* a) {
  CallRanges r;
  const int64_t li = a->ld_in ? a->ld_in : a->h, lo = a->ld_out ? a->ld_out : a->h;
  const int64_t es = elem_size(a->dtype), mh = a->m > 0 ? (a->m - 1) * lo + a->h : 0;
  const int64_t tb = a->m > 0 ? ((a->m - 1) * li + a->h) * es : 0;
  for (int k = 0; k < a->n; ++k) { r.in[r.nin] = a->partials[k]; r.in_n[r.nin++] = tb; }
  if (a->residual_in) { r.in[r.nin] = a->residual_in; r.in_n[r.nin++] = tb; }
  if (a->weight && !a->skip_norm) { r.in[r.nin] = a->weight; r.in_n[r.nin++] = a->h * es; }
  if (a->residual_out) { r.out[r.nout] = a->residual_out; r.out_n[r.nout++] = mh * es; }
  if (a->out) { r.out[r.nout] = a->out; r.out_n[r.nout++] = mh * (a->out_fp32 ? 4 : es); }
  if (a->quant) {
    const int64_t ns = a->quant == AR_QUANT_FP8_E4M3_PER_GROUP ? a->m * (a->h / a->group_size) : a->m;
    r.out[r.nout] = a->q_out; r.out_n[r.nout++] = mh;
    r.out[r.nout] = a->scale_out; r.out_n[r.nout++] = ns * 4;
  }
  return r;
}

}  // namespace

extern "C" ar_status ar_fused_reduce_rmsnorm_batch(ar_ctx* ctx, const ar_fused_args* calls, int count,
                                                   void* stream) {
  if (!calls || count < 1 || count > AR_MAX_BATCH) return AR_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {  // each call by the single-call rules (checked before any context use)
    const ar_status v = ar_fused_reduce_rmsnorm(nullptr, &calls[i], stream);
    if (v != AR_ERR_NOT_INITIALIZED) return v;
  }
  const ar_fused_args& c0 = calls[0];
  for (int i = 1; i < count; ++i) {
    const ar_fused_args& c = calls[i];
    if (c.n != c0.n || c.dtype != c0.dtype || c.quant != c0.quant || (c.skip_norm != 0) != (c0.skip_norm != 0) ||
        (c.out_fp32 != 0) != (c0.out_fp32 != 0))
      return AR_ERR_INVALID_ARG;
  }
  // the calls run at the same time: no call may write what another call reads or writes
  CallRanges rg[AR_MAX_BATCH];
  for (int i = 0; i < count; ++i) rg[i] = ranges_of(&calls[i]);
  for (int i = 0; i < count; ++i)
    for (int j = 0; j < count; ++j) {
      if (i == j) continue;
      for (int o = 0; o < rg[i].nout; ++o) {
        for (int k = 0; k < rg[j].nin; ++k)
          if (overlaps(rg[i].out[o], rg[i].out_n[o], rg[j].in[k], rg[j].in_n[k])) return AR_ERR_OVERLAP;
        for (int k = 0; k < rg[j].nout; ++k)
          if (overlaps(rg[i].out[o], rg[i].out_n[o], rg[j].out[k], rg[j].out_n[k])) return AR_ERR_OVERLAP;
      }
    }
  if (!ctx) return AR_ERR_NOT_INITIALIZED;

  // one launch when every call can take the staged path with one stage per CTA
  bool one = true;
  int64_t total_rows = 0, max_stage = 0;
  int max_row_packs = 1;
  for (int i = 0; i < count; ++i) {
    const ar_fused_args& a = calls[i];
    bool vec = (a.h % 8) == 0 && a.h <= 8192 && (a.ld_in % 8) == 0 && (a.ld_out % 8) == 0;
    for (int r = 0; r < a.n; ++r) vec = vec && aligned(a.partials[r], 16);
    vec = vec && aligned(a.residual_in, 16) && aligned(a.residual_out, 16) && aligned(a.weight, 16) &&
          aligned(a.out, 16) && (!a.quant || aligned(a.q_out, 8));
    one = one && vec;
    total_rows += a.m;
    const int64_t stage = (int64_t)(a.n + (a.residual_in ? 1 : 0)) * a.h * elem_size(a.dtype);
    if (stage > max_stage) max_stage = stage;
    if ((int)(a.h / 8) > max_row_packs) max_row_packs = (int)(a.h / 8);
  }
  one = one && max_stage <= ctx->max_dyn_smem && total_rows <= 0x7FFFFFFFLL;
  if (total_rows == 0) {
    ctx->last_variant = "none";
    return AR_OK;
  }
  if (!one) {
    for (int i = 0; i < count; ++i) {
      const ar_status st = ar_fused_reduce_rmsnorm(ctx, &calls[i], stream);
      if (st != AR_OK) return st;
    }
    ctx->last_variant = "fused_batch_sequential";
    return AR_OK;
  }

  ar::BatchParams bp;
  memset(&bp, 0, sizeof(bp));
  bp.count = count;
  bp.sp.stages = 1;
  bp.sp.err = ctx->d_status;
  bp.sp.wait_cycles = ctx->wait_cycles ? ctx->wait_cycles : 2000000000LL;
  bp.sp.stall_first = ctx->test_stall;
  int64_t acc = 0;
  for (int i = 0; i < count; ++i) {
    const ar_fused_args& a = calls[i];
    ar::fill_fused_params(bp.call[i], a, (int)(a.h / 8), 1);
    bp.call[i].prefetch = ctx->prefetch;
    bp.row_start[i] = acc;
    acc += a.m;
  }
  bp.row_start[count] = acc;
  const bool quant = c0.quant != AR_QUANT_NONE;
  const void* fn = c0.dtype == AR_DTYPE_BF16 ? ar::batch_kernel_bf16(c0.n, quant) : ar::batch_kernel_f16(c0.n, quant);
  if (!fn) return AR_ERR_UNSUPPORTED;
  int block = ((max_row_packs + 1) / 2 + 31) / 32 * 32;
  if (block < 32) block = 32;
  DeviceGuard g(ctx->device);
  void* args[1] = {&bp};
  const ar_status st = launch(ctx, fn, (unsigned)total_rows, (unsigned)block, 1, args, (size_t)max_stage, stream);
  if (st == AR_OK) ctx->last_variant = "fused_batch";
  return st;
}

}  // extern "C"
