/*
 * libar: fused N-way partial reduce + residual add + RMSNorm (+ per-token FP8 E4M3)
 * on one GB300 (sm_103a).
 *
 * The N "ranks" of a tensor-parallel all-reduce are N separate device buffers on one
 * GPU.  The library sums them and, in the fused form, applies the residual add,
 * RMSNorm (plain or gemma (1 + w) weighting) and an optional dynamic per-token FP8
 * epilogue, all in one kernel launch on the caller's stream.
 *
 * Sources (ROCm/aiter pull-request pages):
 *   [P1] "[HIP] fix(custom-ar): gfx1250 fused all-reduce + RMSNorm"
 *   [P2] "[OUTDATED] perf: optimize fused AllReduce + RMSNorm (custom_all_reduce)"
 *   [P3] "[HIP] [Perf] Specialize partial tiles in two-stage custom all-reduce"
 *
 * Numerics (bit-exact with the unfused composition, [P1] Changes; [P2] Technical
 * Details / 2stage):
 *   s   = round_T(((float)x_0 + (float)x_1) + ... + (float)x_{N-1})   fp32, rank order
 *   z   = round_T((float)s + (float)residual_in)                      (z = s if no residual)
 *   y   = round_T(z * rsqrt(mean_j(z_j^2) + eps) * w'),  w' = w or (1 + w)
 *   q   = e4m3_satfinite(y / scale), scale = max_j |y_j| / 448     (per row, of the ROUNDED y)
 * round_T is IEEE round-to-nearest-even.  The sum s and residual_out are bit-exact; y is
 * within one unit in the last place of the exactly-evaluated formula's rounding; FP8
 * codes follow from y exactly (IEEE fp32 division, saturating round-to-nearest-even).
 *
 * Ownership and side effects: the caller owns every buffer and the stream.  The compute
 * entry points never allocate, free or synchronise; they validate arguments on the host,
 * launch exactly one kernel on `stream` (or nothing), and return.  All pointers except
 * the host array of partial pointers are device pointers; the partial-pointer values
 * are copied into the kernel parameters, so that array may be reused as soon as the call
 * returns.  Inputs are not modified (except through the permitted exact aliases).
 *
 * Errors: every function returns an ar_status.  Argument errors are detected before
 * anything is launched and leave all buffers untouched.  AR_ERR_CUDA reports a failed
 * launch; ar_last_error() gives the CUDA message.  Nothing throws across this ABI.
 *
 * Threads: one context may be used by one host thread at a time; distinct contexts
 * are independent.  A context owns one small device status word (see ar_device_status)
 * and no other device memory.
 */
#ifndef AR_H
#define AR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ar_ctx ar_ctx;

typedef enum {
  AR_OK = 0,
  AR_ERR_INVALID_ARG = 1,     /* null pointer, n out of range, bad size, dtype, flag or eps */
  AR_ERR_UNSUPPORTED = 2,     /* device is not sm_103 / feature not available */
  AR_ERR_ALIGNMENT = 3,       /* a pointer is not aligned to its element size */
  AR_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed */
  AR_ERR_NOT_INITIALIZED = 5, /* ctx is NULL */
  AR_ERR_OVERLAP = 6          /* an output overlaps an input or another output (not an allowed exact alias) */
} ar_status;

typedef enum { AR_DTYPE_F32 = 0, AR_DTYPE_F16 = 1, AR_DTYPE_BF16 = 2 } ar_dtype;

/* Largest N (number of partial buffers).  TP8 is the widest group on the pages ([P2] Test
 * Results; [P1] Test results runs TP2/TP4). */
#define AR_MAX_PARTIALS 8

/* FP8 epilogue modes.  PER_GROUP (the per-group form that [P1] Changes names without a
 * group size or scale rule, here with both fixed): every run of group_size consecutive elements
 * of a row gets its own scale amax_group / 448 and codes by the per-token rules; scales
 * are [m, h / group_size] fp32 row-major. */
enum { AR_QUANT_NONE = 0, AR_QUANT_FP8_E4M3_PER_TOKEN = 1, AR_QUANT_FP8_E4M3_PER_GROUP = 2 };

/*
 * Create a context for CUDA device `device` (flags: must be 0).  Queries the SM count,
 * L2 size and cluster limits once and prepares the kernels (function attributes), so that
 * later calls can be captured in a CUDA graph.  Counterpart of constructing the
 * communicator, CustomAllreduce(group, device, max_size) ([P3] bench_allreduce_tail.py
 * listing).  Returns AR_ERR_UNSUPPORTED on a device other than compute capability 10.3.
 * The calling thread's current device is left unchanged.
 */
ar_status ar_init(ar_ctx** ctx, int device, unsigned flags);

/* Release a context (NULL is accepted).  Counterpart of CustomAllreduce.close() ([P3]). */
ar_status ar_destroy(ar_ctx* ctx);

/*
 * Plain sum-reduce of n partials ([P2] Technical Details / 2stage: one thread reduces one
 * 16-byte pack across all inputs in fp32, in input order, then downcasts once; [P3]
 * Proposed modifications: full tiles without predicates, leftover packs and elements by
 * a tail path).  Counterpart of custom_all_reduce(x) / tensor_model_parallel_all_reduce.
 *
 *   out[i] = round_T(sum_{r=0..n-1} (float)partials[r][i]) for i in [0, numel)
 *
 * out:      device, numel elements of dtype; may equal partials[k] exactly (in place),
 *           must not overlap any partial otherwise.
 * partials: HOST array of n device pointers, each numel elements of dtype.
 * n:        1..AR_MAX_PARTIALS.   numel: >= 0 (0 launches nothing and accepts any
 *           pointer values, NULL included).
 * dtype:    AR_DTYPE_F32, AR_DTYPE_F16 or AR_DTYPE_BF16 (fp32: the fp32 sum is stored).
 * stream:   cudaStream_t (NULL = legacy default stream).
 * Pointers must be aligned to the element size; 16-byte-aligned pointers take the vector
 * path, others a scalar path with the same results.  Large 16-bit arrays of 4 to 6
 * partials (at least 131072 elements per SM, a multiple of a row length of 2048..8192)
 * are summed by the staged fused kernel on the array viewed as rows, without residual or
 * norm: the same bits.
 */
ar_status ar_reduce_sum(ar_ctx* ctx, void* out, const void* const* partials, int n, int64_t numel,
                        ar_dtype dtype, void* stream);

/*
 * Arguments of the fused call.  Arrays are row-major with rows of h elements; rows may be
 * padded (row strides ld_in / ld_out; [P1] Changes sends padded or strided rows to the
 * unfused path, here they stay fused).  Counterpart of
 * tensor_model_parallel_fused_allreduce_rmsnorm(x, res, w, eps, gemma_norm=) and of the
 * unfused rmsnorm2d_fwd_with_add(out, x, res, res_out, w, eps, gemma, 0) ([P1] the
 * bench_ar_rms.py listing).
 */
typedef struct {
  int n;                                   /* number of partials, 1..AR_MAX_PARTIALS */
  const void* partials[AR_MAX_PARTIALS];   /* device, [m, h] of dtype each */
  const void* residual_in;                 /* device [m, h] or NULL (then z = s) */
  void* residual_out;                      /* device [m, h] or NULL */
  const void* weight;                      /* device [h] of dtype, required unless skip_norm */
  void* out;                               /* device [m, h]: y (the bf16/fp16 "mirror" when quant is on);
                                              NULL allowed only when quant is on */
  float eps;                               /* finite, >= 0 */
  int gemma;                               /* != 0: weight factor is (1 + w) ([P1] gemma_norm) */
  int quant;                               /* AR_QUANT_NONE, _FP8_E4M3_PER_TOKEN or _FP8_E4M3_PER_GROUP */
  void* q_out;                             /* device [m, h] E4M3 bytes, required when quant is on */
  float* scale_out;                        /* device fp32 scales, required when quant is on: [m] per
                                              token, [m, h / group_size] per group */
  int64_t m;                               /* rows (tokens), >= 0 (0 launches nothing; then
                                              only weight must be non-NULL) */
  int64_t h;                               /* hidden size, >= 1 */
  ar_dtype dtype;                          /* AR_DTYPE_BF16 or AR_DTYPE_F16 */
  int skip_norm;                           /* != 0: no RMSNorm; the output is z (the rounded sum plus
                                              residual), the FP8 epilogue quantises z (all-reduce +
                                              dynamic per-token FP8); weight may be NULL, eps and
                                              gemma are ignored */
  int out_fp32;                            /* != 0: `out` is [m, h] fp32 and receives the normalised
                                              row before its rounding to dtype (the FP8 epilogue still
                                              quantises the dtype-rounded row) */
  int group_size;                          /* per-group FP8: 8, 16, 32, 64, 128 or 256 elements,
                                              dividing h, with h <= 8192; ignored otherwise */
  int64_t ld_in;                           /* elements between the starts of consecutive rows of
                                              the partials and residual_in; 0 means h (contiguous),
                                              else >= h (padded or strided rows) */
  int64_t ld_out;                          /* the same for residual_out, out and q_out; 0 means h.
                                              Strides that keep rows 16-byte aligned (multiples of 8)
                                              take the vector kernels, others the element-wise ones */
} ar_fused_args;

/*
 * Fused reduce + residual add + RMSNorm (+ per-token FP8) in one launch ([P1] Changes:
 * fixed rank-order accumulation, same bf16/fp16 rounding as the unfused path, gemma_norm,
 * per-token FP8 output that quantises the rounded output like
 * dynamic_per_token_scaled_quant, optional bf16 mirror).
 *
 * Per row: z and residual_out as in the header comment; y written to `out` if non-NULL;
 * with quant, scale_out[row] = amax / 448 (fp32) and q_out = e4m3(y / scale), with an
 * all-zero row giving scale 0 and codes 0.  E4M3 is the OCP "fn" format (max 448).
 * Aliasing: residual_out and out may each be EXACTLY one of the [m, h] inputs
 * (residual_in or a partial) when ld_in and ld_out give the same stride, because every
 * element is read before the same thread writes it; any other overlap between an output and an input, or between two outputs,
 * is refused with AR_ERR_OVERLAP before anything is launched.
 */
ar_status ar_fused_reduce_rmsnorm(ar_ctx* ctx, const ar_fused_args* args, void* stream);

/*
 * Read and clear the context's device status word.  The staged variants wait on their
 * shared-memory copies (and, in the cluster form, on the peer CTAs' totals) with a bound
 * (about a second); if a wait ever runs out, the kernel stops early, its outputs are
 * incomplete, and it records code 1 here.  0 means no wait
 * has run out since the last read.  Synchronises the device (a blocking copy): call it
 * outside graph capture, e.g. after a batch of calls.  No counterpart on the pages.
 */
ar_status ar_device_status(ar_ctx* ctx, int* code);

/*
 * Several independent fused calls in one launch, so a batch of decode-sized calls pays
 * one launch instead of `count` (for the interleaved small and large fused calls that
 * [P1] Changes describes).
 *
 * calls: host array of `count` (1..AR_MAX_BATCH) argument blocks, each valid for
 * ar_fused_reduce_rmsnorm on its own and all with the same n, dtype, quant, skip_norm and
 * out_fp32.  The calls run concurrently, so no call may write memory that another call
 * reads or writes (AR_ERR_OVERLAP); inputs may be shared (for example one weight).  When
 * every call has 16-byte-aligned rows of at most 8192 elements (h a multiple of 8) this is
 * one kernel with one CTA per row of every call; otherwise the calls are launched one
 * after another (same results).  Results equal those of the separate calls within the
 * single-call bars (residual_out and FP8 from the same y bit-exact, y within one ulp).
 */
#define AR_MAX_BATCH 16
ar_status ar_fused_reduce_rmsnorm_batch(ar_ctx* ctx, const ar_fused_args* calls, int count, void* stream);

/*
 * ar_fused_reduce_rmsnorm over buffers in host memory: the same operation, arguments and
 * error rules, where any buffer (partials, residual_in/out, weight, out, q_out, scale_out)
 * may instead be page-locked host memory (cudaHostAlloc / cudaMallocHost, or
 * cudaHostRegister'ed) that the device can address.  The kernel reads the inputs from, and
 * writes the results into, that memory directly across the CPU-GPU link (on GB300 the
 * NVLink-C2C link to the Grace CPU), so the host<->device transfer and the computation are
 * one pass with no device staging buffers.  There is no counterpart on the pages; it is the
 * end-to-end form of the call for data that lives on the host.
 *
 * Each pointer is looked up with cudaPointerGetAttributes: page-locked host memory is
 * replaced by its device address, device memory of the context's device is used as is,
 * and anything else (pageable host memory, another device's memory) returns
 * AR_ERR_INVALID_ARG without launching (ar_last_error says why).  Only the kernels that
 * reach memory through plain loads and stores run (the one-CTA-per-row and cluster
 * forms); AR_OPT_FORCE_VARIANT = 3 (staged) returns AR_ERR_UNSUPPORTED here.
 *
 * Asynchronous like the device form: the results are in host memory once `stream` has
 * been synchronised, and the host must not write the inputs or read the outputs before.
 * Nothing is allocated; the call can be captured in a CUDA graph.
 */
ar_status ar_fused_reduce_rmsnorm_host(ar_ctx* ctx, const ar_fused_args* args, void* stream);

/*
 * Allocation-free form of ar_fused_reduce_rmsnorm, for callers that cannot call
 * cudaMalloc where they need this op: an engine that has handed all device memory to a
 * fixed plan (weights, KV cache, activations) up front, code running inside a stream
 * capture (allocation is not allowed there in the global capture mode), or a loop that
 * must not let an allocation synchronise the device.  Such callers cannot create a
 * context, because ar_init allocates the staged kernel's status word; this entry point
 * takes no context.  There is no counterpart on the pages.
 *
 * It runs the staged kernel only: arguments follow ar_fused_reduce_rmsnorm's rules, and
 * in addition h must be a multiple of 8 and at most 8192 and every pointer 16-byte
 * aligned (8-byte for q_out); otherwise it returns AR_ERR_UNSUPPORTED without launching.
 * The device is the calling thread's current device.
 *
 * Scratch: the kernel's one status word lives in a static device array of
 * AR_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that loads the
 * library holds until the process exits.  A call whose scratch need exceeded that size
 * would be refused with AR_ERR_UNSUPPORTED; the staged kernel needs 4 bytes at any size.
 * Every call clears the word on `stream` before its launch (a cudaMemsetAsync, which
 * allocates nothing).  All calls share the array, so calls that overlap on the GPU
 * (different streams without ordering) race on it; a bounded wait that runs out (about a
 * second) leaves incomplete outputs and code 1 in that word, which this interface does not
 * read back.
 *
 * The first call on a device does a one-time set-up (device attributes, the kernels'
 * shared-memory limit and the array's device address via cudaGetSymbolAddress); make that
 * first call before any stream capture.  Later calls launch one memset and one kernel.
 */
#define AR_NOALLOC_SCRATCH_BYTES 256
ar_status ar_fused_reduce_rmsnorm_noalloc(const ar_fused_args* args, void* stream);

/* Static description of a status code. */
const char* ar_status_string(ar_status s);

/* The CUDA error text of the last AR_ERR_CUDA on this context ("" if none). */
const char* ar_last_error(const ar_ctx* ctx);

/* Name of the kernel variant the last successful call launched (tests assert on it):
 * "reduce_vec", "reduce_vec_tail", "reduce_scalar", "reduce_staged" (a large 16-bit sum of
 * 4-6 partials run by the staged fused kernel on the array viewed as rows, without residual
 * or norm), "reduce_rows", "fused_row_vec", "fused_cluster_vec", "fused_staged",
 * "fused_staged_cluster" (rows longer than 8192 elements split over a cluster of staged CTAs),
 * "fused_scalar", "fused_cluster_scalar", "fused_batch", "fused_batch_sequential" or "none"
 * (empty call). */
const char* ar_last_variant(const ar_ctx* ctx);

/* Tuning and test overrides (0 = automatic for each, except AR_OPT_PDL).  Values outside
 * the documented range return AR_ERR_INVALID_ARG. */
typedef enum {
  AR_OPT_FORCE_VARIANT = 0,  /* 0 auto, 1 row, 2 cluster, 3 staged, 4 scalar (tail) */
  AR_OPT_CLUSTER_SIZE = 1,   /* 0 auto, else 1, 2, 4, 8 or 16 CTAs per row (with
                                AR_OPT_FORCE_VARIANT = 3 and 2..8: the staged cluster form) */
  AR_OPT_PACKS_PER_THREAD = 2, /* 0 auto, else 1, 2 or 4 16-byte packs per thread (1 or 2 in
                                  the staged cluster form) */
  AR_OPT_REDUCE_UNROLL = 3,  /* 0 auto, else 1 or 4 packs per thread per tile (a forced value
                                also keeps large 16-bit sums off the staged kernel) */
  AR_OPT_STAGES = 4,         /* 0 auto, else 1..4 shared-memory stages per CTA (staged variant) */
  AR_OPT_PDL = 5,            /* 1 (the default): launch with programmatic dependent launch, so
                                a kernel may be scheduled while its predecessor on the stream
                                still runs (every kernel here waits for its predecessors to
                                complete before it reads memory); 0: ordinary stream order */
  AR_OPT_WAIT_CYCLES = 6,    /* bound of one staged-kernel wait in SM clock cycles (1e3..8e9);
                                0 (the default): 2e9, about a second */
  AR_OPT_TEST_STALL = 7,     /* test hook, 0 (the default) or 1: the staged kernels arm each CTA's
                                first stage without issuing its copies, so that wait runs out and
                                the call ends early with code 1 in the status word (exercises the
                                failure path; outputs are then incomplete) */
  AR_OPT_L2_PREFETCH = 8     /* 1 (the default): the kernels on device memory prefetch their first
                                rows (or tile) of input into L2 before waiting for the previous
                                kernel on the stream, so those reads overlap its tail; 0: off.
                                Results are the same either way */
} ar_option;
ar_status ar_set_option(ar_ctx* ctx, ar_option opt, int64_t value);

/* Read-only facts about the context. */
typedef enum {
  AR_INFO_SM_COUNT = 0,
  AR_INFO_L2_BYTES = 1,
  AR_INFO_REDUCE_TILE_PACKS = 2, /* 16-byte packs per tile of the per-thread reduce kernel:
                                    with AR_OPT_REDUCE_UNROLL forced, of that form; else of the
                                    four-pack form (the automatic choice uses it for 16-bit sums
                                    of one to three partials of at least one wave of tiles, and
                                    one-pack tiles of 256 packs, a divisor, otherwise) */
  AR_INFO_DEVICE = 3
} ar_info;
ar_status ar_get_info(const ar_ctx* ctx, ar_info key, int64_t* value);

#ifdef __cplusplus
}
#endif
#endif /* AR_H */
